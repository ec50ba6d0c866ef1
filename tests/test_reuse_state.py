"""la_backward_with_forward_state: the backward that takes the per-piece state sums from the forward.

The forward's first kernel sums k_j v_j^T, k_j and v_j over each piece of rows; the backward needs the
same sums.  Non-causal, and on the SIMT and D = 256 paths, the reusing entry point must give exactly
what la_backward gives (the sums are the same numbers, so the gradients are bit-identical).  Causal on the
tensor-core kernels it also takes g from the forward and forms delta_i = dO_i . O_i from the stored O
(in the two walks, LA_TC_SWEEP = 0 here, or as the single sweep, test_sweep.py), which rounds
differently from la_backward's g and delta formed from the state: there it must agree with la_backward
and with the oracle to within the tolerance.  It must refuse (LA_ERR_STATE, nothing computed) when the
workspace holds sums of other K, V or of another work split -- or none, because a backward has since used
them up -- and is plain la_backward on the SIMT path.
For bf16 with D = 256 what is reused is the normaliser g_i, which the forward keeps in a backward-sized
workspace together with a record of Q, K, shape and mask: the same bit-identity and refusal rules hold.
"""
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

LA_ERR_STATE = 7


def _tensors(B, H, N, D, dtype, seed):
    x = inputs.generate(B, H, N, D, seed=seed, dtype=dtype)
    return x, {n: U.to_device(x[n], dtype) for n in ("Q", "K", "V", "dO")}


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("bf16", 256), ("f32", 64)])
def test_reuse_is_bit_identical_to_la_backward(monkeypatch, causal, dtype, D):
    import torch
    from bwd_la_fwd_gb300 import la
    monkeypatch.setenv("LA_TC_SWEEP", "0")
    B, H, N = 2, 3, 777
    _, t = _tensors(B, H, N, D, dtype, seed=71)
    code = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    ws = la.new_workspace(B, H, N, D, causal, code, True)
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], causal, workspace=ws)
    got = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], causal, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    ref = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], causal)
    torch.cuda.synchronize()
    if causal and dtype == "bf16" and D <= 128:  # g from the forward, delta from the stored O
        for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
            U.assert_close(name, U.to_f64(a), U.to_f64(r), dtype)
        return
    for a, r in zip(got, ref):
        assert torch.equal(a, r)


def test_reuse_matches_the_oracle(oracle_lib):
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D, causal = 1, 2, 300, 128, 1
    x, t = _tensors(B, H, N, D, "bf16", seed=72)
    ws = la.new_workspace(B, H, N, D, causal, la.LA_BF16, True)
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], causal, workspace=ws)
    dQ, dK, dV = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], causal, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    f = U.stored_to_f64(x, "bf16")
    r = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], True)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), r):
        U.assert_close(name, U.to_f64(got), ref, "bf16")


def test_reuse_without_a_forward_reports_state_error():
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 2, 513, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=73)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)  # zero-filled: no state recorded
    dQ = torch.full_like(t["Q"], 7.0)
    la.la_backward(t["Q"], t["K"], t["V"], t["Q"], t["dO"], True, dQ=dQ, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE
    assert bool((dQ == 7.0).all())  # nothing was computed
    assert la.la_get_status(ws) == 0  # the status is cleared once read


def test_reuse_after_a_forward_on_other_keys_reports_state_error():
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 2, 513, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=74)
    K2 = t["K"].clone()
    ws = la.new_workspace(B, H, N, D, 0, la.LA_BF16, True)
    O, _ = la.la_forward(t["Q"], K2, t["V"], False, workspace=ws)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], False, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE


def test_reuse_with_another_work_split_reports_state_error(monkeypatch):
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 3, 1000, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=75)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)
    monkeypatch.setenv("LA_TC_MAX_CTAS", "5")
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], True, workspace=ws)
    monkeypatch.delenv("LA_TC_MAX_CTAS")
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE


def test_simt_call_on_the_workspace_clears_the_record():
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 2, 513, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=76)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], True, workspace=ws)
    # an fp32 call (SIMT kernels, another layout of the same workspace bytes) in between
    small = {n: torch.randn(1, 1, 64, 64, device="cuda") for n in ("Q", "K", "V")}
    assert la.la_workspace_bytes(1, 1, 64, 64, True, la.LA_F32, False) <= ws.numel()
    la.la_forward(small["Q"], small["K"], small["V"], True, workspace=ws)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE
    # a fresh forward records the state again
    la.la_forward(t["Q"], t["K"], t["V"], True, O=O, workspace=ws)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == 0


@pytest.mark.parametrize("fwd_causal", [1, 0])
def test_reuse_after_a_forward_with_the_other_mask_reports_state_error(fwd_causal):
    """A causal forward leaves each piece's own sums, a non-causal one the head totals; a backward with the
    other mask must not take them."""
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 2, 700, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=77)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], bool(fwd_causal), workspace=ws)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], not fwd_causal, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE


@pytest.mark.parametrize("case", ["other_queries", "forward_sized_workspace", "other_mask"])
def test_wide_reuse_without_matching_forward_reports_state_error(case):
    """bf16 D = 256: the reusing backward checks the record of the forward's g (Q, K, strides, shape, mask)
    on the device; when it does not match, the row kernel and the three walks compute nothing."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 1, 2, 300, 256
    _, t = _tensors(B, H, N, D, "bf16", seed=81)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)
    Q = t["Q"].clone() if case == "other_queries" else t["Q"]
    fws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, False) if case == "forward_sized_workspace" else ws
    O, _ = la.la_forward(Q, t["K"], t["V"], case != "other_mask", workspace=fws)
    dQ, dK, dV = (torch.full_like(t["Q"], 7.0) for _ in range(3))
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, dQ=dQ, dK=dK, dV=dV, workspace=ws,
                   reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE
    for g in (dQ, dK, dV):
        assert bool((g == 7.0).all())  # nothing was computed
    # the plain backward on the same workspace then computes, and the record check is not sticky
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, dQ=dQ, workspace=ws)
    assert la.la_get_status(ws) == 0
    assert not bool((dQ == 7.0).any())


def test_a_backward_uses_up_the_forward_sums():
    """The backward keeps its reverse-direction sums in the slots that held the forward's sums: a second
    reusing backward after one forward finds no forward sums (LA_ERR_STATE, nothing computed); a fresh
    forward makes reuse possible again, with the same results."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 2, 3, 777, 128
    _, t = _tensors(B, H, N, D, "bf16", seed=78)
    ws = la.new_workspace(B, H, N, D, 1, la.LA_BF16, True)
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], True, workspace=ws)
    first = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    dQ = torch.full_like(t["Q"], 7.0)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, dQ=dQ, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE
    assert bool((dQ == 7.0).all())
    la.la_forward(t["Q"], t["K"], t["V"], True, O=O, workspace=ws)
    again = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    for a, b in zip(first, again):
        assert torch.equal(a, b)
