"""The causal backward as one reverse sweep per head (bf16, D = 128, the backward that reuses the forward).

The sweep takes g_i and each head's total state from the forward (kept in a backward-sized workspace)
and delta_i = dO_i . O_i from the forward's output, and forms dQ, dK and dV of each chunk together, last
chunk first.  LA_TC_SWEEP = 1 makes every eligible reusing backward run it (0: never, the two walks,
whose dQ walk then also takes g and delta from the forward and O), so that these cases cover both forms
whatever the size heuristic picks.  Checked here against the oracle: ragged and exact
chunk counts, one and two rows, one chunk, several heads walked by one CTA (LA_TC_MAX_CTAS), strided operands
(bit-identical to the contiguous call), and the refusals: a forward that kept nothing (forward-sized
workspace), a second backward on one forward's record, another K.  The two-walk form of the same call
is checked against the same oracle values.
"""
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

LA_ERR_STATE = 7


def _run(t, B, H, N, D, ws, fwd_ws=None):
    import torch
    from bwd_la_fwd_gb300 import la
    O, g = la.la_forward(t["Q"], t["K"], t["V"], True, workspace=ws if fwd_ws is None else fwd_ws)
    grads = la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    return O, grads


@pytest.mark.parametrize("B,H,N,cap", [(1, 2, 300, 0), (1, 1, 128, 0), (1, 3, 2, 0), (1, 1, 129, 0),
                                        (2, 3, 777, 2), (1, 2, 1024, 1)])
@pytest.mark.parametrize("mode", ["1", "0"])
def test_reusing_backward_matches_the_oracle(monkeypatch, oracle_lib, B, H, N, cap, mode):
    from bwd_la_fwd_gb300 import la
    D = 128
    monkeypatch.setenv("LA_TC_SWEEP", mode)
    if cap:
        monkeypatch.setenv("LA_TC_MAX_CTAS", str(cap))  # one CTA walks several heads
    x = inputs.generate(B, H, N, D, seed=900 + N + cap, dtype="bf16")
    t = {n: U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO")}
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    _, (dQ, dK, dV) = _run(t, B, H, N, D, ws)
    assert la.la_get_status(ws) == 0
    f = U.stored_to_f64(x, "bf16")
    r = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], True)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), r):
        U.assert_close(name, U.to_f64(got), ref, "bf16")


def test_single_row(monkeypatch, oracle_lib):
    """N = 1: dQ and dK vanish by the definition (dW_00 = (dO_0 . v_0 - delta_0) / g_0 = 0); they are checked
    to be zero within the tolerance times the size of the two terms that cancel, |dO_0 . v_0| / |g_0|
    times |k_0| or |q_0| (the sweep forms both terms from bf16 operands: dO / g and the stored O)."""
    import numpy as np
    from bwd_la_fwd_gb300 import la
    monkeypatch.setenv("LA_TC_SWEEP", "1")
    B, H, N, D = 1, 3, 1, 128
    x = inputs.generate(B, H, N, D, seed=913, dtype="bf16")
    t = {n: U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO")}
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    _, grads = _run(t, B, H, N, D, ws)
    assert la.la_get_status(ws) == 0
    got = dict(zip(("dQ", "dK", "dV"), (U.to_f64(a) for a in grads)))
    f = U.stored_to_f64(x, "bf16")
    _, g = oracle_lib.forward(f["Q"], f["K"], f["V"], True)
    _, _, dV = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], True)
    U.assert_close("dV", got["dV"], dV, "bf16")
    dov = np.abs(np.sum(f["dO"] * f["V"], axis=-1, keepdims=True)) / np.abs(g[..., None])
    for name, other in (("dQ", f["K"]), ("dK", f["Q"])):
        assert np.all(np.isfinite(got[name])), name
        scale = dov * np.max(np.abs(other), axis=-1, keepdims=True)
        assert np.all(np.abs(got[name]) <= U.TOL["bf16"] * scale + 1e-30), f"{name}: {np.max(np.abs(got[name]) / scale):.3e}"


def test_strided_operands_are_bit_identical(monkeypatch):
    """[B,N,H,D] views: O is read and dQ, dK, dV are written row by row with the caller's strides."""
    import torch
    from bwd_la_fwd_gb300 import la
    monkeypatch.setenv("LA_TC_SWEEP", "1")
    B, H, N, D = 2, 3, 300, 128
    x = inputs.generate(B, H, N, D, seed=911, dtype="bf16")
    t = {n: U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO")}
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    _, ref = _run(t, B, H, N, D, ws)
    bnhd = lambda a: a.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    ts = {k: bnhd(v) for k, v in t.items()}
    O = bnhd(torch.empty_like(t["Q"]))
    outs = [bnhd(torch.empty_like(t["Q"])) for _ in range(3)]
    ws2 = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    la.la_forward(ts["Q"], ts["K"], ts["V"], True, O=O, workspace=ws2)
    la.la_backward(ts["Q"], ts["K"], ts["V"], O, ts["dO"], True, dQ=outs[0], dK=outs[1], dV=outs[2], workspace=ws2,
                   reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws2) == 0
    for name, a, b in zip(("dQ", "dK", "dV"), outs, ref):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("mode", ["1", "0"])
@pytest.mark.parametrize("case", ["forward_sized_workspace", "second_backward", "other_keys"])
def test_refusals_compute_nothing(monkeypatch, case, mode):
    """Both forms of the causal reusing backward (the sweep, and the two walks whose dQ walk takes g and
    O from the forward) refuse a workspace whose forward kept nothing, was used up or had other keys."""
    import torch
    from bwd_la_fwd_gb300 import la
    monkeypatch.setenv("LA_TC_SWEEP", mode)
    B, H, N, D = 1, 2, 513, 128
    x = inputs.generate(B, H, N, D, seed=912, dtype="bf16")
    t = {n: U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO")}
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    K = t["K"].clone() if case == "other_keys" else t["K"]
    # the same buffer, offered to the forward at the forward's size: it keeps neither g nor the totals
    fws = ws[: la.la_workspace_bytes(B, H, N, D, True, la.LA_BF16, False)] if case == "forward_sized_workspace" else ws
    O, _ = la.la_forward(t["Q"], K, t["V"], True, workspace=fws)
    if case == "second_backward":
        la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, workspace=ws, reuse_forward_state=True)
        assert la.la_get_status(ws) == 0
    dQ, dK, dV = (torch.full_like(t["Q"], 7.0) for _ in range(3))
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, dQ=dQ, dK=dK, dV=dV, workspace=ws,
                   reuse_forward_state=True)
    assert la.la_get_status(ws) == LA_ERR_STATE
    for g in (dQ, dK, dV):
        assert bool((g == 7.0).all())  # nothing was computed
    # a fresh forward on the backward-sized workspace makes the sweep possible again
    O, _ = la.la_forward(t["Q"], t["K"], t["V"], True, O=O, workspace=ws)
    la.la_backward(t["Q"], t["K"], t["V"], O, t["dO"], True, dQ=dQ, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == 0
    assert not bool((dQ == 7.0).any())
