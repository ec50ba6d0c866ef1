"""Strided operands on the GPU: [B,N,H,D] views and the slices of a fused [B,N,3,H,D] QKV tensor go to the
library as they are (no transpose copy) and give exactly what the contiguous calls give on the same
values, on every path (tensor cores: bf16 with D = 32 ... 128 and, on the wide kernels, D = 256; CUDA cores:
fp32), causal and non-causal, forward, backward and the backward that reuses the forward's sums; one case
is also checked against the oracle.
bf16 with D = 32 or 64 runs on the tensor-core kernels with the columns past D zero-extended by the tensor
maps: the fused cases check that no store reaches past an operand's D columns into its neighbour's.
"""
import numpy as np
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [("bf16", 128), ("bf16", 64), ("bf16", 32), ("bf16", 256), ("f32", 64)]


def _bnhd(t):
    """A [B,N,H,D] copy of a contiguous [B,H,N,D] tensor, returned as its [B,H,N,D] view."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def _run(Q, K, V, dO, causal, outs=None, reuse=False):
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = Q.shape
    dt = la.LA_BF16 if Q.dtype == torch.bfloat16 else la.LA_F32
    ws = la.new_workspace(B, H, N, D, causal, dt, True)
    O = None if outs is None else outs[0]
    O, g = la.la_forward(Q, K, V, causal, O=O, workspace=ws)
    kw = {} if outs is None else {"dQ": outs[1], "dK": outs[2], "dV": outs[3]}
    dQ, dK, dV = la.la_backward(Q, K, V, O, dO, causal, workspace=ws, reuse_forward_state=reuse, **kw)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    return [t.clone() for t in (O, g, dQ, dK, dV)]


def _inputs(dtype, D, seed, B=2, H=3, N=300):
    x = inputs.generate(B, H, N, D, seed, dtype=dtype)
    return x, [U.to_device(x[n], dtype) for n in ("Q", "K", "V", "dO")]


@pytest.mark.parametrize("reuse", [False, True])
@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype,D", CASES)
def test_bnhd_views_match_contiguous(dtype, D, causal, reuse):
    import torch
    _, (Q, K, V, dO) = _inputs(dtype, D, seed=400 + D + causal)
    ref = _run(Q, K, V, dO, causal, reuse=reuse)
    Qs, Ks, Vs, dOs = (_bnhd(t) for t in (Q, K, V, dO))
    assert not Qs.is_contiguous()
    outs = [_bnhd(torch.empty_like(Q)) for _ in range(4)]
    got = _run(Qs, Ks, Vs, dOs, causal, outs=outs, reuse=reuse)
    for name, a, b in zip(("O", "g", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name
    assert torch.equal(outs[1], ref[2])  # the results landed in the strided outputs


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype,D", CASES)
def test_fused_qkv_slices_match_contiguous(dtype, D, causal):
    """Q, K, V read from one fused [B,N,3,H,D] projection output, dQ, dK, dV written into one fused
    gradient tensor of the same shape (outputs that interleave, row by row, without meeting)."""
    import torch
    _, (Q, K, V, dO) = _inputs(dtype, D, seed=410 + D + causal, B=2, H=4, N=257)
    B, H, N, _ = Q.shape
    fused = torch.empty(B, N, 3, H, D, dtype=Q.dtype, device=Q.device)
    for k, t in enumerate((Q, K, V)):
        fused[:, :, k] = t.permute(0, 2, 1, 3)
    Qs, Ks, Vs = (fused[:, :, k].permute(0, 2, 1, 3) for k in range(3))
    grad = torch.empty_like(fused)
    dQs, dKs, dVs = (grad[:, :, k].permute(0, 2, 1, 3) for k in range(3))
    ref = _run(Q, K, V, dO, causal)
    got = _run(Qs, Ks, Vs, dO, causal, outs=[torch.empty_like(Q), dQs, dKs, dVs])
    for name, a, b in zip(("O", "g", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name
    for k, r in enumerate(ref[2:]):
        assert torch.equal(grad[:, :, k].permute(0, 2, 1, 3), r)


def test_strided_against_the_oracle(oracle_lib):
    x, (Q, K, V, dO) = _inputs("bf16", 128, seed=420, B=1, H=2, N=333)
    got = _run(*(_bnhd(t) for t in (Q, K, V, dO)), 1)
    f = U.stored_to_f64(x, "bf16")
    O, g = oracle_lib.forward(f["Q"], f["K"], f["V"], True)
    dQ, dK, dV = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], True)
    for name, a, r in zip(("O", "g", "dQ", "dK", "dV"), got, (O, g, dQ, dK, dV)):
        U.assert_close(name, U.to_f64(a), r, "bf16")


def test_reuse_with_other_key_strides_reports_state_error():
    """The forward's sums belong to K and V as laid out then: a reusing backward that reads the same K
    buffer with other strides must refuse."""
    import torch
    from bwd_la_fwd_gb300 import la
    _, (Q, K, V, dO) = _inputs("bf16", 128, seed=430, B=1, H=2, N=300)
    Kb = _bnhd(K)
    ws = la.new_workspace(1, 2, 300, 128, 1, la.LA_BF16, True)
    O, _ = la.la_forward(Q, Kb, V, True, workspace=ws)
    K_other = torch.as_strided(Kb, Kb.shape, (Kb.stride(0), 300 * 128, 128, 1))  # the same buffer read as [B,H,N,D]
    la.la_backward(Q, K_other, V, O, dO, True, workspace=ws, reuse_forward_state=True)
    assert la.la_get_status(ws) == 7


@pytest.mark.parametrize("causal", [1, 0])
def test_bnhd_views_at_the_standard_shape(causal):
    """The 4-D tensor-map kernels at the benchmark's shape (B = 4, H = 16, N = 4096, D = 128, bf16): every
    output equals the contiguous call's bit for bit, forward and the reusing backward."""
    import torch
    B, H, N, D = 4, 16, 4096, 128
    g = torch.Generator(device="cuda").manual_seed(440 + causal)
    Q, K = (torch.randn(B, H, N, D, device="cuda", generator=g) / D ** 0.5 for _ in range(2))
    V, dO = (torch.randn(B, H, N, D, device="cuda", generator=g) for _ in range(2))
    Q, K, V, dO = (t.to(torch.bfloat16) for t in (Q, K, V, dO))
    ref = _run(Q, K, V, dO, causal, reuse=True)
    outs = [_bnhd(torch.empty_like(Q)) for _ in range(4)]
    got = _run(*(_bnhd(t) for t in (Q, K, V, dO)), causal, outs=outs, reuse=True)
    for name, a, b in zip(("O", "g", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name
