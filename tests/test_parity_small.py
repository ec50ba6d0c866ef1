"""GPU parity against the explicit fp64 oracle, element by element, at sizes the oracle finishes in
seconds: every supported D, fp32 and bf16 storage, causal and non-causal, several segments of rows
plus a ragged tail, and the degenerate sizes (N = 1, 2, around tile edges)."""
import numpy as np
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


def _check(oracle_lib, B, H, N, D, dtype, causal, seed):
    x = inputs.generate(B, H, N, D, seed, dtype=dtype)
    got = U.run_library(x, dtype, causal)
    f = U.stored_to_f64(x, dtype)
    O, g = oracle_lib.forward(f["Q"], f["K"], f["V"], causal)
    dQ, dK, dV = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    ref = {"O": O, "g": g, "dQ": dQ, "dK": dK, "dV": dV}
    return {k: U.assert_close(k, got[k], ref[k], dtype) for k in ref}


def test_tiny_case_fp32(oracle_lib):
    """B=1, H=2, N=64, D=16, fp32, seed 0: elementwise relative error <= 1e-5."""
    for causal in (1, 0):
        _check(oracle_lib, 1, 2, 64, 16, "f32", causal, seed=0)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
def test_several_segments_and_ragged_tail(oracle_lib, D, dtype, causal):
    seg = max(256, 2 * D)
    _check(oracle_lib, 1, 2, 2 * seg + 37, D, dtype, causal, seed=100 + D)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [2, 63, 127, 128, 129, 255, 257])
def test_edge_lengths(oracle_lib, N, dtype, causal):
    _check(oracle_lib, 1, 3, N, 64, dtype, causal, seed=7 + N)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
def test_single_row(oracle_lib, D, dtype, causal):
    """N = 1: the one weight is W_00 = g_0, so O_0 = v_0, dV_0 = dO_0, and dW_00 = (dO_0 . v_0 - delta_0) / g_0
    vanishes (delta_0 = dO_0 . O_0 = dO_0 . v_0): dQ and dK are zero by the definition.  O, g and dV are
    checked as everywhere; dQ and dK, whose normalised error has no scale here, are checked to be zero
    within the tolerance times the size of the two terms that cancel, |dO_0 . v_0| / |g_0| times |k_0| or
    |q_0| (bf16 storage rounds operands of the tensor-core products, e.g. dO / g, before that difference is
    taken)."""
    x = inputs.generate(1, 3, 1, D, 7 + D, dtype=dtype)
    got = U.run_library(x, dtype, causal)
    f = U.stored_to_f64(x, dtype)
    O, g = oracle_lib.forward(f["Q"], f["K"], f["V"], causal)
    dQ, dK, dV = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    for name, r in (("O", O), ("g", g), ("dV", dV)):
        U.assert_close(name, got[name], r, dtype)
    dov = np.abs(np.sum(f["dO"] * f["V"], axis=-1, keepdims=True)) / np.abs(g[..., None])  # [B,H,1,1]
    for name, other in (("dQ", f["K"]), ("dK", f["Q"])):
        assert np.all(np.isfinite(got[name])), name
        scale = dov * np.max(np.abs(other), axis=-1, keepdims=True)
        assert np.all(np.abs(got[name]) <= U.TOL[dtype] * scale + 1e-30), f"{name}: {np.max(np.abs(got[name]) / scale):.3e}"


@pytest.mark.parametrize("D", [64, 128])
def test_many_heads_short_sequences(oracle_lib, D):
    _check(oracle_lib, 3, 5, 130, D, "bf16", 1, seed=21)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("ctas", [1, 3, 7])
def test_multi_chunk_slices(oracle_lib, monkeypatch, ctas, causal):
    """Few CTAs, so that each one walks several chunks and pieces of several heads (tensor-core path)."""
    monkeypatch.setenv("LA_TC_MAX_CTAS", str(ctas))
    _check(oracle_lib, 1, 3, 549, 128, "bf16", causal, seed=31 + ctas)


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("D", [32, 64])
def test_multi_chunk_slices_narrow_heads(oracle_lib, monkeypatch, D, causal):
    """The tensor-core kernels on D = 32, 64 (columns past D zero-extended), several chunks and pieces per CTA."""
    monkeypatch.setenv("LA_TC_MAX_CTAS", "3")
    _check(oracle_lib, 2, 3, 549, D, "bf16", causal, seed=41 + D)


@pytest.mark.parametrize("dtype,D,launches", [("bf16", 16, 8), ("bf16", 32, 5), ("bf16", 64, 5), ("bf16", 128, 5),
                                              ("bf16", 256, 5), ("f32", 64, 8), ("f32", 128, 8)])
def test_path_taken(dtype, D, launches):
    """bf16 with D = 32, 64, 128 runs on the tensor-core kernels of 128 columns (backward: sums, combine, dQ
    walk, combine, dK/dV walk), bf16 with D = 256 on the wide tensor-core kernels (backward: g, row terms,
    dQ, dK, dV), the rest (bf16 with D = 16, fp32) on the CUDA-core kernels (backward: 8 launches)."""
    import torch
    from bwd_la_fwd_gb300 import la
    x = inputs.generate(1, 2, 300, D, 3, dtype=dtype)
    Q, K, V, dO = (U.to_device(x[n], dtype) for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(1, 2, 300, D, True, la.LA_BF16 if dtype == "bf16" else la.LA_F32, True)
    O, _ = la.la_forward(Q, K, V, True, workspace=ws)
    n0 = la.la_launch_count()
    la.la_backward(Q, K, V, O, dO, True, workspace=ws)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    assert la.la_launch_count() - n0 == launches


@pytest.mark.parametrize("N,whole", [(128, True), (256, False)])
def test_noncausal_whole_heads_need_no_combine(oracle_lib, N, whole):
    """Non-causal, bf16 D = 128, B = 1, H = 2: with one chunk per CTA, a head of one chunk is one CTA's
    whole slice, so its piece sums are the head's totals and no combine kernel runs (forward 2 launches,
    backward 3, reusing backward 2); a head of two chunks spans two CTAs and takes the combine (3, 5, 3).
    Both agree with the oracle, and the reusing backward with the plain one bit for bit."""
    import torch
    from bwd_la_fwd_gb300 import la
    x = inputs.generate(1, 2, N, 128, 5, dtype="bf16")
    Q, K, V, dO = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(1, 2, N, 128, False, la.LA_BF16, True)
    n0 = la.la_launch_count()
    O, g = la.la_forward(Q, K, V, False, workspace=ws)
    n1 = la.la_launch_count()
    plain = la.la_backward(Q, K, V, O, dO, False, workspace=ws)
    n2 = la.la_launch_count()
    la.la_forward(Q, K, V, False, O=O, workspace=ws)
    n3 = la.la_launch_count()
    reuse = la.la_backward(Q, K, V, O, dO, False, workspace=ws, reuse_forward_state=True)
    n4 = la.la_launch_count()
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    assert (n1 - n0, n2 - n1, n4 - n3) == ((2, 3, 2) if whole else (3, 5, 3))
    for a, b in zip(plain, reuse):
        assert torch.equal(a, b)
    _check(oracle_lib, 1, 2, N, 128, "bf16", False, seed=5)


def test_repeatable_and_workspace_reusable():
    """Two calls on one workspace give bit-identical results (no state leaks between calls)."""
    import torch
    from bwd_la_fwd_gb300 import la
    x = inputs.generate(2, 2, 700, 128, 5, dtype="bf16")
    Q, K, V, dO = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(2, 2, 700, 128, True, la.LA_BF16, True)
    outs = []
    for _ in range(2):
        O, g = la.la_forward(Q, K, V, True, workspace=ws)
        grads = la.la_backward(Q, K, V, O, dO, True, workspace=ws)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (O, g, *grads)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert la.la_get_status(ws) == 0


@pytest.mark.parametrize("ctas", [1, 3])
def test_first_chunk_of_each_piece_waits_for_its_tiles(oracle_lib, monkeypatch, ctas):
    """Non-causal forward, few CTAs, fresh workspaces: the first chunk of every piece (right after a short
    carry load) must read its Q tile only after the tile has landed; repeated, so that a read that races
    the copy shows up as a wrong normaliser in that chunk."""
    import torch
    from bwd_la_fwd_gb300 import la
    monkeypatch.setenv("LA_TC_MAX_CTAS", str(ctas))
    x = inputs.generate(1, 3, 549, 128, 31 + ctas, dtype="bf16")
    f = U.stored_to_f64(x, "bf16")
    O_ref, g_ref = oracle_lib.forward(f["Q"], f["K"], f["V"], False)
    Q, K, V = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V"))
    for _ in range(4):
        ws = la.new_workspace(1, 3, 549, 128, False, la.LA_BF16, False)
        O, g = la.la_forward(Q, K, V, False, workspace=ws)
        torch.cuda.synchronize()
        assert la.la_get_status(ws) == 0
        U.assert_close("g", U.to_f64(g), g_ref, "bf16")
        U.assert_close("O", U.to_f64(O), O_ref, "bf16")


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 300])
def test_wide_heads_edge_lengths(oracle_lib, N, causal):
    """bf16 D = 256 (the wide tensor-core kernels: one CTA per head and 128-column output half) at lengths
    around the 128-row chunk; at N = 1 dQ and dK vanish by the definition and are checked as in
    test_single_row."""
    if N > 1:
        _check(oracle_lib, 1, 3, N, 256, "bf16", causal, seed=61 + N)
        return
    x = inputs.generate(1, 3, 1, 256, 61, dtype="bf16")
    got = U.run_library(x, "bf16", causal)
    f = U.stored_to_f64(x, "bf16")
    O, g = oracle_lib.forward(f["Q"], f["K"], f["V"], causal)
    dQ, dK, dV = oracle_lib.backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    for name, r in (("O", O), ("g", g), ("dV", dV)):
        U.assert_close(name, got[name], r, "bf16")
    dov = np.abs(np.sum(f["dO"] * f["V"], axis=-1, keepdims=True)) / np.abs(g[..., None])
    for name, other in (("dQ", f["K"]), ("dK", f["Q"])):
        scale = dov * np.max(np.abs(other), axis=-1, keepdims=True)
        assert np.all(np.abs(got[name]) <= U.TOL["bf16"] * scale + 1e-30), name


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("ctas", [2, 4])
def test_wide_heads_several_heads_per_cta(oracle_lib, monkeypatch, ctas, causal):
    """bf16 D = 256 with the grid capped (LA_TC_MAX_CTAS): each CTA walks several heads in turn, each from a
    zero state, and the g pass (one CTA per head) several heads too."""
    monkeypatch.setenv("LA_TC_MAX_CTAS", str(ctas))
    _check(oracle_lib, 2, 3, 300, 256, "bf16", causal, seed=71 + ctas)
