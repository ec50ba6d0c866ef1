"""GPU parity at the full workload sizes, on the launch configuration the benchmark times.

The benchmark times la_forward followed by la_backward_with_forward_state on the forward's workspace (the
backward takes what the forward left there -- its per-piece K^T V sums, and for the causal single sweep
g and each head's total state -- instead of recomputing it).  Every case here runs exactly that
sequence, then the plain la_backward on the same workspace; both backwards' outputs are checked against
the oracle (the two are bit-identical when the reusing one runs as the two walks too).

The explicit oracle costs O(N^2 D) per head, so at these sizes it checks sampled outputs it can compute
one row at a time (O_i, g_i, dQ_i cost O(N D) each; dK_j, dV_j cost O((N - j) N D), so they are sampled
near the end of causal heads).  Whole heads are checked against the fp64 running-state form (itself
pinned to the explicit oracle at small sizes): every head up to N = 8192, so that every piece of the
work split -- including pieces that start or end inside an interior head -- is compared, and eight heads
spread over the batch beyond that (the running-state form of all 64 heads of N = 65536 would take
minutes of host time).  Sizes: the paper's standalone shape (B=4 H=16 N=4096 D=128, causal and
non-causal), the head-size sweep (D = 32, 64, 256 at N = 4096), the sequence-length sweep (N = 1024 ...
65536 at D = 128) and two layers of the 1.4B-class step (B=8 H=16 N=2048 D=128).
"""
import numpy as np
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


def _heads_f64(x, heads, B, H, N, D):
    return {k: inputs.to_f64(v.reshape(B * H, N, D)[heads], "bf16").reshape(1, len(heads), N, D) for k, v in x.items()}


def _sample_rows(N):
    base = [0, 1, 2, 63, 64, 127, 128, 129, 255, 256, 257, 511, 512, 513, N // 2, N - 129, N - 128, N - 2, N - 1]
    return sorted({r for r in base if 0 <= r < N})


def _compared_heads(BH, N):
    if N <= 8192:
        return list(range(BH))
    return sorted({0, 1, BH // 4, BH // 2 - 1, BH // 2, 3 * BH // 4 + 1, BH - 2, BH - 1})


def _check_full(oracle_lib, B, H, N, D, seed, causal, layer=0, layers=1):
    import torch
    from bwd_la_fwd_gb300 import la
    x = inputs.generate(B, H, N, D, seed, dtype="bf16", layers=layers)
    if layers > 1:
        x = x[layer]
    Q, K, V, dO = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(B, H, N, D, causal, la.LA_BF16, True)
    O, g = la.la_forward(Q, K, V, causal, workspace=ws)
    # the benchmark's backward: the forward's state sums reused from the workspace
    dQ, dK, dV = la.la_backward(Q, K, V, O, dO, causal, workspace=ws, reuse_forward_state=True)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    heads = _compared_heads(B * H, N)
    host = lambda v: v.reshape(B * H, N, -1)[heads].double().cpu().numpy().reshape(1, len(heads), N, -1)
    got = {k: host(v) for k, v in {"O": O, "g": g, "dQ": dQ, "dK": dK, "dV": dV}.items()}
    got["g"] = got["g"].reshape(1, len(heads), N)
    # the plain backward recomputes those sums
    plain = la.la_backward(Q, K, V, O, dO, causal, workspace=ws)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    got_plain = {k: host(v) for k, v in zip(("dQ", "dK", "dV"), plain)}
    del plain
    f = _heads_f64(x, heads, B, H, N, D)

    # whole heads against the fp64 running-state form
    rO, rg = oracle_lib.prefix_forward(f["Q"], f["K"], f["V"], causal)
    rdQ, rdK, rdV = oracle_lib.prefix_backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    for name, ref in (("O", rO), ("g", rg), ("dQ", rdQ), ("dK", rdK), ("dV", rdV)):
        U.assert_close(name, got[name], ref, "bf16")
    for name, ref in (("dQ", rdQ), ("dK", rdK), ("dV", rdV)):
        U.assert_close(name, got_plain[name], ref, "bf16")

    # sampled rows of the first and last compared heads against the explicit definition
    ends = [0, len(heads) - 1]
    fe = {k: v[:, ends] for k, v in f.items()}
    ge = {k: v[:, ends] for k, v in got.items()}
    rows = _sample_rows(N)
    flat = np.array([k * N + r for k in range(2) for r in rows])
    sO, sg = oracle_lib.forward_rows(fe["Q"], fe["K"], fe["V"], causal, flat)
    sdQ = oracle_lib.dq_rows(fe["Q"], fe["K"], fe["V"], fe["dO"], causal, flat)
    U.assert_close("O", ge["O"].reshape(-1, D)[flat], sO, "bf16")
    U.assert_close("g", ge["g"].reshape(-1)[flat], sg, "bf16")
    U.assert_close("dQ", ge["dQ"].reshape(-1, D)[flat], sdQ, "bf16")
    kv_rows = [N - 3, N - 2, N - 1] if causal else [0, N // 2, N - 1]
    kflat = np.array([k * N + r for k in range(2) for r in kv_rows if r >= 0])
    sdK, sdV = oracle_lib.dkdv_rows(fe["Q"], fe["K"], fe["V"], fe["dO"], causal, kflat)
    U.assert_close("dK", ge["dK"].reshape(-1, D)[kflat], sdK, "bf16")
    U.assert_close("dV", ge["dV"].reshape(-1, D)[kflat], sdV, "bf16")


@pytest.mark.parametrize("causal", [1, 0])
def test_standard_shape(oracle_lib, causal):
    _check_full(oracle_lib, 4, 16, 4096, 128, seed=1, causal=causal)


@pytest.mark.parametrize("D", [32, 64, 256])
def test_head_size_sweep(oracle_lib, D):
    _check_full(oracle_lib, 4, 16, 4096, D, seed=2, causal=1)


@pytest.mark.parametrize("N", [1024, 2048, 8192, 16384, 32768, 65536])
def test_sequence_length_sweep(oracle_lib, N):
    _check_full(oracle_lib, 4, 16, N, 128, seed=3, causal=1)


@pytest.mark.parametrize("layer", [0, 1])
def test_decoder_step_layers(oracle_lib, layer):
    _check_full(oracle_lib, 8, 16, 2048, 128, seed=4, causal=1, layer=layer, layers=2)


def test_peak_memory_within_floor_margin():
    """Peak device memory of a causal fwd + bwd at the standard shape, everything allocated by torch, is
    within 1.2x of the O(BHND) I/O floor (8 tensors plus the fp32 normaliser)."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 4, 16, 4096, 128
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    Q, K, V, dO = (torch.randn(B, H, N, D, device="cuda", dtype=torch.bfloat16) for _ in range(4))
    ws = la.new_workspace(B, H, N, D, True, la.LA_BF16, True)
    O, g = la.la_forward(Q, K, V, True, workspace=ws)
    grads = la.la_backward(Q, K, V, O, dO, True, workspace=ws)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    floor = 8 * B * H * N * D * 2 + 4 * B * H * N
    assert peak <= 1.2 * floor, (peak, floor)
    del grads
