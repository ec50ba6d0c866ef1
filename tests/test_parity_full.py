"""GPU parity at the full workload sizes, on the launch configuration the benchmark times.

The explicit oracle costs O(N^2 D) per head, so at these sizes it checks sampled outputs it can compute
one row at a time (O_i, g_i, dQ_i cost O(N D) each; dK_j, dV_j cost O((N - j) N D), so they are sampled
near the end of causal heads).  Whole heads are also checked against the fp64 running-state form (itself
pinned to the explicit oracle at small sizes).  Sizes: the paper's standalone shape (B=4 H=16 N=4096
D=128, causal and non-causal), the head-size sweep (D = 32, 64, 256 at N = 4096), the sequence-length
sweep (N = 1024 ... 65536 at D = 128) and two layers of the 1.4B-class step (B=8 H=16 N=2048 D=128).
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


def _check_full(oracle_lib, B, H, N, D, seed, causal, layer=0, layers=1):
    import torch
    from bwd_la_fwd_gb300 import la
    x = inputs.generate(B, H, N, D, seed, dtype="bf16", layers=layers)
    if layers > 1:
        x = x[layer]
    Q, K, V, dO = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V", "dO"))
    ws = la.new_workspace(B, H, N, D, causal, la.LA_BF16, True)
    O, g = la.la_forward(Q, K, V, causal, workspace=ws)
    dQ, dK, dV = la.la_backward(Q, K, V, O, dO, causal, workspace=ws)
    torch.cuda.synchronize()
    assert la.la_get_status(ws) == 0
    out = {"O": O, "g": g, "dQ": dQ, "dK": dK, "dV": dV}
    heads = [0, B * H - 1]
    f = _heads_f64(x, heads, B, H, N, D)
    got = {k: v.reshape(B * H, N, -1)[heads].double().cpu().numpy().reshape(1, len(heads), N, -1)
           for k, v in out.items()}
    got["g"] = got["g"].reshape(1, len(heads), N)

    # whole heads against the fp64 running-state form
    rO, rg = oracle_lib.prefix_forward(f["Q"], f["K"], f["V"], causal)
    rdQ, rdK, rdV = oracle_lib.prefix_backward(f["Q"], f["K"], f["V"], f["dO"], causal)
    for name, ref in (("O", rO), ("g", rg), ("dQ", rdQ), ("dK", rdK), ("dV", rdV)):
        U.assert_close(name, got[name], ref, "bf16")

    # sampled rows against the explicit definition
    rows = _sample_rows(N)
    flat = np.array([h * N + r for h in range(len(heads)) for r in rows])
    sO, sg = oracle_lib.forward_rows(f["Q"], f["K"], f["V"], causal, flat)
    sdQ = oracle_lib.dq_rows(f["Q"], f["K"], f["V"], f["dO"], causal, flat)
    U.assert_close("O", got["O"].reshape(-1, D)[flat], sO, "bf16")
    U.assert_close("g", got["g"].reshape(-1)[flat], sg, "bf16")
    U.assert_close("dQ", got["dQ"].reshape(-1, D)[flat], sdQ, "bf16")
    kv_rows = [N - 3, N - 2, N - 1] if causal else [0, N // 2, N - 1]
    kflat = np.array([h * N + r for h in range(len(heads)) for r in kv_rows if r >= 0])
    sdK, sdV = oracle_lib.dkdv_rows(f["Q"], f["K"], f["V"], f["dO"], causal, kflat)
    U.assert_close("dK", got["dK"].reshape(-1, D)[kflat], sdK, "bf16")
    U.assert_close("dV", got["dV"].reshape(-1, D)[kflat], sdV, "bf16")


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
