"""The index-checked build (LA_CHECKED): the same sources compiled so that every global-memory index a
kernel computes itself for a workspace array or the normaliser -- tensor-core path: slots of the
per-piece sums, per-chunk column sums, per-row statistics; CUDA-core path: segment states, row statistics
and their per-column partials -- is checked against the array's extent, a violation being recorded as
LA_ERR_BOUNDS instead of performed.  On odd and edge shapes of every configuration (bf16 D = 32 to 256 on
tensor cores, fp32 and bf16 D = 16 on CUDA cores, both masks, ragged tails, one row, several chunks and
heads per CTA; the causal reusing backward also as the single sweep, which reads the forward's kept g
and head totals) no index leaves its array (status LA_OK) and the results are bit-identical to the
product build's.
"""
import ctypes
import os

import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

# (dtype, B, H, N, D, causal, CTA cap or None)
CASES = [
    ("bf16", 1, 2, 1, 128, 1, None),
    ("bf16", 1, 3, 63, 128, 0, None),
    ("bf16", 2, 3, 300, 128, 1, None),
    ("bf16", 2, 3, 1000, 128, 1, 4),   # slices of several chunks, straddling heads
    ("bf16", 2, 3, 1000, 128, 0, 4),
    ("bf16", 2, 2, 257, 64, 1, 3),
    ("bf16", 1, 3, 129, 32, 0, None),
    ("bf16", 1, 2, 1, 256, 1, None),
    ("bf16", 2, 2, 300, 256, 1, 2),    # D = 256: several heads per CTA
    ("bf16", 1, 3, 129, 256, 0, None),
    ("f32", 2, 2, 700, 64, 1, None),   # CUDA-core kernels: several segments per head
    ("f32", 1, 2, 300, 128, 0, None),
    ("bf16", 2, 3, 513, 16, 1, None),
    ("f32", 1, 2, 1, 256, 1, None),
]
# the causal reusing backward forced to the single sweep (bf16, D = 128)
SWEEP_CASES = [
    ("bf16", 1, 2, 1, 128, 1, None),
    ("bf16", 2, 3, 300, 128, 1, 2),    # several heads per CTA
    ("bf16", 1, 2, 1000, 128, 1, None),
]


@pytest.fixture(scope="module")
def libs():
    from bwd_la_fwd_gb300 import build, la
    path = build.LIB_CHECKED
    if not os.path.exists(path):
        build.build(checked=True)
    return la.load_library(), la.open_library(path)


def _run(lib, t, B, H, N, D, causal, dt):
    """Forward, reusing backward and plain backward through the C ABI; returns (statuses, outputs)."""
    import torch
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nb = lib.la_workspace_bytes(B, H, N, D, causal, dt, 1)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    O = torch.empty_like(t["Q"])
    g = torch.empty(B, H, N, device="cuda")
    grads = [torch.empty_like(t["Q"]) for _ in range(6)]
    statuses = []
    assert lib.la_forward(p(t["Q"]), p(t["K"]), p(t["V"]), causal, p(O), p(g), B, H, N, D, dt, p(ws), nb, st) == 0
    statuses.append(lib.la_get_status(p(ws), st))
    assert lib.la_backward_with_forward_state(p(t["Q"]), p(t["K"]), p(t["V"]), p(O), p(t["dO"]), p(grads[0]),
                                              p(grads[1]), p(grads[2]), causal, B, H, N, D, dt, p(ws), nb, st) == 0
    statuses.append(lib.la_get_status(p(ws), st))
    assert lib.la_backward(p(t["Q"]), p(t["K"]), p(t["V"]), p(O), p(t["dO"]), p(grads[3]), p(grads[4]),
                           p(grads[5]), causal, B, H, N, D, dt, p(ws), nb, st) == 0
    statuses.append(lib.la_get_status(p(ws), st))
    torch.cuda.synchronize()
    return statuses, [O, g, *grads]


@pytest.mark.parametrize("dtype,B,H,N,D,causal,cap", CASES)
def test_checked_build_finds_no_index_out_of_range_and_matches(libs, monkeypatch, dtype, B, H, N, D, causal, cap):
    _check(libs, monkeypatch, dtype, B, H, N, D, causal, cap)


@pytest.mark.parametrize("dtype,B,H,N,D,causal,cap", SWEEP_CASES)
def test_checked_build_single_sweep(libs, monkeypatch, dtype, B, H, N, D, causal, cap):
    monkeypatch.setenv("LA_TC_SWEEP", "1")
    _check(libs, monkeypatch, dtype, B, H, N, D, causal, cap)


def _check(libs, monkeypatch, dtype, B, H, N, D, causal, cap):
    import torch
    if cap is not None:
        monkeypatch.setenv("LA_TC_MAX_CTAS", str(cap))
    x = inputs.generate(B, H, N, D, seed=90 + N + D, dtype=dtype)
    t = {n: U.to_device(x[n], dtype) for n in ("Q", "K", "V", "dO")}
    dt = 1 if dtype == "bf16" else 0
    product, checked = libs
    st_p, out_p = _run(product, t, B, H, N, D, causal, dt)
    st_c, out_c = _run(checked, t, B, H, N, D, causal, dt)
    assert st_p == [0, 0, 0]
    assert st_c == [0, 0, 0], [product.la_status_string(s).decode() for s in st_c]
    names = ["O", "g", "dQ (reuse)", "dK (reuse)", "dV (reuse)", "dQ", "dK", "dV"]
    for name, a, b in zip(names, out_p, out_c):
        assert torch.equal(a, b), name
