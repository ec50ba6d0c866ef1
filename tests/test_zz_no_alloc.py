"""la_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin given only input and output buffers by a framework that owns all allocation, code
that must not call cudaMalloc because it can block and synchronise the device) cannot hand the library a
workspace; this entry point uses a fixed device array inside the library instead.  The test calls it
through the C ABI, twice in a row on the same scratch, and compares each result with la_forward's on a
workspace allocated the usual way, within the parity tolerances of the other tests, and reads the
scratch's device status after each call.  It needs nothing that earlier tests leave behind, so it passes
alone in a fresh process or after the rest of the suite.
"""
import ctypes

import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # LA_NOALLOC_SCRATCH_BYTES in include/la.h


def _lib():
    from bwd_la_fwd_gb300 import la
    lib = la.load_library()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.la_forward_noalloc.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp]
    lib.la_forward_noalloc.restype = i
    lib.la_noalloc_get_status.argtypes = [vp]
    lib.la_noalloc_get_status.restype = i
    return lib


@pytest.mark.parametrize("dtype,D,causal", [("bf16", 128, 1), ("bf16", 128, 0), ("f32", 64, 1)])
def test_noalloc_forward_matches_la_forward_twice(dtype, D, causal):
    import torch
    from bwd_la_fwd_gb300 import la
    lib = _lib()
    B, H, N = 2, 3, 777
    x = inputs.generate(B, H, N, D, seed=55, dtype=dtype)
    Q, K, V = (U.to_device(x[n], dtype) for n in ("Q", "K", "V"))
    code = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    assert 0 < la.la_workspace_bytes(B, H, N, D, causal, code, False) <= SCRATCH_BYTES
    ws = la.new_workspace(B, H, N, D, causal, code, False)
    O_ref, g_ref = la.la_forward(Q, K, V, causal, workspace=ws)
    stream = torch.cuda.current_stream()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for call in range(2):
        O = torch.full_like(Q, float("nan"))
        g = torch.full((B, H, N), float("nan"), device=Q.device)
        rc = lib.la_forward_noalloc(p(Q), p(K), p(V), causal, p(O), p(g), B, H, N, D, code,
                                    ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, la.la_status_string(rc)
        # the device status of the scratch array: no bounded wait ran out in this call
        st = lib.la_noalloc_get_status(ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, la.la_status_string(st)
        for name, got, ref in (("O", O, O_ref), ("g", g, g_ref)):
            a, r = U.to_f64(got), U.to_f64(ref)
            U.assert_close(name, a, r, dtype)


def test_noalloc_rejects_problems_beyond_the_scratch():
    import torch
    from bwd_la_fwd_gb300 import la
    lib = _lib()
    B, H, N, D = 64, 16, 4096, 128  # needs far more than 32 MiB of state slots
    assert la.la_workspace_bytes(B, H, N, D, 1, la.LA_BF16, False) > SCRATCH_BYTES
    dummy = torch.empty(16, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.la_forward_noalloc(p, p, p, 1, p, None, B, H, N, D, la.LA_BF16, None)
    assert rc == 3  # LA_ERR_WORKSPACE, returned before anything is enqueued


def test_noalloc_rejects_bad_arguments_before_enqueuing():
    """An argument error is found on the host: the call returns LA_ERR_INVALID_ARG and the scratch's
    status word is untouched (a misaligned input pointer here)."""
    import torch
    from bwd_la_fwd_gb300 import la
    lib = _lib()
    B, H, N, D = 1, 2, 256, 128
    buf = torch.zeros(B * H * N * D + 8, device="cuda", dtype=torch.bfloat16)
    good = ctypes.c_void_p(buf.data_ptr())
    odd = ctypes.c_void_p(buf.data_ptr() + 2)  # not 16-byte aligned
    out = torch.empty(B * H * N * D, device="cuda", dtype=torch.bfloat16)
    rc = lib.la_forward_noalloc(odd, good, good, 1, ctypes.c_void_p(out.data_ptr()), None, B, H, N, D,
                                la.LA_BF16, None)
    assert rc == 1  # LA_ERR_INVALID_ARG
    assert lib.la_noalloc_get_status(None) == 0
