"""Thin ctypes binding over the C ABI declared in include/la.h.

Argument marshalling only: every step of the computation runs in the CUDA library.  PyTorch supplies
device memory and the current stream.  If the compiled library is missing, ``load_library`` raises;
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

LA_F32 = 0
LA_BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libla_gb300.so"
_lock = threading.Lock()
_lib = None

_STATUS = {0: "LA_OK", 1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_WORKSPACE", 4: "LA_ERR_CUDA",
           5: "LA_ERR_TIMEOUT", 6: "LA_ERR_BOUNDS", 7: "LA_ERR_STATE"}


class LAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {la_status_string(status)} ({status})")


def library_path() -> str:
    return os.path.join(_HERE, LIB_NAME)


def load_library():
    """Load the compiled CUDA library (built by ``bwd_la_fwd_gb300.build``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: run `python -m bwd_la_fwd_gb300.build` "
                               "(or __graft_entry__.build()); there is no CPU fallback")
        _lib = open_library(path)
        return _lib


def open_library(path: str):
    """A ctypes handle on a build of the library at `path`, with every entry point's C signature set
    (load_library() opens the product build with it; the tests also open the index-checked build)."""
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.la_version.argtypes = []
    lib.la_version.restype = i
    lib.la_launch_count.argtypes = []
    lib.la_launch_count.restype = ctypes.c_ulonglong
    lib.la_status_string.argtypes = [i]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.la_workspace_bytes.restype = sz
    lib.la_forward.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp, sz, vp]
    lib.la_forward.restype = i
    lib.la_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
    lib.la_backward.restype = i
    lib.la_backward_with_forward_state.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
    lib.la_backward_with_forward_state.restype = i
    lp = ctypes.POINTER(ctypes.c_longlong)
    lib.la_forward_strided.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, lp, vp, sz, vp]
    lib.la_forward_strided.restype = i
    lib.la_backward_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, lp, i, vp, sz, vp]
    lib.la_backward_strided.restype = i
    lib.la_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
    lib.la_decode_step.restype = i
    lib.la_state_append.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.la_state_append.restype = i
    lib.la_get_status.argtypes = [vp, vp]
    lib.la_get_status.restype = i
    lib.la_forward_noalloc.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, i, vp]
    lib.la_forward_noalloc.restype = i
    lib.la_noalloc_get_status.argtypes = [vp]
    lib.la_noalloc_get_status.restype = i
    return lib


def la_status_string(status: int) -> str:
    if _lib is not None:
        return _lib.la_status_string(int(status)).decode()
    return _STATUS.get(int(status), "LA_UNKNOWN_STATUS")


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _shape(Q):
    if Q.dim() != 4:
        raise ValueError(f"expected a [B, H, N, D] tensor, got shape {tuple(Q.shape)}")
    return tuple(int(s) for s in Q.shape)


def _check_like(Q, *others):
    for t in (Q, *others):
        if t is None:
            continue
        if t.shape != Q.shape or t.dtype != Q.dtype or t.device != Q.device:
            raise ValueError("all [B,H,N,D] tensors must share shape, dtype and device")
        if t.stride(-1) != 1:
            raise ValueError("the D elements of each row must be contiguous (stride(-1) == 1)")


def _strides(*ts):
    """(batch, head, row) element strides of each [B,H,N,D] view, as the strided entry points take them."""
    vals = [int(x) for t in ts for x in t.stride()[:3]]
    return (ctypes.c_longlong * len(vals))(*vals)


def la_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load_library().la_launch_count())


def la_workspace_bytes(B: int, H: int, N: int, D: int, causal: bool, dtype: int, backward: bool) -> int:
    return int(load_library().la_workspace_bytes(B, H, N, D, int(bool(causal)), int(dtype), int(bool(backward))))


def new_workspace(B: int, H: int, N: int, D: int, causal: bool, dtype: int, backward: bool, device="cuda"):
    """Zero-filled device workspace of the size the library asks for (torch owns it)."""
    import torch
    n = la_workspace_bytes(B, H, N, D, causal, dtype, backward)
    if n == 0:
        raise LAError(1, "la_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def la_forward(Q, K, V, causal: bool, O=None, normaliser=None, workspace=None, stream=None):
    """O, g = la_forward(Q, K, V, causal): normalised linear attention forward on [B,H,N,D] tensors.

    The tensors may be strided views (a [B,N,H,D] tensor permuted to [B,H,N,D], a slice of a fused QKV
    projection) as long as each row's D elements are contiguous; they go to the library as they are."""
    import torch
    B, H, N, D = _shape(Q)
    _check_like(Q, K, V, O)
    dt = _dtype_code(Q)
    if O is None:
        O = torch.empty_like(Q)
    if normaliser is None:
        normaliser = torch.empty((B, H, N), dtype=torch.float32, device=Q.device)
    if workspace is None:
        workspace = new_workspace(B, H, N, D, causal, dt, False, Q.device)
    st = load_library().la_forward_strided(_ptr(Q), _ptr(K), _ptr(V), int(bool(causal)), _ptr(O), _ptr(normaliser),
                                           B, H, N, D, dt, _strides(Q, K, V, O), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != 0:
        raise LAError(st, "la_forward")
    return O, normaliser


def la_backward(Q, K, V, O, dO, causal: bool, dQ=None, dK=None, dV=None, workspace=None, stream=None,
                reuse_forward_state: bool = False):
    """dQ, dK, dV = la_backward(Q, K, V, O, dO, causal): gradients of sum(dO * O).

    With ``reuse_forward_state`` the call is la_backward_with_forward_state: it takes the per-piece state
    sums that the last la_forward on ``workspace`` (same K, V, shape) left there instead of recomputing
    them; the workspace must then be given (and sized for the backward at that forward)."""
    import torch
    B, H, N, D = _shape(Q)
    _check_like(Q, K, V, O, dO, dQ, dK, dV)
    dt = _dtype_code(Q)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(Q) if dK is None else dK
    dV = torch.empty_like(Q) if dV is None else dV
    if workspace is None:
        if reuse_forward_state:
            raise ValueError("reuse_forward_state needs the workspace the forward ran with")
        workspace = new_workspace(B, H, N, D, causal, dt, True, Q.device)
    st = load_library().la_backward_strided(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV),
                                            int(bool(causal)), B, H, N, D, dt, _strides(Q, K, V, O, dO, dQ, dK, dV),
                                            int(bool(reuse_forward_state)), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if st != 0:
        raise LAError(st, "la_backward_with_forward_state" if reuse_forward_state else "la_backward")
    return dQ, dK, dV


def la_get_status(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status recorded in the workspace."""
    return int(load_library().la_get_status(_ptr(workspace), _stream_ptr(stream)))


def la_forward_noalloc(Q, K, V, causal: bool, O=None, normaliser=None, stream=None):
    """The forward without a workspace argument: the library's fixed scratch array on the current device
    serves instead (for callers that cannot allocate device memory).  Returns (O, normaliser)."""
    import torch
    B, H, N, D = _shape(Q)
    _check_like(Q, K, V)
    if O is None:
        O = torch.empty_like(Q)
    if normaliser is None:
        normaliser = torch.empty((B, H, N), device=Q.device, dtype=torch.float32)
    st = load_library().la_forward_noalloc(_ptr(Q), _ptr(K), _ptr(V), int(bool(causal)), _ptr(O), _ptr(normaliser),
                                           B, H, N, D, _dtype_code(Q), _stream_ptr(stream))
    if st != 0:
        raise LAError(st, "la_forward_noalloc")
    return O, normaliser


def la_noalloc_get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status of the fixed scratch array."""
    return int(load_library().la_noalloc_get_status(_stream_ptr(stream)))


class DecodeState:
    """The carried state of the recurrent (decode) form, per (b, h): S [B,H,D,D], z [B,H,D], a [B,H,D] of
    the accumulator type (float32 for bf16 tokens, float64 for float32 tokens) and the count n (int32
    [B,H]).  Zero-filled is the empty state; the library updates the tensors in place."""

    def __init__(self, B: int, H: int, D: int, token_dtype, device="cuda"):
        import torch
        acc = torch.float32 if token_dtype == torch.bfloat16 else torch.float64
        if token_dtype not in (torch.bfloat16, torch.float32):
            raise TypeError(f"unsupported dtype {token_dtype}: use torch.bfloat16 or torch.float32")
        self.B, self.H, self.D, self.token_dtype = B, H, D, token_dtype
        self.S = torch.zeros((B, H, D, D), dtype=acc, device=device)
        self.z = torch.zeros((B, H, D), dtype=acc, device=device)
        self.a = torch.zeros((B, H, D), dtype=acc, device=device)
        self.n = torch.zeros((B, H), dtype=torch.int32, device=device)

    def _args(self):
        return _ptr(self.S), _ptr(self.z), _ptr(self.a), _ptr(self.n)


def la_decode_step(state: DecodeState, q, k, v, o=None, normaliser=None, stream=None):
    """o, g = la_decode_step(state, q, k, v): append one token per (b, h) ([B,H,D] tensors) to ``state``
    and return its output and normaliser (row n - 1 of the causal forward over the tokens taken so far)."""
    import torch
    if q.dim() != 3 or tuple(q.shape) != (state.B, state.H, state.D):
        raise ValueError(f"expected [B, H, D] = {(state.B, state.H, state.D)} tokens, got {tuple(q.shape)}")
    for t in (k, v, o):
        if t is not None and (t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous()):
            raise ValueError("q, k, v, o must share shape and dtype and be contiguous")
    if q.dtype != state.token_dtype:
        raise ValueError("token dtype does not match the state")
    o = torch.empty_like(q) if o is None else o
    if normaliser is None:
        normaliser = torch.empty((state.B, state.H), dtype=torch.float32, device=q.device)
    st = load_library().la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(normaliser), *state._args(),
                                       state.B, state.H, state.D, _dtype_code(q), _stream_ptr(stream))
    if st != 0:
        raise LAError(st, "la_decode_step")
    return o, normaliser


def la_state_append(state: DecodeState, K, V, stream=None):
    """Append N tokens per (b, h) ([B,H,N,D] tensors) to ``state``: S += K^T V, z += sum k, a += sum v,
    n += N."""
    B, H, N, D = _shape(K)
    _check_like(K, V)
    if (B, H, D) != (state.B, state.H, state.D) or K.dtype != state.token_dtype:
        raise ValueError("K, V do not match the state's B, H, D and token dtype")
    st = load_library().la_state_append(_ptr(K), _ptr(V), *state._args(), B, H, N, D, _dtype_code(K),
                                        _stream_ptr(stream))
    if st != 0:
        raise LAError(st, "la_state_append")
    return state
