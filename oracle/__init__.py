"""fp64 CPU oracle for normalised linear attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline and ``--impl
reference`` legs) may import this package.  The CUDA library never imports, links or calls it, and it
imports nothing from the library.

Two independent C implementations live here, compiled with plain ``gcc`` into ``liblaoracle.so``:

* ``la_oracle.c`` -- the explicit O(N^2 D) definition (normalised weights formed row by row), and
* ``la_prefix.c`` -- the O(N D^2) running-state form of the same definition, used to pin the first.

Source: "Transformer Based Linear Attention with Optimized GPU Kernel Implementation" (Gerami &
Duraiswami, arXiv 2510.21956); sciencestack.ai page, TL;DR (forward/backward formulation,
normalisation scheme, analytical gradients, O(N D^2) time, O(N D) memory).  The pages print no formula;
the reading implemented is W_ij = m_ij (c + q_i . k_j), g_i = sum_j W_ij, O_i = sum_j W_ij v_j / g_i,
with c = 1 unless a test sets it.

Every entry point takes and returns float64 numpy arrays laid out [B, H, N, D] (normaliser [B, H, N]).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = ("la_oracle.c", "la_prefix.c")
_LIB_PATH = os.path.join(_HERE, "liblaoracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into ``oracle/liblaoracle.so`` (gcc, fp64, no fast-math)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    if not force and os.path.exists(_LIB_PATH):
        lib_m = os.path.getmtime(_LIB_PATH)
        if all(os.path.getmtime(s) <= lib_m for s in srcs):
            return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, *srcs, "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        LP = ctypes.POINTER(ctypes.c_long)
        I = ctypes.c_int
        Dbl = ctypes.c_double
        lib.la_oracle_forward.argtypes = [P, P, P, L, L, L, L, I, Dbl, P, P, I]
        lib.la_oracle_backward.argtypes = [P, P, P, P, L, L, L, L, I, Dbl, P, P, P, I]
        lib.la_oracle_weights.argtypes = [P, P, L, L, I, Dbl, P]
        lib.la_oracle_forward_rows.argtypes = [P, P, P, L, L, L, L, I, Dbl, LP, L, P, P, I]
        lib.la_oracle_dq_rows.argtypes = [P, P, P, P, L, L, L, L, I, Dbl, LP, L, P, I]
        lib.la_oracle_dkdv_rows.argtypes = [P, P, P, P, L, L, L, L, I, Dbl, LP, L, P, P, I]
        lib.la_prefix_forward.argtypes = [P, P, P, L, L, L, L, I, Dbl, P, P, I]
        lib.la_prefix_backward.argtypes = [P, P, P, P, L, L, L, L, I, Dbl, P, P, P, I]
        for fn in ("la_oracle_forward", "la_oracle_backward", "la_oracle_weights", "la_oracle_forward_rows",
                   "la_oracle_dq_rows", "la_oracle_dkdv_rows", "la_prefix_forward", "la_prefix_backward"):
            getattr(lib, fn).restype = ctypes.c_int
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape4(x: np.ndarray):
    if x.ndim != 4:
        raise ValueError(f"expected a [B, H, N, D] array, got shape {x.shape}")
    return x.shape


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed (rc={rc})")


def forward(Q, K, V, causal: bool, c: float = 1.0, threads: int = 0):
    """Explicit forward. Returns (O [B,H,N,D], g [B,H,N]) in float64."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, D = _shape4(Q)
    O = np.empty_like(Q)
    g = np.empty((B, H, N), dtype=np.float64)
    _check(_load().la_oracle_forward(_ptr(Q), _ptr(K), _ptr(V), B, H, N, D, int(causal), c, _ptr(O), _ptr(g),
                                     threads), "forward")
    return O, g


def backward(Q, K, V, dO, causal: bool, c: float = 1.0, threads: int = 0):
    """Explicit backward of L = sum dO * O. Returns (dQ, dK, dV) in float64."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, D = _shape4(Q)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    _check(_load().la_oracle_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, D, int(causal), c, _ptr(dQ),
                                      _ptr(dK), _ptr(dV), threads), "backward")
    return dQ, dK, dV


def weights(q, k, causal: bool, c: float = 1.0):
    """Normalised weights A (N x N) of one head, from q, k of shape [N, D]."""
    q, k = _f64(q), _f64(k)
    N, D = q.shape
    A = np.empty((N, N), dtype=np.float64)
    _check(_load().la_oracle_weights(_ptr(q), _ptr(k), N, D, int(causal), c, _ptr(A)), "weights")
    return A


def _rows(rows) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1)).astype(np.dtype("l"))


def forward_rows(Q, K, V, causal: bool, rows, c: float = 1.0, threads: int = 0):
    """O_i and g_i at flat row indices ((b*H + h)*N + i). Returns (O_rows [R,D], g_rows [R])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, D = _shape4(Q)
    r = _rows(rows)
    O = np.empty((r.size, D), dtype=np.float64)
    g = np.empty(r.size, dtype=np.float64)
    lib = _load()
    _check(lib.la_oracle_forward_rows(_ptr(Q), _ptr(K), _ptr(V), B, H, N, D, int(causal), c,
                                      r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), r.size, _ptr(O), _ptr(g),
                                      threads), "forward_rows")
    return O, g


def dq_rows(Q, K, V, dO, causal: bool, rows, c: float = 1.0, threads: int = 0):
    """dQ_i at flat row indices. Returns [R, D]."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, D = _shape4(Q)
    r = _rows(rows)
    dQ = np.empty((r.size, D), dtype=np.float64)
    _check(_load().la_oracle_dq_rows(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, D, int(causal), c,
                                     r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), r.size, _ptr(dQ), threads),
           "dq_rows")
    return dQ


def dkdv_rows(Q, K, V, dO, causal: bool, rows, c: float = 1.0, threads: int = 0):
    """dK_j, dV_j at flat row indices (cost O((N-j) N D) each when causal). Returns ([R,D], [R,D])."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, D = _shape4(Q)
    r = _rows(rows)
    dK = np.empty((r.size, D), dtype=np.float64)
    dV = np.empty((r.size, D), dtype=np.float64)
    _check(_load().la_oracle_dkdv_rows(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, D, int(causal), c,
                                       r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), r.size, _ptr(dK), _ptr(dV),
                                       threads), "dkdv_rows")
    return dK, dV


def prefix_forward(Q, K, V, causal: bool, c: float = 1.0, threads: int = 0):
    """O(N D^2) running-state forward. Returns (O, g) in float64."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, D = _shape4(Q)
    O = np.empty_like(Q)
    g = np.empty((B, H, N), dtype=np.float64)
    _check(_load().la_prefix_forward(_ptr(Q), _ptr(K), _ptr(V), B, H, N, D, int(causal), c, _ptr(O), _ptr(g),
                                     threads), "prefix_forward")
    return O, g


def prefix_backward(Q, K, V, dO, causal: bool, c: float = 1.0, threads: int = 0):
    """O(N D^2) running-state backward. Returns (dQ, dK, dV) in float64."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, D = _shape4(Q)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    _check(_load().la_prefix_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, N, D, int(causal), c, _ptr(dQ),
                                      _ptr(dK), _ptr(dV), threads), "prefix_backward")
    return dQ, dK, dV


# ---------------------------------------------------------------- recurrent (decode) form ---
# The causal forward written as a recurrence over tokens.  The state of the tokens taken so far is
# S = sum_j k_j v_j^T (S[d][e] = sum_j k_j[d] v_j[e]), z = sum_j k_j, a = sum_j v_j and their count n:
# the d x d state that accumulates one outer product k_t v_t^T per time step (cloud.baidu.com article
# 9404082, section 2, the state-matrix recurrence), with the normalisation of the reading above, so that
# token t's output g_t = c n + q_t . z, o_t = (c a + S^T q_t) / g_t equals row t of the causal forward.
# Plain numpy in float64; every array is [B, H, ...].

def state_append(S, z, a, n, K, V):
    """State after appending tokens K, V ([B,H,T,D]) to (S [B,H,D,D], z [B,H,D], a [B,H,D], n [B,H])."""
    K, V = _f64(K), _f64(V)
    S2 = _f64(S) + np.einsum("bhtd,bhte->bhde", K, V)
    z2 = _f64(z) + K.sum(axis=2)
    a2 = _f64(a) + V.sum(axis=2)
    n2 = np.asarray(n, dtype=np.int64) + K.shape[2]
    return S2, z2, a2, n2


def decode_step(S, z, a, n, q, k, v, c: float = 1.0):
    """One token per (b, h) (q, k, v [B,H,D]): appends (k, v), then g = c n + q . z and
    o = (c a + S^T q) / g on the new state.  Returns (o [B,H,D], g [B,H], S, z, a, n)."""
    S2, z2, a2, n2 = state_append(S, z, a, n, _f64(k)[:, :, None, :], _f64(v)[:, :, None, :])
    q = _f64(q)
    g = c * n2 + np.einsum("bhd,bhd->bh", q, z2)
    o = (c * a2 + np.einsum("bhde,bhd->bhe", S2, q)) / g[..., None]
    return o, g, S2, z2, a2, n2


def empty_state(B: int, H: int, D: int):
    """The state of no tokens."""
    return (np.zeros((B, H, D, D)), np.zeros((B, H, D)), np.zeros((B, H, D)), np.zeros((B, H), dtype=np.int64))
