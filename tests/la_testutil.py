"""Helpers shared by the parity tests: move seeded inputs to the GPU, run the library, compare.

Tolerances (fixed for this method; the forward and backward are one rounding of an fp32-accumulated
result for bf16 I/O):
  * fp32 I/O: elementwise |x - r| / max(|r|, 1e-3 max|r|, 1e-6) <= 1e-5 per tensor;
  * bf16 I/O: max|x - r| / max(max|r|, 1e-3) <= 2e-2 per tensor (O, dQ, dK, dV);
  * normaliser (fp32 output in both cases): elementwise relative 1e-5 (fp32 I/O) or 1e-3 (bf16 I/O).
The absolute floors only matter where a reference tensor is exactly zero (dQ at N = 1 is 0 by the
definition); every tensor here is O(1) in scale (Q, K ~ N(0, 1/D), V, dO ~ N(0, 1)).
"""
from __future__ import annotations

import numpy as np

from bwd_la_fwd_gb300 import inputs

TOL = {"f32": 1e-5, "bf16": 2e-2}
TOL_G = {"f32": 1e-5, "bf16": 1e-3}


def to_device(arr: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def run_library(x: dict, dtype: str, causal: bool, backward: bool = True):
    """Forward (and backward, fed the library's own O) on the GPU; returns float64 numpy arrays."""
    import torch
    from bwd_la_fwd_gb300 import la
    Q, K, V = (to_device(x[n], dtype) for n in ("Q", "K", "V"))
    B, H, N, D = Q.shape
    ws = la.new_workspace(B, H, N, D, causal, la.LA_BF16 if dtype == "bf16" else la.LA_F32, backward)
    O, g = la.la_forward(Q, K, V, causal, workspace=ws)
    out = {"O": O, "g": g}
    if backward:
        dO = to_device(x["dO"], dtype)
        dQ, dK, dV = la.la_backward(Q, K, V, O, dO, causal, workspace=ws)
        out.update(dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    st = la.la_get_status(ws)
    assert st == 0, f"device status {la.la_status_string(st)}"
    return {k: to_f64(v) for k, v in out.items()}


def err_rel_elem(x: np.ndarray, r: np.ndarray) -> float:
    floor = 1e-3 * float(np.max(np.abs(r))) if r.size else 0.0
    den = np.maximum(np.abs(r), max(floor, 1e-6))
    return float(np.max(np.abs(x - r) / den)) if r.size else 0.0


def err_norm_maxabs(x: np.ndarray, r: np.ndarray) -> float:
    m = float(np.max(np.abs(r))) if r.size else 0.0
    return float(np.max(np.abs(x - r)) / max(m, 1e-3)) if r.size else 0.0


def tensor_error(x, r, dtype: str) -> float:
    return err_rel_elem(x, r) if dtype == "f32" else err_norm_maxabs(x, r)


def assert_close(name: str, x, r, dtype: str):
    if name == "g":
        e = err_rel_elem(x, r)
        tol = TOL_G[dtype]
    else:
        e = tensor_error(x, r, dtype)
        tol = TOL[dtype]
    assert np.all(np.isfinite(x)), f"{name}: non-finite values"
    assert e <= tol, f"{name}: error {e:.3e} > {tol:.1e} ({dtype})"
    return e


def stored_to_f64(x: dict, dtype: str) -> dict:
    return {k: inputs.to_f64(v, dtype) for k, v in x.items()}
