"""The Python binding's own argument checks, on CPU: they raise before any library call or GPU work."""
import pytest


def test_rows_must_be_contiguous():
    import torch
    from bwd_la_fwd_gb300 import la
    Q = torch.empty(1, 2, 8, 64, dtype=torch.bfloat16)
    bad = torch.as_strided(torch.empty(2 * 8 * 64 * 2, dtype=torch.bfloat16), (1, 2, 8, 64), (2048, 1024, 128, 2))
    with pytest.raises(ValueError, match="contiguous"):
        la.la_forward(Q, bad, Q, True)


def test_operands_must_share_shape_and_dtype():
    import torch
    from bwd_la_fwd_gb300 import la
    Q = torch.empty(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        la.la_forward(Q, torch.empty(1, 2, 9, 64, dtype=torch.bfloat16), Q, True)
    with pytest.raises(ValueError, match="dtype"):
        la.la_backward(Q, Q, Q, Q, Q.float(), True)


def test_unsupported_dtype_is_refused():
    import torch
    from bwd_la_fwd_gb300 import la
    Q = torch.empty(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        la.la_forward(Q, Q, Q, True)


def test_decode_state_checks():
    import torch
    from bwd_la_fwd_gb300 import la
    with pytest.raises(TypeError):
        la.DecodeState(1, 2, 64, torch.float16, device="cpu")
    st = la.DecodeState(1, 2, 64, torch.bfloat16, device="cpu")
    assert st.S.dtype == torch.float32 and st.S.shape == (1, 2, 64, 64) and st.n.dtype == torch.int32
    assert la.DecodeState(1, 2, 64, torch.float32, device="cpu").S.dtype == torch.float64
    q = torch.empty(1, 2, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="expected"):
        la.la_decode_step(st, q, q, q)
    K = torch.empty(1, 2, 5, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="match"):
        la.la_state_append(st, K, K)


def test_missing_library_fails_loudly(monkeypatch):
    """Without the compiled CUDA library every entry raises: there is no CPU or torch fallback."""
    import torch
    from bwd_la_fwd_gb300 import la
    monkeypatch.setattr(la, "_lib", None)
    monkeypatch.setattr(la, "library_path", lambda: "/nonexistent/liblagb300.so")
    Q = torch.empty(1, 2, 8, 64, dtype=torch.bfloat16)
    for call in (lambda: la.la_forward(Q, Q, Q, True),
                 lambda: la.la_backward(Q, Q, Q, Q, Q, True),
                 lambda: la.la_workspace_bytes(1, 2, 8, 64, True, la.LA_BF16, True),
                 lambda: la.la_launch_count()):
        with pytest.raises(RuntimeError, match="no CPU fallback"):
            call()


def test_product_package_never_imports_the_oracle():
    """The oracle is test infrastructure: no module of the product package imports or loads it."""
    import os
    import re
    pkg = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bwd_la_fwd_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b)|liblaoracle", re.M)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(root, f), encoding="utf-8") as fh:
                    assert not pat.search(fh.read()), f
