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
