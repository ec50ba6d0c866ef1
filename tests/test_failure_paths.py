"""Failure handling on the device, made to happen without faulting the GPU.

Every barrier wait in the tensor-core kernels is bounded.  When one runs out, the kernel records
LA_ERR_TIMEOUT in the workspace status word, every role of the CTA stops, the producer lets the copies it
has already issued land, and TMEM is released before the CTA exits -- so the context stays usable and the
next call computes normally.  Two test hooks of the sums kernel make that happen on purpose: with
LA_TEST_DROP_LOAD = k, CTA 0 issues no load at all for its k-th chunk (no expected-bytes arrive and no
copy), so the MMA issuer's wait for that stage can only run out; LA_TEST_WAIT_NS shortens every wait's
bound from 2 s.  No arrive is dropped for a copy that was issued, and nothing faults, traps or spins
without a bound.
"""
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


def _forward(x, ws, causal):
    import torch
    from bwd_la_fwd_gb300 import la
    Q, K, V = (U.to_device(x[n], "bf16") for n in ("Q", "K", "V"))
    O, g = la.la_forward(Q, K, V, causal, workspace=ws)
    torch.cuda.synchronize()
    return O, g


@pytest.mark.parametrize("causal", [1, 0])
def test_wait_that_runs_out_reports_timeout_and_the_next_call_is_exact(monkeypatch, causal):
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, N, D = 2, 2, 2048, 128
    x = inputs.generate(B, H, N, D, seed=21, dtype="bf16")
    # four CTAs: each walks 16 chunks, so the dropped load sits mid-slice with later copies in flight
    monkeypatch.setenv("LA_TC_MAX_CTAS", "4")
    ws_ref = la.new_workspace(B, H, N, D, causal, la.LA_BF16, False)
    O_ref, g_ref = _forward(x, ws_ref, causal)
    assert la.la_get_status(ws_ref) == 0

    ws = la.new_workspace(B, H, N, D, causal, la.LA_BF16, False)
    monkeypatch.setenv("LA_TEST_WAIT_NS", "20000000")  # 20 ms
    monkeypatch.setenv("LA_TEST_DROP_LOAD", "5")
    _forward(x, ws, causal)  # the call itself is accepted: the condition is found on the device
    st = la.la_get_status(ws)
    assert st == 5, la.la_status_string(st)  # LA_ERR_TIMEOUT
    assert la.la_get_status(ws) == 0  # reading the status cleared it

    # the same workspace and device, hooks off: bit-identical to a call that never saw the failure
    monkeypatch.delenv("LA_TEST_WAIT_NS")
    monkeypatch.delenv("LA_TEST_DROP_LOAD")
    O2, g2 = _forward(x, ws, causal)
    assert la.la_get_status(ws) == 0
    assert torch.equal(O2, O_ref)
    assert torch.equal(g2, g_ref)

