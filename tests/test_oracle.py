"""Pins of the fp64 oracle to facts other than itself (CPU only).

The oracle implements the reading W_ij = m_ij (c + q_i . k_j), g_i = sum_j W_ij, O_i = sum_j W_ij v_j / g_i
of "Transformer Based Linear Attention with Optimized GPU Kernel Implementation" (sciencestack.ai page,
TL;DR) and the exact gradients of L = sum dO . O.  Each test below would fail on a plausible slip in
it: a dropped term (the constant c, the -delta_i in dW), a wrong sign, an index off by one on the
causal mask, or a transposed operand (q_j . k_i).

  * hand-worked D = 1 example (tests/golden/d1_n3_worked.txt), causal and non-causal;
  * the independent O(N D^2) running-state form;
  * central finite differences of L for every entry of Q, K, V (the "analytical gradients");
  * invariants: rows of the normalised weights sum to one; causal outputs ignore future tokens;
    shifting V by a constant row shifts O by it; O is linear in V;
  * closed forms: K = 0 or Q = 0 gives (prefix) means of V, N = 1 gives O = V, dQ = dK = 0, dV = dO, c = 0 with D = 1
    gives a q-independent ratio, and the matching gradients;
  * the recurrent (decode) form: token by token it reproduces the hand-worked causal values and the
    explicit causal rows, and a block append followed by decoding continues the forward.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from bwd_la_fwd_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "d1_n3_worked.txt")


def _tiny(seed=0, B=1, H=2, N=64, D=16):
    t = inputs.generate(B, H, N, D, seed, dtype="f32")
    return {k: inputs.to_f64(v, "f32") for k, v in t.items()}


def _rel(x, r):
    """Max abs difference over max(max |r|, 1): the tensors here are O(1) in scale."""
    return np.max(np.abs(x - r)) / max(np.max(np.abs(r)), 1.0)


# --------------------------------------------------------------------------------- golden ---

def _load_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, name, row, val = line.split()
            vals[(a, name, int(row))] = float(Fraction(val))
    return vals


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("form", ["explicit", "prefix"])
def test_golden_d1_worked_example(oracle_lib, causal, form):
    gv = _load_golden()
    arr = {n: np.array([gv[("input", n, i)] for i in range(3)]).reshape(1, 1, 3, 1) for n in ("q", "k", "v", "dO")}
    if form == "explicit":
        O, g = oracle_lib.forward(arr["q"], arr["k"], arr["v"], causal)
        dQ, dK, dV = oracle_lib.backward(arr["q"], arr["k"], arr["v"], arr["dO"], causal)
    else:
        O, g = oracle_lib.prefix_forward(arr["q"], arr["k"], arr["v"], causal)
        dQ, dK, dV = oracle_lib.prefix_backward(arr["q"], arr["k"], arr["v"], arr["dO"], causal)
    got = {"O": O, "g": g, "dQ": dQ, "dK": dK, "dV": dV}
    for name, x in got.items():
        x = x.reshape(-1)
        for i in range(3):
            want = gv[(str(causal), name, i)]
            assert abs(x[i] - want) <= 1e-13 * max(1.0, abs(want)), (name, i, x[i], want)


# ---------------------------------------------------------------------- explicit vs prefix ---

@pytest.mark.parametrize("c", [1.0, 2.0])
@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("shape", [(1, 2, 64, 16), (1, 1, 1, 4), (2, 1, 7, 3), (1, 3, 33, 8), (1, 1, 40, 1)])
def test_explicit_matches_prefix_form(oracle_lib, causal, shape, c):
    """Both forms at the library's c = 1 and at c = 2, so that every place c enters either form (the
    weights, the normaliser, the a and e terms of O and dV) is compared."""
    B, H, N, D = shape
    x = _tiny(seed=11 + N, B=B, H=H, N=N, D=D)
    O, g = oracle_lib.forward(x["Q"], x["K"], x["V"], causal, c=c)
    Op, gp = oracle_lib.prefix_forward(x["Q"], x["K"], x["V"], causal, c=c)
    assert _rel(O, Op) < 1e-12 and _rel(g, gp) < 1e-12
    gr = oracle_lib.backward(x["Q"], x["K"], x["V"], x["dO"], causal, c=c)
    grp = oracle_lib.prefix_backward(x["Q"], x["K"], x["V"], x["dO"], causal, c=c)
    for a, b in zip(gr, grp):
        assert _rel(a, b) < 1e-12


# ------------------------------------------------------------------------ finite differences ---

@pytest.mark.parametrize("causal", [1, 0])
def test_gradients_match_central_differences(oracle_lib, causal):
    """Every entry of Q, K, V of the tiny case (B=1, H=2, N=64, D=16): |FD - analytic| <= 1e-7 rel."""
    x = _tiny(seed=0)
    Q, K, V, dO = x["Q"], x["K"], x["V"], x["dO"]
    dQ, dK, dV = oracle_lib.backward(Q, K, V, dO, causal)
    h = 1e-6

    def loss(Q_, K_, V_):
        return float(np.sum(oracle_lib.forward(Q_, K_, V_, causal, threads=1)[0] * dO))

    for name, grad in (("Q", dQ), ("K", dK), ("V", dV)):
        fd = np.empty_like(grad)
        base = {"Q": Q, "K": K, "V": V}
        flat = base[name].reshape(-1)
        for idx in range(flat.size):
            orig = flat[idx]
            flat[idx] = orig + h
            lp = loss(base["Q"], base["K"], base["V"])
            flat[idx] = orig - h
            lm = loss(base["Q"], base["K"], base["V"])
            flat[idx] = orig
            fd.reshape(-1)[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad)) / np.max(np.abs(grad))
        assert err < 1e-7, (name, err)


# ------------------------------------------------------------------------------- invariants ---

@pytest.mark.parametrize("causal", [1, 0])
def test_normalised_weights_rows_sum_to_one(oracle_lib, causal):
    x = _tiny(seed=3)
    for h in range(2):
        A = oracle_lib.weights(x["Q"][0, h], x["K"][0, h], causal)
        assert np.max(np.abs(A.sum(axis=1) - 1.0)) < 1e-13
        if causal:
            assert np.all(np.triu(A, 1) == 0.0)
        # the weights themselves are the definition: A_ij (c + q_i.k_j) / sum, checked at one entry
        i, j = 40, 17
        w = 1.0 + x["Q"][0, h, i] @ x["K"][0, h, j]
        row = 1.0 + x["K"][0, h, : (i + 1 if causal else 64)] @ x["Q"][0, h, i]
        assert abs(A[i, j] - w / row.sum()) < 1e-14


def test_causal_outputs_ignore_future_tokens(oracle_lib):
    x = _tiny(seed=4)
    t = 37
    O, g = oracle_lib.forward(x["Q"], x["K"], x["V"], True)
    dQ, dK, dV = oracle_lib.backward(x["Q"], x["K"], x["V"], x["dO"], True)
    rng = np.random.default_rng(99)
    y = {k: v.copy() for k, v in x.items()}
    for name in ("Q", "K", "V"):
        y[name][:, :, t + 1:] += rng.standard_normal(y[name][:, :, t + 1:].shape)
    O2, g2 = oracle_lib.forward(y["Q"], y["K"], y["V"], True)
    dQ2, _, _ = oracle_lib.backward(y["Q"], y["K"], y["V"], x["dO"], True)
    assert np.array_equal(O[:, :, : t + 1], O2[:, :, : t + 1])
    assert np.array_equal(g[:, :, : t + 1], g2[:, :, : t + 1])
    assert np.array_equal(dQ[:, :, : t + 1], dQ2[:, :, : t + 1])
    assert not np.allclose(O[:, :, t + 1:], O2[:, :, t + 1:])
    # dK_j, dV_j only see dO_i for i >= j
    z = {k: v.copy() for k, v in x.items()}
    z["dO"][:, :, :t] += rng.standard_normal(z["dO"][:, :, :t].shape)
    _, dK3, dV3 = oracle_lib.backward(x["Q"], x["K"], x["V"], z["dO"], True)
    assert np.allclose(dK[:, :, t:], dK3[:, :, t:], rtol=0, atol=1e-12)
    assert np.allclose(dV[:, :, t:], dV3[:, :, t:], rtol=0, atol=1e-12)
    assert not np.allclose(dV[:, :, :t], dV3[:, :, :t])


@pytest.mark.parametrize("causal", [1, 0])
def test_shift_and_linearity_in_v(oracle_lib, causal):
    x = _tiny(seed=5)
    O, _ = oracle_lib.forward(x["Q"], x["K"], x["V"], causal)
    u = np.linspace(-2.0, 3.0, 16)
    Os, _ = oracle_lib.forward(x["Q"], x["K"], x["V"] + u, causal)
    assert np.max(np.abs(Os - (O + u))) < 1e-12
    V2 = np.random.default_rng(6).standard_normal(x["V"].shape)
    O2, _ = oracle_lib.forward(x["Q"], x["K"], V2, causal)
    O12, _ = oracle_lib.forward(x["Q"], x["K"], 2.0 * x["V"] - 3.0 * V2, causal)
    assert np.max(np.abs(O12 - (2.0 * O - 3.0 * O2))) < 1e-12
    # rows of A sum to one, so sum_j dV_j = sum_i dO_i
    _, _, dV = oracle_lib.backward(x["Q"], x["K"], x["V"], x["dO"], causal)
    assert np.max(np.abs(dV.sum(axis=2) - x["dO"].sum(axis=2))) < 1e-12


# ------------------------------------------------------------------------------ closed forms ---

@pytest.mark.parametrize("zero", ["K", "Q"])
def test_zero_keys_or_queries_give_prefix_means(oracle_lib, zero):
    x = _tiny(seed=7)
    x[zero] = np.zeros_like(x[zero])
    V, dO = x["V"], x["dO"]
    n = np.arange(1, 65, dtype=np.float64)[None, None, :, None]
    O, g = oracle_lib.forward(x["Q"], x["K"], V, True)
    assert np.max(np.abs(O - np.cumsum(V, axis=2) / n)) < 1e-13
    assert np.max(np.abs(g - n[..., 0])) == 0.0
    Onc, gnc = oracle_lib.forward(x["Q"], x["K"], V, False)
    assert np.max(np.abs(Onc - V.mean(axis=2, keepdims=True))) < 1e-13
    assert np.all(gnc == 64.0)
    dQ, dK, dV = oracle_lib.backward(x["Q"], x["K"], V, dO, True)
    # dV_j = sum_{i >= j} dO_i / (i + 1)
    want = np.flip(np.cumsum(np.flip(dO / n, axis=2), axis=2), axis=2)
    assert np.max(np.abs(dV - want)) < 1e-13
    if zero == "K":
        assert np.max(np.abs(dQ)) == 0.0
    else:
        assert np.max(np.abs(dK)) == 0.0


def test_single_token_returns_v(oracle_lib):
    x = _tiny(seed=8, N=1)
    for causal in (0, 1):
        O, g = oracle_lib.forward(x["Q"], x["K"], x["V"], causal)
        assert np.max(np.abs(O - x["V"])) < 1e-15
        assert np.max(np.abs(g - (1.0 + np.sum(x["Q"] * x["K"], axis=-1)))) < 1e-15


def test_single_token_gradients(oracle_lib):
    """N = 1: O_0 = v_0, so delta_0 = dO_0 . v_0 and dW_00 = (dO_0 . v_0 - delta_0) / g_0 = 0: dQ = dK = 0,
    and dV_0 = (W_00 / g_0) dO_0 = dO_0.  A sign error in the delta term would leave dW_00 = 2 dO.v / g."""
    x = _tiny(seed=8, N=1)
    for causal in (0, 1):
        dQ, dK, dV = oracle_lib.backward(x["Q"], x["K"], x["V"], x["dO"], causal)
        assert np.max(np.abs(dQ)) < 1e-14 and np.max(np.abs(dK)) < 1e-14
        assert np.max(np.abs(dV - x["dO"])) < 1e-14


def test_equal_keys_noncausal_give_mean(oracle_lib):
    x = _tiny(seed=9)
    x["K"][:] = x["K"][:, :, :1]
    O, _ = oracle_lib.forward(x["Q"], x["K"], x["V"], False)
    assert np.max(np.abs(O - x["V"].mean(axis=2, keepdims=True))) < 1e-12


def test_pure_linear_kernel_d1_is_query_independent(oracle_lib):
    """c = 0, D = 1, positive q, k: O_i = sum_{j<=i} k_j v_j / sum_{j<=i} k_j and dQ = 0."""
    rng = np.random.default_rng(10)
    q = rng.uniform(0.5, 2.0, (1, 1, 20, 1))
    k = rng.uniform(0.5, 2.0, (1, 1, 20, 1))
    v = rng.standard_normal((1, 1, 20, 1))
    dO = rng.standard_normal((1, 1, 20, 1))
    O, _ = oracle_lib.forward(q, k, v, True, c=0.0)
    want = np.cumsum(k * v, axis=2) / np.cumsum(k, axis=2)
    assert np.max(np.abs(O - want)) < 1e-13
    dQ, _, _ = oracle_lib.backward(q, k, v, dO, True, c=0.0)
    assert np.max(np.abs(dQ)) < 1e-13


# ------------------------------------------------------------------------- sampled rows ---

@pytest.mark.parametrize("causal", [1, 0])
def test_sampled_rows_match_full(oracle_lib, causal):
    x = _tiny(seed=12, B=2, H=2, N=50, D=8)
    O, g = oracle_lib.forward(x["Q"], x["K"], x["V"], causal)
    dQ, dK, dV = oracle_lib.backward(x["Q"], x["K"], x["V"], x["dO"], causal)
    rows = np.array([0, 1, 49, 50, 77, 120, 199])
    Or, gr = oracle_lib.forward_rows(x["Q"], x["K"], x["V"], causal, rows)
    assert _rel(Or, O.reshape(-1, 8)[rows]) < 1e-14 and _rel(gr, g.reshape(-1)[rows]) < 1e-14
    dQr = oracle_lib.dq_rows(x["Q"], x["K"], x["V"], x["dO"], causal, rows)
    assert _rel(dQr, dQ.reshape(-1, 8)[rows]) < 1e-13
    dKr, dVr = oracle_lib.dkdv_rows(x["Q"], x["K"], x["V"], x["dO"], causal, rows)
    assert _rel(dKr, dK.reshape(-1, 8)[rows]) < 1e-13 and _rel(dVr, dV.reshape(-1, 8)[rows]) < 1e-13


def test_conditioning_of_tiny_case(oracle_lib):
    """min_i g_i / n_i on the tiny case: the normaliser stays well away from zero."""
    x = _tiny(seed=0)
    _, g = oracle_lib.forward(x["Q"], x["K"], x["V"], True)
    n = np.arange(1, 65, dtype=np.float64)
    assert np.min(g / n) > 0.1


# ------------------------------------------------------------- recurrent (decode) form ---

def _decode_all(oracle_lib, x, start_state=None):
    B, H, N, D = x["Q"].shape
    st = oracle_lib.empty_state(B, H, D) if start_state is None else start_state
    outs, gs = [], []
    for t in range(N):
        o, g, *st = oracle_lib.decode_step(*st, x["Q"][:, :, t], x["K"][:, :, t], x["V"][:, :, t])
        outs.append(o)
        gs.append(g)
    return np.stack(outs, axis=2), np.stack(gs, axis=2), st


def test_decode_golden_d1_worked_example(oracle_lib):
    """Token by token, the recurrence reproduces the hand-worked causal outputs and normalisers."""
    gv = _load_golden()
    x = {n: np.array([gv[("input", m, i)] for i in range(3)]).reshape(1, 1, 3, 1)
         for n, m in (("Q", "q"), ("K", "k"), ("V", "v"))}
    O, g, st = _decode_all(oracle_lib, x)
    for i in range(3):
        assert abs(O.reshape(-1)[i] - gv[("1", "O", i)]) <= 1e-15
        assert abs(g.reshape(-1)[i] - gv[("1", "g", i)]) <= 1e-15
    assert int(st[3].reshape(-1)[0]) == 3


@pytest.mark.parametrize("shape", [(2, 2, 20, 5), (1, 1, 1, 3), (1, 3, 9, 1)])
def test_decode_matches_explicit_causal_rows(oracle_lib, shape):
    """Output t of the recurrence is row t of the explicit (N x N weights) causal forward."""
    B, H, N, D = shape
    x = _tiny(seed=21, B=B, H=H, N=N, D=D)
    O_ref, g_ref = oracle_lib.forward(x["Q"], x["K"], x["V"], True)
    O, g, _ = _decode_all(oracle_lib, x)
    assert _rel(O, O_ref) < 1e-13 and _rel(g, g_ref) < 1e-13


def test_state_append_then_decode_continues_the_forward(oracle_lib):
    """A block of T tokens appended at once, then the rest decoded one by one: the outputs are rows
    T.. of the explicit causal forward over all tokens, and the final state equals the token-by-token
    one (appending is order- and grouping-free)."""
    x = _tiny(seed=22, B=1, H=2, N=30, D=6)
    O_ref, _ = oracle_lib.forward(x["Q"], x["K"], x["V"], True)
    T = 17
    st = oracle_lib.state_append(*oracle_lib.empty_state(1, 2, 6), x["K"][:, :, :T], x["V"][:, :, :T])
    rest = {k: v[:, :, T:] for k, v in x.items()}
    O, _, st_end = _decode_all(oracle_lib, rest, start_state=st)
    assert _rel(O, O_ref[:, :, T:]) < 1e-13
    _, _, st_seq = _decode_all(oracle_lib, x)
    for a_, b_ in zip(st_end, st_seq):
        assert np.max(np.abs(np.asarray(a_, dtype=np.float64) - b_)) < 1e-12
