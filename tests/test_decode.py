"""GPU parity of the recurrent (decode) form against the fp64 oracle.

la_decode_step appends one token per (b, h) to the carried state (S, z, a, n) and returns its output;
la_state_append appends a block of tokens.  Output t of the recurrence is row t of the causal forward,
so the oracle here is the explicit (N x N weights) causal forward, plus the oracle's own state
recurrence for the state arrays.  Tolerances are those of the forward (fp32 I/O: elementwise 1e-5;
bf16 I/O: normalised max-abs 2e-2; normaliser 1e-5 / 1e-3); the state, kept in the accumulator type
(fp64 for fp32 tokens, fp32 for bf16 tokens), is compared at normalised max-abs 1e-12 / 1e-5.
"""
import numpy as np
import pytest

import la_testutil as U
from bwd_la_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu

STATE_TOL = {"f32": 1e-12, "bf16": 1e-5}


def _torch_dtype(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _tokens(x, dtype, name, t):
    """Token t of tensor `name` ([B,H,N,D] numpy, stored bits/values) as a contiguous [B,H,D] device tensor."""
    return U.to_device(np.ascontiguousarray(x[name][:, :, t]), dtype)


def _check_state(state, ref, dtype):
    S, z, a, n = ref
    for name, got, want in (("S", state.S, S), ("z", state.z, z), ("a", state.a, a)):
        e = U.err_norm_maxabs(U.to_f64(got), want)
        assert e <= STATE_TOL[dtype], f"state {name}: {e:.3e}"
    assert np.array_equal(state.n.cpu().numpy(), np.asarray(n))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
def test_decode_sequence_matches_causal_forward(oracle_lib, dtype, D):
    from bwd_la_fwd_gb300 import la
    B, H, N = 2, 3, 40
    x = inputs.generate(B, H, N, D, seed=300 + D, dtype=dtype)
    f = U.stored_to_f64(x, dtype)
    state = la.DecodeState(B, H, D, _torch_dtype(dtype))
    outs, gs = [], []
    for t in range(N):
        o, g = la.la_decode_step(state, *(_tokens(x, dtype, n, t) for n in ("Q", "K", "V")))
        outs.append(U.to_f64(o))
        gs.append(U.to_f64(g))
    O_ref, g_ref = oracle_lib.forward(f["Q"], f["K"], f["V"], True)
    U.assert_close("O", np.stack(outs, axis=2), O_ref, dtype)
    U.assert_close("g", np.stack(gs, axis=2), g_ref, dtype)
    _check_state(state, oracle_lib.state_append(*oracle_lib.empty_state(B, H, D), f["K"], f["V"]), dtype)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 32)])
def test_append_then_decode_continues_the_forward(oracle_lib, dtype, D):
    """A prompt of T tokens appended as a block, then tokens decoded one by one: outputs are rows T.. of
    the causal forward over all tokens (T spans several token blocks and a ragged tail)."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, T, extra = 1, 2, 300, 6
    x = inputs.generate(B, H, T + extra, D, seed=310 + D, dtype=dtype)
    f = U.stored_to_f64(x, dtype)
    state = la.DecodeState(B, H, D, _torch_dtype(dtype))
    Kp = U.to_device(np.ascontiguousarray(x["K"][:, :, :T]), dtype)
    Vp = U.to_device(np.ascontiguousarray(x["V"][:, :, :T]), dtype)
    la.la_state_append(state, Kp, Vp)
    _check_state(state, oracle_lib.state_append(*oracle_lib.empty_state(B, H, D), f["K"][:, :, :T],
                                                f["V"][:, :, :T]), dtype)
    outs = []
    for t in range(T, T + extra):
        o, _ = la.la_decode_step(state, *(_tokens(x, dtype, n, t) for n in ("Q", "K", "V")))
        outs.append(U.to_f64(o))
    torch.cuda.synchronize()
    rows = [(b * H + h) * (T + extra) + t for b in range(B) for h in range(H) for t in range(T, T + extra)]
    O_rows, _ = oracle_lib.forward_rows(f["Q"], f["K"], f["V"], True, rows)
    U.assert_close("O", np.stack(outs, axis=2).reshape(-1, D), O_rows, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("D", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 33, 77])
def test_state_append_matches_oracle(oracle_lib, dtype, D, N):
    from bwd_la_fwd_gb300 import la
    B, H = 2, 2
    x = inputs.generate(B, H, N, D, seed=320 + N + D, dtype=dtype)
    f = U.stored_to_f64(x, dtype)
    state = la.DecodeState(B, H, D, _torch_dtype(dtype))
    K, V = (U.to_device(x[n], dtype) for n in ("K", "V"))
    la.la_state_append(state, K, V)
    la.la_state_append(state, K, V)  # appended twice: the sums double, n = 2 N
    S, z, a, n = oracle_lib.state_append(*oracle_lib.empty_state(B, H, D), f["K"], f["V"])
    _check_state(state, oracle_lib.state_append(S, z, a, n, f["K"], f["V"]), dtype)


def test_heads_with_different_counts(oracle_lib):
    """Heads may carry states of different lengths: one decode step from a state that the oracle built
    with 5 tokens in one head and 12 in the other."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, D, dtype = 1, 2, 64, "bf16"
    x = inputs.generate(B, H, 13, D, seed=330, dtype=dtype)
    f = U.stored_to_f64(x, dtype)
    ref = oracle_lib.empty_state(B, H, D)
    for h, T in ((0, 5), (1, 12)):
        st = oracle_lib.state_append(*(r[:, h:h + 1] for r in ref), f["K"][:, h:h + 1, :T], f["V"][:, h:h + 1, :T])
        for r, s in zip(ref, st):
            r[:, h:h + 1] = s
    state = la.DecodeState(B, H, D, torch.bfloat16)
    state.S.copy_(torch.from_numpy(ref[0]))
    state.z.copy_(torch.from_numpy(ref[1]))
    state.a.copy_(torch.from_numpy(ref[2]))
    state.n.copy_(torch.from_numpy(ref[3].astype(np.int32)))
    t_of = {0: 5, 1: 12}
    q, k, v = (np.stack([f[n][:, h, t_of[h]] for h in range(H)], axis=1) for n in ("Q", "K", "V"))
    qd, kd, vd = (U.to_device(np.stack([x[n][:, h, t_of[h]] for h in range(H)], axis=1), dtype)
                  for n in ("Q", "K", "V"))
    o, g = la.la_decode_step(state, qd, kd, vd)
    o_ref, g_ref, *st = oracle_lib.decode_step(*ref, q, k, v)
    U.assert_close("O", U.to_f64(o), o_ref, dtype)
    U.assert_close("g", U.to_f64(g), g_ref, dtype)
    _check_state(state, st, dtype)


def test_decode_steps_replay_in_a_cuda_graph(oracle_lib):
    """The decode step enqueues one kernel and never synchronises, so a run of steps can be captured in
    a CUDA graph and replayed; replaying it equals running the steps eagerly."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, D, steps, dtype = 2, 4, 128, 4, "bf16"
    x = inputs.generate(B, H, steps, D, seed=340, dtype=dtype)
    toks = [[_tokens(x, dtype, n, t) for n in ("Q", "K", "V")] for t in range(steps)]
    eager = la.DecodeState(B, H, D, torch.bfloat16)
    ref_out = [la.la_decode_step(eager, *tk)[0].clone() for tk in toks]
    graphed = la.DecodeState(B, H, D, torch.bfloat16)
    outs = [torch.empty_like(toks[0][0]) for _ in range(steps)]
    gs = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(steps)]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for t in range(steps):
            la.la_decode_step(graphed, *toks[t], o=outs[t], normaliser=gs[t], stream=stream)
    graph.replay()
    torch.cuda.synchronize()
    for a_, b_ in zip(outs, ref_out):
        assert torch.equal(a_, b_)
    assert torch.equal(graphed.S, eager.S) and torch.equal(graphed.n, eager.n)


def test_full_heads_after_a_long_prompt(oracle_lib):
    """The standard head layout (B = 4, H = 16, D = 128, bf16) after a 4096-token prompt: two decode
    steps, checked on sampled heads against the explicit causal rows 4096 and 4097."""
    import torch
    from bwd_la_fwd_gb300 import la
    B, H, T, D, dtype = 4, 16, 4096, 128, "bf16"
    x = inputs.generate(B, H, T + 2, D, seed=350, dtype=dtype)
    state = la.DecodeState(B, H, D, torch.bfloat16)
    la.la_state_append(state, *(U.to_device(np.ascontiguousarray(x[n][:, :, :T]), dtype) for n in ("K", "V")))
    outs = [U.to_f64(la.la_decode_step(state, *(_tokens(x, dtype, n, t) for n in ("Q", "K", "V")))[0])
            for t in (T, T + 1)]
    torch.cuda.synchronize()
    assert np.all(state.n.cpu().numpy() == T + 2)
    heads = [(0, 0), (1, 7), (3, 15)]
    for b, h in heads:
        f = {n: inputs.to_f64(x[n][b:b + 1, h:h + 1], dtype) for n in ("Q", "K", "V")}
        O_rows, _ = oracle_lib.forward_rows(f["Q"], f["K"], f["V"], True, [T, T + 1])
        got = np.stack([o[b, h] for o in outs])
        U.assert_close("O", got, O_rows, dtype)
