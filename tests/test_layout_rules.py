"""The host-side memory rules of the strided and the decode entry points against brute force, on CPU.

`la_forward_strided` takes (batch, head, row) element strides per operand; the D elements of a row are
contiguous.  Its contract (include/la.h):
  * an operand is accepted when its rows cannot overlap: ordered by stride, the dimensions of extent > 1
    nest, and every stride is a multiple of 16 bytes; rows that do overlap are always refused;
  * the output may not meet an input: with equal strides the two are compared element by element (so
    interleaved slices of one fused tensor pass), otherwise by address range.
`la_decode_step` / `la_state_append`: the state arrays (S, z, a, n) meet neither each other nor a token
or output buffer; the outputs meet no token input and not each other; token inputs may share memory.
Each case below is a random small layout (seeded) whose element sets or address ranges are enumerated in
Python.  The call
returns LA_ERR_INVALID_ARG (1) when refused.  An accepted call reaches its first CUDA call, which fails
here with LA_ERR_CUDA (4): there is no device, so nothing runs.  These tests are skipped wherever a CUDA
device is present, so that no accepted call with made-up pointers can ever launch work.
"""
import ctypes
import random

import pytest

ARENA = 0x1000_0000      # base of the small address range the operands are placed in
FAR = 0x4000_0000        # K and V, far from the arena
WS = 0x8000_0000         # workspace, far from everything


def _no_device():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


pytestmark = pytest.mark.skipif(not _no_device(), reason="uses made-up device pointers: CPU-only test")


@pytest.fixture(scope="module")
def lib():
    from bwd_la_fwd_gb300 import la
    return la.load_library()


def _elements(base, st, ext, D):
    """Element offsets (from the arena) of every element of an operand, and its rows' element sets."""
    rows = []
    for b in range(ext[0]):
        for h in range(ext[1]):
            for n in range(ext[2]):
                r0 = base + b * st[0] + h * st[1] + n * st[2]
                rows.append(set(range(r0, r0 + D)))
    return rows


def _nested(st, ext, D):
    """The documented acceptance rule: extent-1 dimensions are never stepped; the others, by stride, nest."""
    dims = sorted((st[k], ext[k]) for k in range(3) if ext[k] > 1)
    need = D
    for s, e in dims:
        if s < need:
            return False
        need = s * e
    return True


def _call(lib, q_base, q_st, o_base, o_st, shape, dtype):
    B, H, N, D = shape
    elem = 4 if dtype == 0 else 2
    contig = [H * N * D, N * D, D]
    strides = list(q_st) + contig + contig + list(o_st)
    arr = (ctypes.c_longlong * 12)(*strides)
    vp = ctypes.c_void_p
    span = B * H * N * D * elem
    return lib.la_forward_strided(vp(ARENA + q_base * elem), vp(FAR), vp(FAR + 2 * span), 1,
                                  vp(ARENA + o_base * elem), vp(0), B, H, N, D, dtype, arr, vp(WS), 1 << 30, vp(0))


def _random_layout(rng, ext, D, unit, nested):
    """Strides (multiples of `unit` elements) for extents ext: nested in a random order with random
    padding, or (nested=False) drawn freely."""
    st = [0, 0, 0]
    if nested:
        order = list(range(3))
        rng.shuffle(order)
        cur = D
        for k in order:
            pad = unit * rng.randrange(0, 3)
            s = -(-cur // unit) * unit + pad
            st[k] = s
            cur = s * ext[k]
    else:
        for k in range(3):
            st[k] = unit * rng.randrange(1, 2 + (ext[0] * ext[1] * ext[2] * D) // unit // 4)
    return st


@pytest.mark.parametrize("dtype", [0, 1])
def test_operand_rows_accepted_only_when_disjoint(lib, dtype):
    rng = random.Random(1000 + dtype)
    unit = 4 if dtype == 0 else 8                  # elements per 16 bytes
    seen = {1: 0, 4: 0}
    for _ in range(300):
        B, H, N, D = rng.randrange(1, 3), rng.randrange(1, 4), rng.randrange(1, 6), rng.choice([16, 32])
        ext = (B, H, N)
        st = _random_layout(rng, ext, D, unit, nested=rng.random() < 0.5)
        rows = _elements(0, st, ext, D)
        overlapping = any(rows[a] & rows[b] for a in range(len(rows)) for b in range(a + 1, len(rows)))
        far = 1 << 22                               # output well away from the input
        rc = _call(lib, 0, st, far, [H * N * D, N * D, D], (B, H, N, D), dtype)
        assert rc in (1, 4), rc
        if overlapping:
            assert rc == 1, (ext, D, st)
        if rc == 4:
            assert not overlapping, (ext, D, st)
        if _nested(st, ext, D):
            assert rc == 4, (ext, D, st)
        seen[rc] += 1
    assert seen[1] > 50 and seen[4] > 50  # both outcomes exercised


@pytest.mark.parametrize("dtype", [0, 1])
def test_output_against_input_with_equal_strides_is_element_exact(lib, dtype):
    """Same layout for Q and O, O shifted by a random multiple of 16 bytes: refused exactly when some
    element of O is an element of Q (interleaved rows that do not meet pass)."""
    rng = random.Random(2000 + dtype)
    unit = 4 if dtype == 0 else 8
    seen = {1: 0, 4: 0}
    for _ in range(400):
        B, H, N, D = rng.randrange(1, 3), rng.randrange(1, 4), rng.randrange(1, 6), rng.choice([16, 32])
        ext = (B, H, N)
        st = _random_layout(rng, ext, D, unit, nested=True)
        span = (B - 1) * st[0] + (H - 1) * st[1] + (N - 1) * st[2] + D
        q_base = 4 * span
        o_base = q_base + unit * rng.randrange(-(span // unit) - 2, span // unit + 3)
        q_el = set().union(*_elements(q_base, st, ext, D))
        o_el = set().union(*_elements(o_base, st, ext, D))
        rc = _call(lib, q_base, st, o_base, st, (B, H, N, D), dtype)
        assert rc == (1 if q_el & o_el else 4), (ext, D, st, o_base - q_base)
        seen[rc] += 1
    assert seen[1] > 20 and seen[4] > 20  # both outcomes exercised


@pytest.mark.parametrize("dtype", [0, 1])
def test_output_against_input_with_other_strides_compares_ranges(lib, dtype):
    """Different layouts for Q and O: refused exactly when their address ranges overlap."""
    rng = random.Random(3000 + dtype)
    unit = 4 if dtype == 0 else 8
    seen = {1: 0, 4: 0}
    for _ in range(400):
        B, H, N, D = rng.randrange(1, 3), rng.randrange(1, 4), rng.randrange(1, 6), rng.choice([16, 32])
        ext = (B, H, N)
        sq = _random_layout(rng, ext, D, unit, nested=True)
        so = _random_layout(rng, ext, D, unit, nested=True)
        eff = lambda s: tuple(D if ext[k] == 1 else s[k] for k in range(3))  # noqa: E731
        if eff(sq) == eff(so):
            continue
        span_q = (B - 1) * sq[0] + (H - 1) * sq[1] + (N - 1) * sq[2] + D
        span_o = (B - 1) * so[0] + (H - 1) * so[1] + (N - 1) * so[2] + D
        q_base = 4 * max(span_q, span_o)
        o_base = q_base + unit * rng.randrange(-(span_o // unit) - 2, span_q // unit + 3)
        ranges_meet = o_base < q_base + span_q and q_base < o_base + span_o
        rc = _call(lib, q_base, sq, o_base, so, (B, H, N, D), dtype)
        assert rc == (1 if ranges_meet else 4), (ext, D, sq, so, o_base - q_base)
        seen[rc] += 1
    assert seen[1] > 20 and seen[4] > 20


# ------------------------------------------------------------------ decode state and tokens ---

def _decode_buffers(rng, B, H, D, dtype, arena_units):
    """Random 16-byte-aligned placements (bytes from the arena) of q, k, v, o, g, S, z, a, n."""
    tok = B * H * D * (2 if dtype == 1 else 4)
    acc = 4 if dtype == 1 else 8
    sizes = {"q": tok, "k": tok, "v": tok, "o": tok, "g": B * H * 4,
             "S": B * H * D * D * acc, "z": B * H * D * acc, "a": B * H * D * acc, "n": B * H * 4}
    place = {name: 16 * rng.randrange(0, arena_units) for name in sizes}
    return place, sizes


def _meet(place, sizes, x, y):
    return place[x] < place[y] + sizes[y] and place[y] < place[x] + sizes[x]


@pytest.mark.parametrize("dtype", [0, 1])
def test_decode_step_refuses_exactly_the_forbidden_overlaps(lib, dtype):
    """The state arrays meet neither each other nor a token or output buffer; o and g meet no token input
    and not each other; the token inputs q, k, v may share memory."""
    rng = random.Random(4000 + dtype)
    vp = ctypes.c_void_p
    seen = {1: 0, 4: 0}
    state = ("S", "z", "a", "n")
    for _ in range(600):
        B, H, D = rng.randrange(1, 3), rng.randrange(1, 3), rng.choice([16, 32])
        place, sizes = _decode_buffers(rng, B, H, D, dtype, arena_units=rng.choice([64, 512, 4096, 1 << 16]))
        bad = any(_meet(place, sizes, s, t) for i, s in enumerate(state) for t in state[i + 1:])
        bad |= any(_meet(place, sizes, s, t) for s in state for t in ("q", "k", "v", "o", "g"))
        bad |= any(_meet(place, sizes, "o", t) for t in ("q", "k", "v"))
        bad |= any(_meet(place, sizes, "g", t) for t in ("q", "k", "v", "o"))
        p = {name: vp(ARENA + off) for name, off in place.items()}
        rc = lib.la_decode_step(p["q"], p["k"], p["v"], p["o"], p["g"], p["S"], p["z"], p["a"], p["n"],
                                B, H, D, dtype, vp(0))
        assert rc == (1 if bad else 4), (B, H, D, place)
        seen[rc] += 1
    assert seen[1] > 50 and seen[4] > 50


@pytest.mark.parametrize("dtype", [0, 1])
def test_state_append_refuses_exactly_the_forbidden_overlaps(lib, dtype):
    """The state arrays meet neither each other nor the appended K, V (which may share memory)."""
    rng = random.Random(5000 + dtype)
    vp = ctypes.c_void_p
    seen = {1: 0, 4: 0}
    state = ("S", "z", "a", "n")
    for _ in range(600):
        B, H, D, N = rng.randrange(1, 3), rng.randrange(1, 3), rng.choice([16, 32]), rng.randrange(1, 6)
        place, sizes = _decode_buffers(rng, B, H, D, dtype, arena_units=rng.choice([64, 512, 4096, 1 << 16]))
        sizes["k"] = sizes["v"] = B * H * N * D * (2 if dtype == 1 else 4)
        bad = any(_meet(place, sizes, s, t) for i, s in enumerate(state) for t in state[i + 1:])
        bad |= any(_meet(place, sizes, s, t) for s in state for t in ("k", "v"))
        p = {name: vp(ARENA + off) for name, off in place.items()}
        rc = lib.la_state_append(p["k"], p["v"], p["S"], p["z"], p["a"], p["n"], B, H, N, D, dtype, vp(0))
        assert rc == (1 if bad else 4), (B, H, D, N, place)
        seen[rc] += 1
    assert seen[1] > 50 and seen[4] > 50
