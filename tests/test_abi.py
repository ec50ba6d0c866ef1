"""The C ABI without a GPU: the library loads, exports every symbol include/la.h declares, sizes its
workspace, and rejects bad arguments on the host before any work is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "la.h")


@pytest.fixture(scope="module")
def lib():
    from bwd_la_fwd_gb300 import build, la
    build.build()
    return la.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("la_forward", "la_backward", "la_workspace_bytes", "la_get_status", "la_status_string",
              "la_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_index_checked_build_exports_the_same_symbols():
    """The LA_CHECKED test build (index checks in the tensor-core kernels) is built from the same sources
    and exposes the same boundary."""
    from bwd_la_fwd_gb300 import build, la
    checked = la.open_library(build.build(checked=True))
    for name in declared_functions():
        assert ctypes.cast(getattr(checked, name), ctypes.c_void_p).value, name
    assert checked.la_version() == la.load_library().la_version()


def test_version_and_status_strings(lib):
    assert lib.la_version() >= 100
    for code, name in [(0, "LA_OK"), (1, "LA_ERR_INVALID_ARG"), (2, "LA_ERR_UNSUPPORTED"),
                       (3, "LA_ERR_WORKSPACE"), (4, "LA_ERR_CUDA"), (5, "LA_ERR_TIMEOUT"), (6, "LA_ERR_BOUNDS"),
                       (7, "LA_ERR_STATE")]:
        assert lib.la_status_string(code).decode() == name
    assert lib.la_status_string(99).decode() == "LA_UNKNOWN_STATUS"


def test_workspace_sizes(lib):
    ws = lib.la_workspace_bytes
    # the standard shape: carried states stay small next to the 8 tensor volumes of fwd + bwd
    floor = 8 * 4 * 16 * 4096 * 128 * 2 + 4 * 4 * 16 * 4096
    for causal in (0, 1):
        b = ws(4, 16, 4096, 128, causal, 1, 1)
        assert 0 < b <= 0.2 * floor
        assert ws(4, 16, 4096, 128, causal, 1, 0) <= b
        assert b % 256 == 0
    for D in (16, 32, 64, 128, 256):
        assert ws(1, 2, 1, D, 1, 0, 1) > 0
    assert ws(1, 1, 1, 48, 1, 1, 1) == 0     # unsupported D
    assert ws(0, 1, 8, 64, 1, 1, 1) == 0     # empty batch
    assert ws(1, 1, 8, 64, 1, 7, 1) == 0     # bad dtype
    # long sequences keep at most 64 segments per head
    assert ws(4, 16, 65536, 128, 1, 1, 1) <= 0.2 * 16 * (8 * 4 * 16 * 65536 * 128 * 2)


def test_backward_workspace_holds_what_the_forward_keeps(lib):
    """On the tensor-core path a backward-sized workspace is also what a causal forward keeps its terms in
    for the reusing backward: beyond the forward-sized part it holds the per-row g and dt (fp32), each
    chunk's y_c, e_c (256 floats) and one total state per head (D x D + 2 D floats at D = 128)."""
    ws = lib.la_workspace_bytes
    for B, H, N in ((1, 1, 1), (2, 3, 549), (4, 16, 4096), (8, 16, 2048)):
        BH, nchunk = B * H, (N + 127) // 128
        extra = ws(B, H, N, 128, 1, 1, 1) - ws(B, H, N, 128, 1, 1, 0)
        assert extra >= 4 * (2 * BH * N + 256 * BH * nchunk + BH * (128 * 128 + 2 * 128))


def test_narrow_bf16_heads_take_the_tensor_core_workspace(lib):
    """bf16 with D = 32, 64 runs on the D = 128 tensor-core kernels (columns past D zero-extended): its
    workspace is the D = 128 one (state slots of 128 x 128 + 2 x 128 floats, per-row and per-chunk sums),
    for any B, H, N and either mask; bf16 D = 256 takes the wide kernels' layout, bf16 D = 16 and fp32 are
    sized by their own D (CUDA-core path)."""
    ws = lib.la_workspace_bytes
    for B, H, N in ((1, 1, 1), (2, 3, 549), (4, 16, 4096)):
        for causal in (0, 1):
            for bw in (0, 1):
                ref = ws(B, H, N, 128, causal, 1, bw)
                assert ws(B, H, N, 64, causal, 1, bw) == ref
                assert ws(B, H, N, 32, causal, 1, bw) == ref
    assert ws(2, 3, 549, 256, 1, 1, 1) != ws(2, 3, 549, 128, 1, 1, 1)
    assert ws(2, 3, 549, 16, 1, 1, 1) < ws(2, 3, 549, 32, 1, 1, 1)
    assert ws(2, 3, 549, 64, 1, 0, 1) < ws(2, 3, 549, 128, 1, 0, 1)   # fp32: CUDA-core states of D x D


def _fwd(lib, Q=0x1000, K=0x2000_0000, V=0x4000_0000, O=0x6000_0000, g=0, B=1, H=1, N=8, D=64, dt=1,
         ws=0x8000_0000, wsb=1 << 30):
    vp = ctypes.c_void_p
    return lib.la_forward(vp(Q), vp(K), vp(V), 1, vp(O), vp(g), B, H, N, D, dt, vp(ws), wsb, vp(0))


def test_forward_rejects_bad_arguments_on_host(lib):
    # every case below returns before any CUDA call, so no GPU is touched
    assert _fwd(lib, D=48) == 2                       # unsupported head size
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, dt=3) == 1
    assert _fwd(lib, Q=0) == 1                        # null input
    assert _fwd(lib, K=0x2000_0008) == 1              # misaligned
    assert _fwd(lib, ws=0) == 3                       # no workspace
    assert _fwd(lib, ws=0x8000_0010) == 3             # misaligned workspace
    assert _fwd(lib, wsb=16) == 3                     # workspace too small
    assert _fwd(lib, O=0x1000) == 1                   # output aliases Q
    assert _fwd(lib, g=0x6000_0000 + 64) == 1         # normaliser inside O
    # a causal forward given a backward-sized workspace also writes its backward part (g and each head's
    # total state for the reusing backward): an output there is refused too
    fwd_b, bwd_b = (lib.la_workspace_bytes(1, 1, 8, 64, 1, 1, bw) for bw in (0, 1))
    assert bwd_b > fwd_b
    assert _fwd(lib, O=0x8000_0000 + fwd_b, wsb=bwd_b) == 1
    assert _fwd(lib, g=0x8000_0000 + bwd_b - 256, wsb=bwd_b) == 1


@pytest.mark.parametrize("entry", ["la_backward", "la_backward_with_forward_state"])
def test_backward_rejects_bad_arguments_on_host(lib, entry):
    vp = ctypes.c_void_p
    base = [0x1000_0000 * (i + 1) for i in range(8)]
    fn = getattr(lib, entry)

    def call(ptrs=base, D=64, ws=0xA000_0000, wsb=1 << 30):
        return fn(*[vp(p) for p in ptrs], 1, 1, 2, 16, D, 1, vp(ws), wsb, vp(0))

    assert call(D=24) == 2
    bad = list(base)
    bad[4] = 0
    assert call(bad) == 1
    bad = list(base)
    bad[6] = base[7]                                  # dK == dV
    assert call(bad) == 1
    bad = list(base)
    bad[5] = base[0] + 16                             # dQ overlaps Q
    assert call(bad) == 1
    assert call(wsb=100) == 3


def test_decode_entries_reject_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p
    tok = [0x1000_0000 * (i + 1) for i in range(4)]          # q, k, v, o
    st = [0x9000_0000 + 0x100_0000 * i for i in range(4)]     # S, z, a, n

    def step(t=tok, s=st, g=0, B=1, H=2, D=64, dt=1):
        return lib.la_decode_step(*[vp(p) for p in t], vp(g), *[vp(p) for p in s], B, H, D, dt, vp(0))

    def append(K=0x1000_0000, V=0x2000_0000, s=st, N=8, D=64, dt=1):
        return lib.la_state_append(vp(K), vp(V), *[vp(p) for p in s], 1, 2, N, D, dt, vp(0))

    assert step(D=48) == 2
    assert step(dt=5) == 1
    assert step(B=0) == 1
    assert step(t=[0] + tok[1:]) == 1                          # null q
    assert step(t=tok[:3] + [tok[0]]) == 1                     # o aliases q
    assert step(s=[st[0], st[0] + 64] + st[2:]) == 1           # z inside S
    assert step(s=st[:3] + [0]) == 1                           # null n
    assert step(s=[st[0] + 8] + st[1:]) == 1                   # misaligned S
    assert step(g=tok[0]) == 1                                 # normaliser inside q
    assert append(D=24) == 2
    assert append(N=-1) == 1
    assert append(K=0) == 1
    assert append(s=[0x1000_0000] + st[1:]) == 1               # S overlaps K
    assert append(K=0, V=0, N=0) == 0                          # nothing to append: nothing launched


def test_strided_entries_reject_bad_layouts_on_host(lib):
    vp = ctypes.c_void_p
    B, H, N, D = 2, 4, 64, 64
    base = [0x1000_0000 * (i + 1) for i in range(8)]

    def fwd(strides, ptrs=base[:4]):
        arr = (ctypes.c_longlong * 12)(*strides)
        return lib.la_forward_strided(*[vp(p) for p in ptrs[:3]], 1, vp(ptrs[3]), vp(0), B, H, N, D, 1, arr,
                                      vp(0xA000_0000), 1 << 30, vp(0))

    def bwd(strides, ptrs=base):
        arr = (ctypes.c_longlong * 24)(*strides)
        return lib.la_backward_strided(*[vp(p) for p in ptrs], 1, B, H, N, D, 1, arr, 0, vp(0xA000_0000), 1 << 30,
                                       vp(0))

    bhnd = [H * N * D, N * D, D]
    assert fwd(bhnd[:2] + [D - 8] + bhnd * 3) == 1            # rows of Q overlap (row stride < D)
    assert fwd([H * N * D, N * D, D + 4] + bhnd * 3) == 1     # row stride not a multiple of 16 bytes
    assert fwd([H * N * D, D, 2 * D] + bhnd * 3) == 1         # heads inside rows, but H of them do not fit
    assert fwd(bhnd * 3 + [0, N * D, D]) == 1                 # zero batch stride with B = 2
    # fused [B,N,3,H,D]: Q, K, V interleave and may; an output interleaved with them must not meet them
    fused = [N * 3 * H * D, D, 3 * H * D]
    q0 = 0x2000_0000
    ptrs = [q0, q0 + 2 * H * D, q0 + 4 * H * D, q0 + 2]      # O one element into Q's first row
    assert fwd(fused * 4, ptrs) == 1
    # backward: dK written over V's rows of the same fused tensor
    bptrs = [q0, q0 + 2 * H * D, q0 + 4 * H * D] + base[3:5] + [0x6000_0000, q0 + 4 * H * D, 0x7000_0000]
    assert bwd(fused * 3 + bhnd * 2 + [bhnd[0] * 2, bhnd[1], bhnd[2]] + fused + bhnd, bptrs) == 1
    # dQ and dK in one fused gradient tensor, overlapping rows (same offset)
    g0 = 0x6000_0000
    bptrs = base[:5] + [g0, g0, g0 + 4 * H * D]
    assert bwd(bhnd * 5 + fused * 3, bptrs) == 1
