// la_api.cu -- the C ABI declared in include/la.h: argument checks, workspace partition, dispatch.
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "../../include/la.h"
#include "la_internal.h"
#include "la_tc_host.h"

namespace la {

static std::atomic<unsigned long long> g_launches{0};

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool supported_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }

// Segment length: long enough that the carried D x D states stay small next to the tensors
// (seg_len >= 2 D keeps them under 1/8 of the bf16 I/O), at least 256 rows, and at most 64 segments
// per head so that the carry chain stays short at long N.
bool make_plan(int B, int H, int N, int D, int causal, int dtype, Plan *p) {
    if (B < 1 || H < 1 || N < 1 || !supported_d(D) || (dtype != LA_F32 && dtype != LA_BF16)) return false;
    const long long BH = (long long)B * H;
    if (BH >= (1LL << 31) || (long long)N * BH * D >= (1LL << 40)) return false;
    memset(p, 0, sizeof(*p));
    p->B = B;
    p->H = H;
    p->N = N;
    p->D = D;
    p->causal = causal ? 1 : 0;
    p->dtype = dtype;
    p->BH = (int)BH;
    for (int k = 0; k < kNumOps; ++k) p->lay[k] = Layout{(long long)H * N * D, (long long)N * D, (long long)D};
    long long seg = 256 > 2 * D ? 256 : 2 * D;
    long long min_for_cap = ((long long)N + 63) / 64;
    min_for_cap = (min_for_cap + 31) / 32 * 32;
    if (seg < min_for_cap) seg = min_for_cap;
    p->seg_len = (int)seg;
    p->nseg = (int)(((long long)N + seg - 1) / seg);
    if (BH * p->nseg >= (1LL << 31)) return false;
    p->acc_bytes = dtype == LA_F32 ? 8 : 4;
    p->use_tc = tc_supported(*p);
    p->use_wide = wide_supported(*p);
    // a state slot holds a D x D matrix and two D-vectors; the tensor-core kernels always work on D = 128
    // (narrower heads are zero-extended), so their slots have that size
    const size_t sd = p->use_tc ? 128 : (size_t)D;
    p->stride = (long long)round_up(sd * sd + 2 * sd, 64);
    if (p->use_tc) {
        // state slots (the forward's sums; in the backward also its reverse sums, in the same slots), each
        // chunk's column sums, and (backward only) per-row g, dt and each chunk's y_c, e_c
        const size_t slots = tc_slot_bytes(*p);
        const size_t nchunk = ((size_t)N + 127) / 128;
        p->off_states = 256;
        p->off_states2 = p->off_states;
        p->off_chunkza = round_up(p->off_states + slots, 256);
        p->bytes_fwd = round_up(p->off_chunkza + (size_t)BH * nchunk * 256 * sizeof(float), 256);
        p->off_flags = p->bytes_fwd;
        p->off_rowstats = p->off_flags;
        p->off_chunkye = round_up(p->off_rowstats + 2 * (size_t)BH * N * sizeof(float), 256);
        p->off_htot = round_up(p->off_chunkye + (size_t)BH * nchunk * 256 * sizeof(float), 256);
        p->bytes_bwd = round_up(p->off_htot + (size_t)BH * (size_t)p->stride * sizeof(float), 256);
        return true;
    }
    if (p->use_wide) {
        // the forward needs only the header; the backward keeps dO / g (bf16) and the row terms g, dt
        p->off_states = 256;
        p->off_rowstats = round_up(p->off_states + (size_t)BH * N * D * 2, 256);
        p->off_flags = p->off_rowstats;
        p->bytes_fwd = 256;
        p->bytes_bwd = round_up(p->off_rowstats + 2 * (size_t)BH * N * sizeof(float), 256);
        return true;
    }
    const size_t states = (size_t)BH * p->nseg * (size_t)p->stride * p->acc_bytes;
    const size_t flags = (size_t)BH * p->nseg * sizeof(uint32_t);
    p->off_states = 256;
    p->off_flags = round_up(p->off_states + states, 256);
    p->off_rowstats = round_up(p->off_flags + flags, 256);
    p->bytes_fwd = p->off_rowstats;
    // g, delta and up to four per-column-block partial sums of delta
    const size_t nblk = D > 64 ? (size_t)D / 64 : 1;
    p->bytes_bwd = round_up(p->off_rowstats + (2 + nblk) * (size_t)BH * N * p->acc_bytes, 256);
    return true;
}

}  // namespace la

using la::Plan;

namespace {

bool aligned(const void *ptr, uintptr_t a) { return ((uintptr_t)ptr % a) == 0; }

struct Range {
    uintptr_t lo, hi;
};

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void *ptr, size_t bytes) { return Range{(uintptr_t)ptr, (uintptr_t)ptr + bytes}; }

// The SIMT path leaves no tensor-core state sums in the workspace: clear the tag that names them.
cudaError_t clear_state_tag(void *ws, cudaStream_t s) {
    return cudaMemsetAsync((unsigned char *)ws + offsetof(la::WsHeader, state_tag), 0,
                           sizeof(((la::WsHeader *)nullptr)->state_tag), s);
}

int check_workspace(const Plan &p, void *ws, size_t ws_bytes, bool backward) {
    if (!ws || !aligned(ws, 256)) return LA_ERR_WORKSPACE;
    if (ws_bytes < (backward ? p.bytes_bwd : p.bytes_fwd)) return LA_ERR_WORKSPACE;
    return LA_OK;
}

// ---- strided operands -------------------------------------------------------------------------
// Each operand is given by its (batch, head, row) element strides; its D row elements are contiguous.
// An operand is accepted when its rows cannot overlap one another: ordered by stride, the dimensions of
// extent > 1 nest (the smallest stride is at least D, each larger one at least the previous stride
// times its extent), and every stride is a multiple of 16 bytes (the tensor-map rule).

// Sets p.lay[op] from strides[0..2] (batch, head, row); a dimension of extent 1 is never stepped, so its
// stride is replaced by one that is always valid.
int set_layout(Plan &p, int op, const long long *st, int elem) {
    const long long ext[3] = {p.B, p.H, p.N};
    long long s[3] = {st[0], st[1], st[2]};
    for (int k = 0; k < 3; ++k) {
        if (ext[k] == 1) s[k] = p.D;
        if (s[k] < 1 || s[k] >= (1LL << 40) / elem || (s[k] * elem) % 16 != 0) return LA_ERR_INVALID_ARG;
    }
    int idx[3] = {0, 1, 2};  // dimensions by increasing stride
    for (int a = 0; a < 3; ++a)
        for (int b = a + 1; b < 3; ++b)
            if (s[idx[b]] < s[idx[a]]) { const int t = idx[a]; idx[a] = idx[b]; idx[b] = t; }
    long long need = p.D;
    for (int k = 0; k < 3; ++k) {
        const int d = idx[k];
        if (ext[d] == 1) continue;
        if (s[d] < need) return LA_ERR_INVALID_ARG;  // rows would overlap
        need = s[d] * ext[d];
    }
    p.lay[op] = la::Layout{s[0], s[1], s[2]};
    return LA_OK;
}

// Elements from an operand's base to one past its last element.
long long span_of(const Plan &p, const la::Layout &l) {
    return (p.B - 1) * l.sb + (p.H - 1) * l.sh + (p.N - 1) * l.sn + p.D;
}

// Whether some row of an operand starting `delta` elements after another one of the same layout meets a
// row of that one: delta = db sb + dh sh + dn sn + dd with |db| < B, |dh| < H, |dn| < N, |dd| < D.  The
// dimensions nest (set_layout), so at each level only the quotients next to delta / stride can work.
bool rows_meet(long long delta, const long long *st, const long long *ext, int n, long long D) {
    if (n == 0) return delta > -D && delta < D;
    const long long s = st[0];
    long long q = delta / s;
    for (long long c = q - 2; c <= q + 2; ++c)
        if (c > -ext[0] && c < ext[0] && rows_meet(delta - c * s, st + 1, ext + 1, n - 1, D)) return true;
    return false;
}

bool operands_meet(const Plan &p, const void *a, const la::Layout &la_, const void *b, const la::Layout &lb,
                   int elem) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    if (!overlap(range_of(a, (size_t)span_of(p, la_) * elem), range_of(b, (size_t)span_of(p, lb) * elem)))
        return false;
    if (la_.sb != lb.sb || la_.sh != lb.sh || la_.sn != lb.sn) return true;  // interleaved other layouts: refuse
    const long long diff = (long long)(pb - pa);
    if (diff % elem != 0) return true;
    long long st[3], ext[3];
    int n = 0;
    const long long s3[3] = {la_.sb, la_.sh, la_.sn}, e3[3] = {p.B, p.H, p.N};
    int idx[3] = {0, 1, 2};  // by decreasing stride
    for (int x = 0; x < 3; ++x)
        for (int y = x + 1; y < 3; ++y)
            if (s3[idx[y]] > s3[idx[x]]) { const int t = idx[x]; idx[x] = idx[y]; idx[y] = t; }
    for (int k = 0; k < 3; ++k)
        if (e3[idx[k]] > 1) {
            st[n] = s3[idx[k]];
            ext[n] = e3[idx[k]];
            ++n;
        }
    return rows_meet(diff / elem, st, ext, n, p.D);
}

}  // namespace

extern "C" {

int la_version(void) { return 100; }

unsigned long long la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

const char *la_status_string(int status) {
    switch (status) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
        case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE";
        case LA_ERR_CUDA: return "LA_ERR_CUDA";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
        case LA_ERR_BOUNDS: return "LA_ERR_BOUNDS";
        case LA_ERR_STATE: return "LA_ERR_STATE";
        default: return "LA_UNKNOWN_STATUS";
    }
}

size_t la_workspace_bytes(int B, int H, int N, int D, int causal, int dtype, int backward) {
    Plan p;
    if (!la::make_plan(B, H, N, D, causal, dtype, &p)) return 0;
    return backward ? p.bytes_bwd : p.bytes_fwd;
}

int la_forward_strided(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B,
                       int H, int N, int D, int dtype, const long long *strides, void *workspace,
                       size_t workspace_bytes, void *stream) {
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || D < 1) return LA_ERR_INVALID_ARG;
    if (!la::supported_d(D)) return LA_ERR_UNSUPPORTED;
    Plan p;
    if (!la::make_plan(B, H, N, D, causal, dtype, &p)) return LA_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O) return LA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return LA_ERR_INVALID_ARG;
    if (normaliser && !aligned(normaliser, 16)) return LA_ERR_INVALID_ARG;
    const int elem = dtype == LA_BF16 ? 2 : 4;
    const int ops[4] = {la::kOpQ, la::kOpK, la::kOpV, la::kOpO};
    int rc;
    if (strides)
        for (int k = 0; k < 4; ++k)
            if ((rc = set_layout(p, ops[k], strides + 3 * k, elem))) return rc;
    if ((rc = check_workspace(p, workspace, workspace_bytes, false))) return rc;
    // O must meet neither an input, the workspace nor the normaliser; the normaliser neither of those
    const void *ins[3] = {Q, K, V};
    for (int k = 0; k < 3; ++k)
        if (operands_meet(p, O, p.lay[la::kOpO], ins[k], p.lay[ops[k]], elem)) return LA_ERR_INVALID_ARG;
    // the bytes of the workspace the forward writes: with a backward-sized workspace, for D = 256 and for
    // the causal tensor-core form, it also keeps g (and, causal, each head's total state) there for the
    // backward
    const bool keep = workspace_bytes >= p.bytes_bwd && (p.use_wide || (p.use_tc && p.causal));
    const size_t ws_used = keep ? p.bytes_bwd : p.bytes_fwd;
    const Range ws_r = range_of(workspace, ws_used), o_r = range_of(O, (size_t)span_of(p, p.lay[la::kOpO]) * elem);
    if (overlap(o_r, ws_r)) return LA_ERR_INVALID_ARG;
    if (normaliser) {
        const Range g_r = range_of(normaliser, (size_t)p.BH * N * 4);
        if (overlap(g_r, ws_r) || overlap(g_r, o_r)) return LA_ERR_INVALID_ARG;
        for (int k = 0; k < 3; ++k)
            if (overlap(g_r, range_of(ins[k], (size_t)span_of(p, p.lay[ops[k]]) * elem))) return LA_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    unsigned char *ws = (unsigned char *)workspace;
    cudaError_t e = p.use_tc ? la::tc_forward(p, Q, K, V, O, normaliser, ws, s, keep) : clear_state_tag(workspace, s);
    if (e == cudaSuccess && p.use_wide)
        e = la::wide_forward(p, Q, K, V, O, normaliser, ws, s, keep);
    else if (e == cudaSuccess && !p.use_tc) e = la::simt_forward(p, Q, K, V, O, normaliser, ws, s);
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int la_forward(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B, int H,
               int N, int D, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
    return la_forward_strided(Q, K, V, causal, O, normaliser, B, H, N, D, dtype, nullptr, workspace, workspace_bytes,
                              stream);
}

static int backward_impl(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ,
                         void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype,
                         const long long *strides, void *workspace, size_t workspace_bytes, void *stream,
                         bool reuse_fwd_state) {
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || D < 1) return LA_ERR_INVALID_ARG;
    if (!la::supported_d(D)) return LA_ERR_UNSUPPORTED;
    Plan p;
    if (!la::make_plan(B, H, N, D, causal, dtype, &p)) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void *q : ptrs)
        if (!q || !aligned(q, 16)) return LA_ERR_INVALID_ARG;
    const int elem = dtype == LA_BF16 ? 2 : 4;
    int rc;
    if (strides)
        for (int k = 0; k < la::kNumOps; ++k)  // strides follow the argument order, which is the operand order
            if ((rc = set_layout(p, k, strides + 3 * k, elem))) return rc;
    if ((rc = check_workspace(p, workspace, workspace_bytes, true))) return rc;
    // each output meets no input, no other output and not the workspace
    const Range ws_r = range_of(workspace, p.bytes_bwd);
    for (int o = la::kOpdQ; o <= la::kOpdV; ++o) {
        if (overlap(range_of(ptrs[o], (size_t)span_of(p, p.lay[o]) * elem), ws_r)) return LA_ERR_INVALID_ARG;
        for (int k = 0; k < la::kNumOps; ++k)
            if (k != o && operands_meet(p, ptrs[o], p.lay[o], ptrs[k], p.lay[k], elem)) return LA_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    unsigned char *ws = (unsigned char *)workspace;
    cudaError_t e = cudaSuccess;
    if (p.use_tc) {
        e = la::tc_backward(p, Q, K, V, O, dO, dQ, dK, dV, ws, s, reuse_fwd_state);
    } else if (p.use_wide) {
        // D = 256: the reusing backward checks the forward's record of g; the plain one recomputes g over
        // the region the forward keeps it in, so that record no longer holds
        if (!reuse_fwd_state) e = clear_state_tag(workspace, s);
        if (e == cudaSuccess) e = la::wide_backward(p, Q, K, V, O, dO, dQ, dK, dV, ws, s, reuse_fwd_state);
    } else {
        e = clear_state_tag(workspace, s);
        if (e == cudaSuccess) e = la::simt_backward(p, Q, K, V, O, dO, dQ, dK, dV, ws, s);
    }
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int la_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ, void *dK,
                void *dV, int causal, int B, int H, int N, int D, int dtype, void *workspace,
                size_t workspace_bytes, void *stream) {
    return backward_impl(Q, K, V, O, dO, dQ, dK, dV, causal, B, H, N, D, dtype, nullptr, workspace, workspace_bytes,
                         stream, false);
}

int la_backward_with_forward_state(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                   void *dQ, void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    return backward_impl(Q, K, V, O, dO, dQ, dK, dV, causal, B, H, N, D, dtype, nullptr, workspace, workspace_bytes,
                         stream, true);
}

int la_backward_strided(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ,
                        void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype, const long long *strides,
                        int reuse_forward_state, void *workspace, size_t workspace_bytes, void *stream) {
    return backward_impl(Q, K, V, O, dO, dQ, dK, dV, causal, B, H, N, D, dtype, strides, workspace, workspace_bytes,
                         stream, reuse_forward_state != 0);
}

int la_get_status(void *workspace, void *stream) {
    if (!workspace || !aligned(workspace, 256)) return LA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    uint32_t status = 0;
    if (cudaMemcpy(&status, workspace, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess) return LA_ERR_CUDA;
    if (status != 0 && cudaMemset(workspace, 0, sizeof(uint32_t)) != cudaSuccess) return LA_ERR_CUDA;
    return (int)status;
}

}  // extern "C"
