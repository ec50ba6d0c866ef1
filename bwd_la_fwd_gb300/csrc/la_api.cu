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
    long long seg = 256 > 2 * D ? 256 : 2 * D;
    long long min_for_cap = ((long long)N + 63) / 64;
    min_for_cap = (min_for_cap + 31) / 32 * 32;
    if (seg < min_for_cap) seg = min_for_cap;
    p->seg_len = (int)seg;
    p->nseg = (int)(((long long)N + seg - 1) / seg);
    if (BH * p->nseg >= (1LL << 31)) return false;
    p->stride = (long long)round_up((size_t)D * D + 2 * (size_t)D, 64);
    p->acc_bytes = dtype == LA_F32 ? 8 : 4;
    p->use_tc = tc_supported(*p);
    if (p->use_tc) {
        // forward-direction slots (forward and backward), reverse-direction slots and per-row g, dt
        // (backward only)
        const size_t slots = tc_slot_bytes(*p);
        const size_t nchunk = ((size_t)N + 127) / 128;
        p->off_states = 256;
        p->off_chunkza = round_up(p->off_states + slots, 256);
        p->off_states2 = round_up(p->off_chunkza + (size_t)BH * nchunk * 256 * sizeof(float), 256);
        p->off_flags = round_up(p->off_states2 + slots, 256);
        p->off_rowstats = p->off_flags;
        p->off_chunkye = round_up(p->off_rowstats + 2 * (size_t)BH * N * sizeof(float), 256);
        p->bytes_fwd = p->off_states2;
        p->bytes_bwd = round_up(p->off_chunkye + (size_t)BH * nchunk * 256 * sizeof(float), 256);
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

// Outputs must not overlap any input, the workspace or each other.
int check_aliasing(const Range *outs, int n_out, const Range *ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlap(outs[i], ins[j])) return LA_ERR_INVALID_ARG;
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j])) return LA_ERR_INVALID_ARG;
    }
    return LA_OK;
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

int la_forward(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B, int H,
               int N, int D, int dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || D < 1) return LA_ERR_INVALID_ARG;
    if (!la::supported_d(D)) return LA_ERR_UNSUPPORTED;
    Plan p;
    if (!la::make_plan(B, H, N, D, causal, dtype, &p)) return LA_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O) return LA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return LA_ERR_INVALID_ARG;
    if (normaliser && !aligned(normaliser, 16)) return LA_ERR_INVALID_ARG;
    int rc = check_workspace(p, workspace, workspace_bytes, false);
    if (rc) return rc;
    const size_t tb = (size_t)p.BH * N * D * (dtype == LA_BF16 ? 2 : 4);
    const Range ins[] = {range_of(Q, tb), range_of(K, tb), range_of(V, tb), range_of(workspace, p.bytes_fwd)};
    Range outs[2] = {range_of(O, tb), range_of(normaliser, normaliser ? (size_t)p.BH * N * 4 : 0)};
    if ((rc = check_aliasing(outs, normaliser ? 2 : 1, ins, 4))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = p.use_tc ? la::tc_forward(p, Q, K, V, O, normaliser, (unsigned char *)workspace, s)
                             : clear_state_tag(workspace, s);
    if (e == cudaSuccess && !p.use_tc) e = la::simt_forward(p, Q, K, V, O, normaliser, (unsigned char *)workspace, s);
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

static int backward_impl(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ,
                         void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype, void *workspace,
                         size_t workspace_bytes, void *stream, bool reuse_fwd_state) {
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || D < 1) return LA_ERR_INVALID_ARG;
    if (!la::supported_d(D)) return LA_ERR_UNSUPPORTED;
    Plan p;
    if (!la::make_plan(B, H, N, D, causal, dtype, &p)) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void *q : ptrs)
        if (!q || !aligned(q, 16)) return LA_ERR_INVALID_ARG;
    int rc = check_workspace(p, workspace, workspace_bytes, true);
    if (rc) return rc;
    const size_t tb = (size_t)p.BH * N * D * (dtype == LA_BF16 ? 2 : 4);
    const Range ins[] = {range_of(Q, tb), range_of(K, tb), range_of(V, tb), range_of(O, tb), range_of(dO, tb),
                         range_of(workspace, p.bytes_bwd)};
    const Range outs[] = {range_of(dQ, tb), range_of(dK, tb), range_of(dV, tb)};
    if ((rc = check_aliasing(outs, 3, ins, 6))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = p.use_tc
                        ? la::tc_backward(p, Q, K, V, dO, dQ, dK, dV, (unsigned char *)workspace, s, reuse_fwd_state)
                        : clear_state_tag(workspace, s);
    if (e == cudaSuccess && !p.use_tc)
        e = la::simt_backward(p, Q, K, V, O, dO, dQ, dK, dV, (unsigned char *)workspace, s);
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int la_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ, void *dK,
                void *dV, int causal, int B, int H, int N, int D, int dtype, void *workspace,
                size_t workspace_bytes, void *stream) {
    return backward_impl(Q, K, V, O, dO, dQ, dK, dV, causal, B, H, N, D, dtype, workspace, workspace_bytes, stream,
                         false);
}

int la_backward_with_forward_state(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                   void *dQ, void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    return backward_impl(Q, K, V, O, dO, dQ, dK, dV, causal, B, H, N, D, dtype, workspace, workspace_bytes, stream,
                         true);
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
