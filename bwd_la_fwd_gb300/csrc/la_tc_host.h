// la_tc_host.h -- parameters of the tensor-core kernels and the host entry points that launch them.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "la_internal.h"
#include "la_tc_common.cuh"

namespace la {
namespace tc {

// Kernel parameters (passed as a __grid_constant__ struct; the tensor maps stay in parameter space).
struct TcParams {
    CUtensorMap tmQ, tmK, tmV, tmdO;  // bf16 maps with the operand's strides (see `flat`); box 64 columns x
                                      // 128 rows of one head, 128-byte swizzle
    CUtensorMap tmO, tmdQ, tmdK, tmdV;  // the outputs, same form (tiles are staged in shared memory)
    Slices sl;
    int H;                  // heads per batch entry: flat head bh = b H + h
    int flat;               // the maps are 3-D over {D, N, B H} (kernels <FLAT = true>), else 4-D over {D, N, H, B}
    int nbox;               // 64-column boxes holding the operands' D columns: 2 for D = 128, 1 for D = 32, 64
                            // (the kernels compute with D = 128; columns past D load as zero and are not stored)
    uint64_t kv_layout;     // hash of K's and V's strides and of D (part of the per-piece sums' identity)
    long long N;
    float *slots;           // per-piece state sums, slot stride `slot_stride` floats
    float *slots_rev;       // backward: per-piece reverse-direction sums
    long long slot_stride;
    uint32_t *status;       // workspace status word
    void *O;                // forward output (bf16)
    float *g;               // forward normaliser (may be null)
    void *dQ, *dK, *dV;     // backward outputs (bf16)
    float *rs_g, *rs_dt;    // backward row statistics: g_i and delta_i / g_i
    float *chunk_ye;        // causal backward: per chunk, y_c = sum dt_i q_i then e_c = sum dO_i / g_i
    float *chunk_za;        // per chunk: z_c = sum k_j then a_c = sum v_j (written by the sums kernel)
    const void *Kp, *Vp;    // K and V: with the shape they identify the per-piece sums in the workspace
    int check_tag;          // backward reusing the forward's sums: 0 no check, else the form expected + 1
    float *combine_slots;   // tc_combine_kernel: the slot array it turns into carries
    int combine_mode;       // tc_combine_kernel: kCombinePrefix, kCombineSuffix or kCombineTotal
    uint64_t combine_tag;   // tc_combine_kernel: the form to record in the workspace tag (0: leave the tag)
    uint64_t wait_ns;       // bound on a single barrier wait (0: the default, tc::kWaitNs)
    int test_drop_load;     // test hook: CTA 0 of the sums kernel issues no load for this iteration (-1: none)
    int whole_heads;        // non-causal, every slice exactly one head: its piece sums are the head's totals,
                            // and no tc_combine_kernel runs
    float *htot;            // one slot per head: the head's total state (S, z, a).  The causal forward's
                            // combine writes it when set; the single-sweep backward starts from it
    uint32_t use_token;     // single-sweep backward: this launch's mark on the forward's record (>= 2)
};

// Extents, in floats, of the workspace arrays that the kernels index themselves (checked in the LA_CHECKED
// build): a slot array (BH + kMaxCtas slots), the per-chunk column sums, the per-row statistics (and the
// caller's normaliser, [B,H,N]).
__host__ __device__ inline long long n_slot_floats(const TcParams &P) {
    return (P.sl.T / P.sl.nchunk + kMaxCtas) * P.slot_stride;
}
__host__ __device__ inline long long n_chunk_floats(const TcParams &P) { return P.sl.T * 256; }
__host__ __device__ inline long long n_row_floats(const TcParams &P) { return P.sl.T / P.sl.nchunk * P.N; }
__host__ __device__ inline long long n_htot_floats(const TcParams &P) { return P.sl.T / P.sl.nchunk * P.slot_stride; }

// Whether slot (h + b) lies wholly inside its array (and slots do not overlap); LA_CHECKED only.
__device__ __forceinline__ bool slot_ok(const TcParams &P, long long h, int b, uint32_t where) {
    const long long base = slot_of(h, b) * P.slot_stride, n = n_slot_floats(P);
    return in_range(base, n, P.status, where) && in_range(base + kSlotF4 * 4 - 1, n, P.status, where) &&
           in_range(kSlotF4 * 4 - 1, P.slot_stride, P.status, where);
}

// Forms of the slot arrays (tc_combine_kernel).
enum : int { kCombinePrefix = 0, kCombineSuffix = 1, kCombineTotal = 2 };
// The per-piece sums kernel records in the workspace header which K, V and slicing the slots hold, and
// tc_combine_kernel in which form (kTagRaw: each piece's own sums; kTagPrefix: the sums over the head's
// earlier pieces; kTagTotals: the head's total); a backward that reuses them instead of recomputing them
// checks the record first.
constexpr uint64_t kTagRaw = 1, kTagPrefix = 2, kTagTotals = 3;
constexpr size_t kTagOffset = 128;  // bytes into the workspace header
static_assert(kTagOffset == offsetof(WsHeader, state_tag), "tag offset");
constexpr int kTagWords = 7;
__host__ __device__ inline void state_tag(const TcParams &P, uint64_t form, uint64_t *t) {
    t[0] = 0x4C415F5354415445ull ^ P.kv_layout;  // marker ("LA_STATE"), folded with K's and V's strides and D
    t[1] = (uint64_t)(uintptr_t)P.Kp;
    t[2] = (uint64_t)(uintptr_t)P.Vp;
    t[3] = (uint64_t)P.sl.T;
    t[4] = (uint64_t)P.N;
    t[5] = (uint64_t)P.sl.G;
    t[6] = form;
}
#ifdef __CUDACC__
__device__ inline void write_state_tag(const TcParams &P, uint64_t form) {
    uint64_t t[kTagWords];
    state_tag(P, form, t);
    volatile uint64_t *w = (volatile uint64_t *)((unsigned char *)P.status + kTagOffset);
    for (int k = 0; k < kTagWords; ++k) w[k] = t[k];
}
__device__ inline bool state_tag_matches(const TcParams &P, uint64_t form) {
    uint64_t t[kTagWords];
    state_tag(P, form, t);
    const volatile uint64_t *w = (const volatile uint64_t *)((const unsigned char *)P.status + kTagOffset);
    bool ok = true;
    for (int k = 0; k < kTagWords; ++k) ok = ok && w[k] == t[k];
    return ok;
}
// The backward keeps its reverse sums in the slots of the forward's sums; its dK/dV walk marks them used,
// and the combine that records new forward sums clears the mark.
__device__ inline volatile uint32_t *fwd_sums_used(const TcParams &P) {
    return (volatile uint32_t *)((unsigned char *)P.status + offsetof(WsHeader, fwd_sums_used));
}
// Set by a backward's dQ walk (CTA 0) when it refused the forward's record, read by its dK / dV walk.
__device__ inline volatile uint32_t *bwd_skip(const TcParams &P) {
    return (volatile uint32_t *)((unsigned char *)P.status + offsetof(WsHeader, bwd_skip));
}
// Set with the tag by the causal forward's combine when it also kept g and the heads' totals.
__device__ inline volatile uint32_t *fwd_terms_kept(const TcParams &P) {
    return (volatile uint32_t *)((unsigned char *)P.status + offsetof(WsHeader, fwd_terms_kept));
}
#endif

}  // namespace tc

// Host helpers shared by the forward and backward launchers (la_tc_fwd.cu).
namespace tc_host {
int sm_count();  // multiprocessors of the current device (cached per device), 0 on error
bool make_map(CUtensorMap *m, const void *ptr, const Plan &p, int op, bool flat);
bool flat_heads(const Plan &p, const int *ops, int n);
bool fill_common(tc::TcParams &P, const Plan &p, unsigned char *ws);
cudaError_t launch_agg(const tc::TcParams &P, cudaStream_t s);  // per-piece K^T V sums into P.slots
// Launches a tensor-core kernel as a programmatic dependent of the previous kernel in the stream (the
// kernels order their global accesses after griddepcontrol.wait, so stream order is kept).
cudaError_t launch_tc(void (*kernel)(const tc::TcParams), dim3 grid, unsigned block, size_t smem,
                      cudaStream_t s, const tc::TcParams &P);
// Turns the piece slots of `slots` into carries (mode: tc::kCombine*; tag_form: the form to record in the
// workspace tag, 0 to leave it).
cudaError_t launch_combine(tc::TcParams P, float *slots, int mode, uint64_t tag_form, cudaStream_t s);
}  // namespace tc_host

// bf16 storage with D = 32, 64 or 128: the tcgen05 kernels (on 128 columns, narrower heads zero-extended by
// the tensor maps); everything else takes the SIMT path.
bool tc_supported(const Plan &p);
// Workspace bytes the tensor-core path needs for its state slots (one direction).
size_t tc_slot_bytes(const Plan &p);
// keep_terms (causal, the workspace is sized for the backward): also keep g_i and each head's total state
// in the workspace, for the single-sweep backward.
cudaError_t tc_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                       unsigned char *ws, cudaStream_t s, bool keep_terms);
// reuse_fwd_state: take the per-piece K^T V sums the forward left in the workspace (tag checked on the
// device, LA_ERR_STATE when it does not match) instead of recomputing them; causal, also the forward's g
// (its dQ walk then forms delta from O), and the call may run as one reverse sweep per head instead of
// the two walks (tc_sweep_chosen).
cudaError_t tc_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s, bool reuse_fwd_state);
// Whether a causal backward that reuses the forward's state runs as the single sweep (la_tc_sweep.cu):
// D = 128 and, unless LA_TC_SWEEP says otherwise (0: never, 1: always), when its estimated time is below
// the two walks'.
bool tc_sweep_chosen(const Plan &p, int nsm);
// The single sweep: one launch, one CTA per head (heads beyond the grid loop).
cudaError_t tc_backward_sweep(const Plan &p, tc::TcParams &P, const void *O, void *dQ, void *dK, void *dV,
                              unsigned char *ws, cudaStream_t s);

// bf16 with D = 256: the tcgen05 kernels of la_tc_wide.cu (one CTA per head and 128-column output half).
bool wide_supported(const Plan &p);
// keep_g: the workspace is sized for the backward; g_i is also kept there, with a record of Q, K and shape.
cudaError_t wide_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                         unsigned char *ws, cudaStream_t s, bool keep_g);
// Reads O (the forward's output) for dt_i = dO_i . O_i / g_i; the workspace holds g, dt and dO / g.
// reuse_g: take g from the forward (record checked on the device, LA_ERR_STATE when it does not match)
// instead of recomputing it.
cudaError_t wide_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O,
                          const void *dO, void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s,
                          bool reuse_g);

}  // namespace la
