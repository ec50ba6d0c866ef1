// la_internal.h -- declarations shared by the CUDA translation units of the library (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace la {

constexpr int kMaxDevices = 64;

// Runs `set` once for the current device and remembers how it ended (state[dev]: 0 not yet, 1 done,
// -1 failed).  Function attributes such as the dynamic shared-memory limit belong to the current
// device's context, so a process that uses several devices sets them on each.  Two threads that race on
// a device's first call both run `set`, which only repeats an idempotent setting.
template <typename F> bool once_per_device(std::atomic<int> *state, F set) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    int s = state[dev].load(std::memory_order_acquire);
    if (s == 0) {
        s = set() ? 1 : -1;
        state[dev].store(s, std::memory_order_release);
    }
    return s > 0;
}

// Device status codes written into the workspace's sticky status word (same values as la_status).
enum : uint32_t { kDevOk = 0, kDevTimeout = 5, kDevBounds = 6, kDevState = 7 };

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
    uint32_t status;      // sticky device status (first error wins); cleared by la_get_status
    uint32_t info[7];     // where the first error happened (kernel id, block, step), for debugging
    uint32_t wide_skip;   // D = 256 backward: its row kernel found no matching forward record, skip the rest
    uint32_t fwd_sums_used; // a backward has put its reverse sums where the recorded forward sums were
    uint32_t fwd_terms_kept; // the recorded causal forward also kept g and each head's total state (a
                             // backward-sized workspace): the single-sweep backward can run on them
    uint32_t bwd_skip;    // tensor-core backward: its dQ walk found no usable forward record, so the
                          // dK / dV walk after it computes nothing either
    uint32_t reserved[20];
    uint64_t state_tag[7]; // which operands and work split the saved sums (or g) belong to, and their form
};
static_assert(sizeof(WsHeader) <= 256, "workspace header must fit in 256 bytes");
static_assert(offsetof(WsHeader, state_tag) == 128, "the state tag sits 128 bytes into the header");

// Element strides of one [B,H,N,D] operand: batch, head and row; the D elements of a row are contiguous.
struct Layout {
    long long sb, sh, sn;
};
enum Operand : int { kOpQ = 0, kOpK, kOpV, kOpO, kOpdO, kOpdQ, kOpdK, kOpdV, kNumOps };

// How one call splits each head's N rows into segments whose D x D states are carried in the
// workspace.  Chosen on the host from (N, D) only, so la_workspace_bytes and the launch agree.
struct Plan {
    int B, H, N, D, causal, dtype;
    int BH;
    int seg_len;        // rows per segment
    int nseg;           // segments per head
    long long stride;   // elements per segment state (S or P: D*D, then two D-vectors), padded
    int acc_bytes;      // accumulator element size: 4 (bf16 storage) or 8 (fp32 storage)
    size_t off_states;  // byte offsets of the workspace regions
    size_t off_states2; // tensor-core backward: reverse-direction slots
    size_t off_flags;
    size_t off_rowstats;
    size_t off_chunkye; // tensor-core causal backward: each chunk's column sums y_c, e_c
    size_t off_chunkza; // tensor-core path: each chunk's column sums z_c = sum k_j, a_c = sum v_j
    size_t off_htot;    // tensor-core path, backward-sized: each head's total state (one slot per head)
    size_t bytes_fwd;   // workspace bytes for the forward / for the backward
    size_t bytes_bwd;
    bool use_tc;        // tcgen05 kernels for bf16 with D <= 128 rather than the SIMT kernels
    bool use_wide;      // tcgen05 kernels for bf16 with D = 256
    Layout lay[kNumOps]; // strides of each operand (make_plan: contiguous [B,H,N,D])
};

// Host-side count of kernels launched by the library (la_launch_count).
void count_launches(unsigned n);

bool make_plan(int B, int H, int N, int D, int causal, int dtype, Plan *p);

// SIMT path (fp32 FFMA, any supported D, fp32 or bf16 storage).
cudaError_t simt_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                         unsigned char *ws, cudaStream_t s);
cudaError_t simt_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O,
                          const void *dO, void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s);

}  // namespace la
