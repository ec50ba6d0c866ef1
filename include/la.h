/*
 * la.h -- C ABI of the GB300 (sm_103a) normalised linear-attention library.
 *
 * Operation.  "Transformer Based Linear Attention with Optimized GPU Kernel Implementation"
 * (A. Gerami, R. Duraiswami, arXiv 2510.21956) describes a linear-attention (LA) head over N tokens,
 * each embedded in a D-dimensional head (shd-paper.top page, abstract), with a forward/backward
 * formulation, a normalisation scheme and analytical gradients, in O(N D^2) time and O(N D) memory
 * (sciencestack.ai page, TL;DR).  The pages print no formula; this library computes, for every
 * (batch b, head h) independently and with rows i, j = 0..N-1:
 *
 *   W_ij = m_ij (1 + q_i . k_j),  m_ij = [j <= i] if causal else 1
 *   g_i  = sum_j W_ij                                  (the normaliser)
 *   O_i  = sum_j W_ij v_j / g_i
 *
 * and the exact gradients of L = sum_i dO_i . O_i with respect to Q, K and V.  The N x N weights are
 * never formed: the kernels carry D x D running states, as the O(N D^2) / O(N D) claims require.
 *
 * Layout.  Q, K, V, O, dO, dQ, dK, dV are dense, contiguous [B, H, N, D] tensors of one element
 * type (LA_F32 = float, LA_BF16 = bfloat16), element (b, h, i, d) at ((b H + h) N + i) D + d (the
 * *_strided entry points take other layouts).  The
 * normaliser is float [B, H, N].  bf16 storage accumulates in fp32, fp32 storage in fp64.  Supported:
 * B, H >= 1 (B*H < 2^31), N >= 1 (B*H*N*D < 2^40), D in {16, 32, 64, 128, 256}.  bf16 with D = 32, 64,
 * 128 runs on the tensor-core kernels of 128 columns (D < 128 zero-extended), bf16 with D = 256 on the wide
 * tensor-core kernels (one CTA per head and 128-column output half); fp32 storage and bf16 with D = 16 run
 * on the CUDA-core (SIMT) kernels.
 *
 * Memory.  Every pointer is a DEVICE pointer except where stated.  The caller owns every buffer; the
 * library never allocates device or host memory and never synchronises the stream (except
 * la_get_status).  Scratch comes from the caller's workspace, whose size is la_workspace_bytes().
 * The workspace must be 256-byte aligned and zero-filled before its first use (cudaMemset or
 * torch.zeros); the library keeps it in a reusable state afterwards.  One workspace must not be used
 * by two calls that can run at the same time.  Outputs must not alias inputs or each other.
 *
 * Streams.  Work is enqueued on `stream` (a cudaStream_t; NULL means the legacy default stream) and
 * the call returns without waiting for it.
 *
 * Errors.  Every entry point returns an la_status.  Argument errors are found on the host before any
 * work is enqueued (nothing is launched).  A launch failure returns LA_ERR_CUDA.  Conditions found on
 * the device (a bounded wait that ran out, a misaligned shared-memory window, a backward that found no
 * matching forward state) are recorded in a sticky status word inside the workspace and reported by
 * la_get_status().  Nothing is thrown across the ABI.
 */
#ifndef LA_GB300_H
#define LA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, aliasing outputs */
    LA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (e.g. an unsupported D) */
    LA_ERR_WORKSPACE = 3,   /* workspace null, misaligned or smaller than la_workspace_bytes() */
    LA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    LA_ERR_TIMEOUT = 5,     /* device: a bounded barrier wait inside a kernel gave up (reported by la_get_status) */
    LA_ERR_BOUNDS = 6,      /* device: an internal layout check failed -- a kernel's shared-memory window was not
                               1024-byte aligned, so it computed nothing; or, in the index-checked test build
                               (libla_gb300_checked.so), an index out of its array was skipped (reported by
                               la_get_status) */
    LA_ERR_STATE = 7        /* device: la_backward_with_forward_state found no matching forward state */
} la_status;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* Library ABI version (major * 100 + minor). */
int la_version(void);

/* Number of CUDA kernels this library has launched in this process (all devices, all calls).  Host
 * counter, incremented at each successful launch; lets a caller count the library's launches inside a
 * timed region. */
unsigned long long la_launch_count(void);

/* Human-readable name of a status code; never NULL. */
const char *la_status_string(int status);

/*
 * Bytes of device workspace that la_forward (backward = 0) or la_backward (backward = 1) needs for
 * this problem.  Host-only, never touches the GPU.  Returns 0 for an invalid or unsupported request.
 * A workspace sized with backward = 1 also serves la_forward on the same shape.
 */
size_t la_workspace_bytes(int B, int H, int N, int D, int causal, int dtype, int backward);

/*
 * Forward pass (sciencestack.ai page, TL;DR: the LA forward pass with its normalisation scheme).
 *   Q, K, V     in : [B,H,N,D] of `dtype`
 *   causal      in : nonzero selects the causal mask j <= i
 *   O           out: [B,H,N,D] of `dtype`, O_i = sum_j W_ij v_j / g_i, rounded once (nearest-even)
 *   normaliser  out: float [B,H,N] with g_i, or NULL to skip it
 *   workspace   in/out: device scratch of workspace_bytes >= la_workspace_bytes(..., backward = 0)
 * Pointers must be 16-byte aligned.  On the tensor-core paths the forward leaves in the workspace what
 * la_backward_with_forward_state reuses: the per-piece sums; when the workspace is backward-sized
 * (workspace_bytes >= la_workspace_bytes(..., backward = 1)) also the normaliser g and, causal with
 * D <= 128, each head's total state, which the single-sweep causal backward starts from.
 */
int la_forward(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B, int H,
               int N, int D, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass (sciencestack.ai page, TL;DR: analytical gradients of the LA head).
 *   Q, K, V, O, dO  in : [B,H,N,D] of `dtype`; O is the forward output, dO = dL/dO
 *   dQ, dK, dV      out: [B,H,N,D] of `dtype`, the gradients of L = sum dO . O
 *   causal          in : must match the forward call
 *   workspace       in/out: workspace_bytes >= la_workspace_bytes(..., backward = 1)
 * For D <= 128, O must be a valid buffer but is not read: the backward recomputes the normaliser g_i and
 * the row terms delta_i = dO_i . O_i from Q, K and V in its accumulator precision, which is both exact to
 * that precision (the stored O is rounded to `dtype`) and one tensor read fewer.  For bf16 with D = 256
 * the backward recomputes g_i and reads O for delta_i, so O must hold la_forward's output for these
 * inputs.  Pointers must be 16-byte aligned.
 */
int la_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ, void *dK,
                void *dV, int causal, int B, int H, int N, int D, int dtype, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Backward pass that reuses what the forward computed.  The forward's first kernel sums k_j v_j^T, k_j
 * and v_j over each piece of rows (the tensor-core path's work split), and both passes need exactly those
 * sums; la_backward recomputes them, this entry point takes them from `workspace` instead, the way an
 * autograd backward takes tensors saved by its forward.  Arguments, checks and results are those of
 * la_backward, with one more condition: the last call on this workspace must have been la_forward on the
 * same K and V buffers (same pointers, unchanged contents) and the same B, H, N, D, dtype and mask.  A
 * backward uses those sums up (it keeps its own reverse-direction sums in the same slots), so each reusing
 * backward needs a forward of its own.  The workspace records which K, V and shape its sums belong to;
 * when the record does not match, the kernels compute nothing and la_get_status reports LA_ERR_STATE.
 * Unchanged contents cannot be checked and are the caller's promise.  Causal on the tensor-core
 * kernels (bf16, D = 32, 64, 128) the call also takes the normaliser g, which la_forward keeps only in a
 * backward-sized workspace, and forms delta_i = dO_i . O_i from O: after a forward given a forward-sized
 * workspace it reports LA_ERR_STATE and computes nothing.  With D = 128 it may run as one reverse sweep
 * per head ("single-sweep causal backward": dQ, dK and dV of each chunk together, Q, K, V, O and dO read
 * once, starting from each head's total state, which la_forward keeps beside g) where that is estimated
 * faster than the two walks, i.e. when the heads fill the GPU (B H of about 100 and more; the
 * environment variable LA_TC_SWEEP = 0 or 1 forbids or forces it).  The causal results equal
 * la_backward's to within rounding, not bit for bit (la_backward forms g and delta from the carried
 * state).  On the SIMT path (fp32 storage, or bf16 with D = 16) there are no such sums to reuse and
 * this call is la_backward.  On the wide path (bf16 with
 * D = 256) the forward forms no piece sums; what is reused there is the normaliser g_i, which la_forward
 * keeps in the workspace when that workspace is backward-sized (la_workspace_bytes(..., backward = 1)),
 * under a record of Q's and K's addresses and strides, the shape and the mask.  A mismatch is
 * LA_ERR_STATE with nothing computed, as above; g is not used up, so several backwards may follow one
 * forward there.
 */
int la_backward_with_forward_state(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                   void *dQ, void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Strided operands: the same passes on tensors laid out other than [B,H,N,D], with no transpose copy --
 * [B,N,H,D] as a projection writes it, or the Q, K and V slices of one fused [B,N,3,H,D] projection
 * output (the LA layer's projections precede the head, shd-paper.top page, abstract).
 *   strides  in : host array, three element strides per operand, in the operands' argument order --
 *                 (batch, head, row) for Q, K, V, O (forward: 12 values) or Q, K, V, O, dO, dQ, dK, dV
 *                 (backward: 24 values); NULL means every operand is contiguous [B,H,N,D].
 * The D elements of a row are contiguous.  Every stride must be a multiple of 16 bytes, and an operand's
 * rows must not overlap one another: ordered by stride, the dimensions of extent > 1 must nest (the
 * smallest stride >= D, each larger one >= the previous stride times its extent).  Inputs may share
 * memory (a fused QKV tensor); an output may not meet an input, another output or the workspace, which
 * is checked element-exactly for operands of equal strides and by address range otherwise.  The
 * normaliser stays contiguous float [B,H,N].  Violations return LA_ERR_INVALID_ARG before any work.
 * la_backward_strided with reuse_forward_state != 0 is la_backward_with_forward_state; the record of the
 * forward's sums then also covers K's and V's strides.  Results are those of the contiguous calls on the
 * same values.
 */
int la_forward_strided(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B,
                       int H, int N, int D, int dtype, const long long *strides, void *workspace,
                       size_t workspace_bytes, void *stream);
int la_backward_strided(const void *Q, const void *K, const void *V, const void *O, const void *dO, void *dQ,
                        void *dK, void *dV, int causal, int B, int H, int N, int D, int dtype, const long long *strides,
                        int reuse_forward_state, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Forward pass without a caller-supplied workspace, for callers that cannot allocate device memory (a
 * plugin that its host framework gives only input and output buffers, code that must not call cudaMalloc
 * because it can block and synchronise the device, a fixed memory budget).  The paper has no counterpart:
 * this is a packaging variant of la_forward.  Arguments and results are those of la_forward; the scratch
 * is a fixed device array of LA_NOALLOC_SCRATCH_BYTES inside the library, held on every device that loads
 * it until the process exits.  Nothing is allocated.
 *   - Returns LA_ERR_WORKSPACE, before enqueuing anything, when la_workspace_bytes(B, H, N, D, causal,
 *     dtype, 0) exceeds LA_NOALLOC_SCRATCH_BYTES; every other argument error is found on the host before
 *     anything is enqueued, as for la_forward.
 *   - The first call on a device looks up the array's device address and clears its status header (a
 *     cudaMemset and a device synchronisation); make it before any stream capture.
 *   - Device-side conditions are recorded in the array's sticky status word: la_noalloc_get_status
 *     reads and clears it.
 *   - All calls on a device share the array: calls whose work overlaps on the GPU race.
 */
#define LA_NOALLOC_SCRATCH_BYTES (32u << 20)
int la_forward_noalloc(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser, int B,
                       int H, int N, int D, int dtype, void *stream);

/*
 * la_get_status for the fixed scratch array of la_forward_noalloc on the current device: synchronises
 * `stream`, then returns and clears the sticky device status left by earlier la_forward_noalloc calls
 * (LA_OK when no call has run on this device yet), or LA_ERR_CUDA if the stream failed.
 */
int la_noalloc_get_status(void *stream);

/*
 * Recurrent (decode) form of the causal head.  The causal forward carries, per (b, h), the state of the
 * tokens taken so far (sciencestack.ai page, TL;DR: O(N D^2) time with an O(D^2) state); a decoder can
 * keep that state and take one token at a time instead of re-running the forward:
 *   S = sum_j k_j v_j^T  (S[d][e] = sum_j k_j[d] v_j[e]),  z = sum_j k_j,  a = sum_j v_j,  n = count.
 * State arrays (device, owned by the caller, updated in place; zero-filled = the empty state):
 *   S  [B,H,D,D],  z [B,H,D],  a [B,H,D]  of the accumulator type: float for LA_BF16, double for LA_F32
 *   n  int [B,H]
 * Rows are independent over (b, h); different heads may hold different counts n.  Pointers must be
 * 16-byte aligned, the state arrays must not overlap each other or any token input or output.  Neither
 * call needs a workspace or reports device-side status.
 */

/*
 * One token per (b, h): appends (k, v) to the state, then
 *   g = n + q . z,   o = (a + S^T q) / g        (state after the append; o rounded once to dtype)
 * which is row n - 1 of la_forward(causal = 1) over the tokens taken so far.
 *   q, k, v     in : [B,H,D] of `dtype`
 *   o           out: [B,H,D] of `dtype`
 *   normaliser  out: float [B,H] with g, or NULL
 */
int la_decode_step(const void *q, const void *k, const void *v, void *o, float *normaliser, void *S, void *z,
                   void *a, int *n, int B, int H, int D, int dtype, void *stream);

/*
 * Appends N >= 0 tokens per (b, h) to the state (a prompt, or a block of tokens whose outputs the caller
 * takes from la_forward): S += K^T V, z += sum k, a += sum v, n += N.
 *   K, V  in : [B,H,N,D] of `dtype` (may be NULL when N = 0)
 */
int la_state_append(const void *K, const void *V, void *S, void *z, void *a, int *n, int B, int H, int N, int D,
                    int dtype, void *stream);

/*
 * Synchronises `stream`, then returns and clears the sticky device status recorded in `workspace`
 * by earlier calls (LA_OK, LA_ERR_TIMEOUT, LA_ERR_BOUNDS or LA_ERR_STATE), or LA_ERR_CUDA if the stream
 * failed.
 */
int la_get_status(void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LA_GB300_H */
