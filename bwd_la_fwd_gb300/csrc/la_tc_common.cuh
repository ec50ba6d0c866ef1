// la_tc_common.cuh -- work decomposition and small helpers shared by the tensor-core (tcgen05) kernels.
//
// Work split.  A head's N rows are cut into chunks of kC = 128 rows (the M of one tcgen05 MMA).  All
// (head, chunk) pairs are laid end to end, head-major, and the resulting list of T chunks is cut into
// G contiguous slices, one per CTA: CTA b owns chunks [lo(b), lo(b+1)) with lo(b) = floor(b T / G).
// With 64 heads and 152 SMs this keeps every SM busy (each slice is ~13.5 chunks and may straddle a head
// boundary) where one CTA per head would leave most SMs idle.  The part of a slice that lies in one head
// is a "piece".  A piece's D x D state sum is stored in workspace slot (head + b): the slots of one CTA's
// pieces are consecutive and never collide with another CTA's, and a head's slots are found from the
// CTAs that cover it.  A small kernel between two walks turns each head's slots into the state carried
// into each piece (the sum over its earlier pieces, its later pieces, or all of them), so no CTA ever
// waits for another inside a kernel.
#pragma once

#include <stdint.h>

#include "la_sm100.cuh"

namespace la {
namespace tc {

constexpr int kC = 128;               // rows per chunk
constexpr int kMaxCtas = 160;         // upper bound on G (>= the 152 SMs of a GB300) used to size the workspace
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single barrier wait

struct Slices {
    long long T;  // total chunks = BH * nchunk
    int G;        // CTAs
    int nchunk;   // chunks per head
};

__host__ __device__ __forceinline__ long long slice_lo(const Slices &s, int b) { return (long long)b * s.T / s.G; }

// CTAs for BH heads of nchunk chunks on nsm SMs.  By default every SM gets a slice, G = min(T, nsm)
// (at most kMaxCtas); slices then straddle head boundaries, and a CTA whose slice does pays a fixed cost
// where its pieces change (the pipeline drained and refilled, the carried state loaded), measured at
// less than one chunk of a causal walk (whose piece changes lead into a zero carry, with no load) and
// about two of a non-causal walk.  When BH k CTAs fit for a divisor k of nchunk, every slice is
// nchunk / k chunks of one head; for full-width heads (D = 128, whose walks share the HBM bandwidth, so
// that fewer CTAs lose little) that split is taken when it gives a CTA no more chunks than the default
// (causal) or at most two more (non-causal).  Narrow heads (D = 32, 64: a half or a quarter of the bytes per
// chunk) measured slower with fewer CTAs and keep the default.  The forward and the backward of one
// mask choose alike.
__host__ __device__ inline long long choose_ctas(long long BH, int nchunk, int nsm, bool causal, bool full_width) {
    const long long T = BH * nchunk;
    long long G = T < nsm ? T : nsm;
    if (G > kMaxCtas) G = kMaxCtas;
    if (G < 1) G = 1;
    if (!full_width) return G;
    for (long long k = nchunk; k >= 1; --k) {  // the largest k that divides nchunk with BH k <= G
        if (nchunk % k != 0 || BH * k > G) continue;
        const long long extra = nchunk / k - (T + G - 1) / G;
        if (BH * k != G && extra <= (causal ? 0 : 2)) G = BH * k;
        break;
    }
    return G;
}

// The CTA whose slice contains flat chunk x: the largest b with floor(b T / G) <= x, i.e. b T < (x + 1) G.
__host__ __device__ __forceinline__ int cta_of(const Slices &s, long long x) {
    const long long b = ((x + 1) * s.G - 1) / s.T;
    return (int)(b < s.G - 1 ? b : s.G - 1);
}

// float4 elements of a slot's data: the D x D matrix and the two D-vectors (D = 128).
constexpr int kSlotF4 = (128 * 128 + 2 * 128) / 4;

// Workspace slot of CTA b's piece of head h.
__host__ __device__ __forceinline__ long long slot_of(long long h, int b) { return h + b; }

// Layout of a slot's D x D matrix (D = 128): the float4 holding columns [4 (16 hf + q), +4) of row d is
// float4 number (2 q + hf) * 128 + d, so that one float4 of a half of all 128 rows is contiguous and the
// threads that own rows d (one per TMEM lane) read or write it in one coalesced access.  The two D-vectors
// follow at float offsets D*D and D*D + D.
__host__ __device__ __forceinline__ long long slot_f4(int d, int hf, int q) {
    return (long long)(2 * q + hf) * 128 + d;
}

struct Piece {
    long long h;  // head (b * H + h flattened)
    int a, e;     // chunk range [a, e) within the head
};

// Iterates over the pieces of CTA b's slice: call first(), then next() while valid.
struct PieceIter {
    long long x, hi;
    int nchunk;
    __host__ __device__ __forceinline__ PieceIter(const Slices &s, int b)
        : x(slice_lo(s, b)), hi(slice_lo(s, b + 1)), nchunk(s.nchunk) {}
    __host__ __device__ __forceinline__ bool valid() const { return x < hi; }
    __host__ __device__ __forceinline__ Piece get() const {
        Piece p;
        p.h = x / nchunk;
        p.a = (int)(x - p.h * nchunk);
        const long long hend = (p.h + 1) * nchunk;
        p.e = (int)((hi < hend ? hi : hend) - p.h * nchunk);
        return p;
    }
    __host__ __device__ __forceinline__ void next() {
        const Piece p = get();
        x = p.h * nchunk + p.e;
    }
};

// The same pieces in reverse: the slice's last piece first (its chunks [a, e) as above).
struct RevPieceIter {
    long long lo, x;
    int nchunk;
    __host__ __device__ __forceinline__ RevPieceIter(const Slices &s, int b)
        : lo(slice_lo(s, b)), x(slice_lo(s, b + 1)), nchunk(s.nchunk) {}
    __host__ __device__ __forceinline__ bool valid() const { return x > lo; }
    __host__ __device__ __forceinline__ Piece get() const {
        Piece p;
        p.h = (x - 1) / nchunk;
        const long long hs = p.h * nchunk;
        p.a = (int)((lo > hs ? lo : hs) - hs);
        p.e = (int)(x - hs);
        return p;
    }
    __host__ __device__ __forceinline__ void next() {
        const Piece p = get();
        x = p.h * nchunk + p.a;
    }
};

// Records the first device-side error in the workspace status word (first error wins).
__device__ __forceinline__ void report(uint32_t *status, uint32_t code, uint32_t where) {
    if (atomicCAS(status, 0u, code) == 0u) status[1] = where;
}

// Per-CTA abort state in shared memory: the flag that a role sets when it gives up, and the bound on any
// single barrier wait of the launch (kWaitNs unless the launch asks for a shorter one).  `flag` is the
// first member, so the kernels pass a pointer to it and the wait finds the bound beside it.
struct AbortState {
    int flag;
    int pad;
    uint64_t limit_ns;
};

// Barrier wait bounded in time and aborted early when another role of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t *status, uint32_t where) {
    if (sm100::mbar_try_wait(bar, parity)) return true;
    const uint64_t limit = reinterpret_cast<volatile AbortState *>(abort_flag)->limit_ns;
    const uint64_t t0 = sm100::globaltimer_ns();
    while (true) {
        if (sm100::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (sm100::globaltimer_ns() - t0 > limit) {
            *abort_flag = 1;
            report(status, 5u, where);
            return false;
        }
    }
}

// Index check of the LA_CHECKED build, for every global-memory index a thread computes itself: an index
// outside [0, n) records LA_ERR_BOUNDS (6) with the place `where` in the workspace status word, and the
// caller skips the access (a load then reads 0).  Tensor-map (TMA) copies need no such check: the maps
// clip them to the operand's extents.  In the normal build the check is the constant true.
__device__ __forceinline__ bool in_range(long long i, long long n, uint32_t *status, uint32_t where) {
#ifdef LA_CHECKED
    if (i >= 0 && i < n) return true;
    report(status, 6u, where);
    return false;
#else
    (void)i;
    (void)n;
    (void)status;
    (void)where;
    return true;
#endif
}

// Byte offset of the 16-byte group holding element column `col8 * 8` of row `row` in a tile written by
// TMA with the 128-byte swizzle (rows of 128 bytes = 64 bf16; group index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int col8) {
    return (uint32_t)row * 128u + (uint32_t)(((col8 ^ row) & 7) << 4);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace tc
}  // namespace la
