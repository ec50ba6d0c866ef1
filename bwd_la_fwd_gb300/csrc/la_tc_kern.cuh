// la_tc_kern.cuh -- device helpers shared by the tcgen05 forward and backward kernels.
#pragma once

#include "la_tc_common.cuh"

namespace la {
namespace tc {

using namespace sm100;

constexpr uint32_t kBox = kC * 128;  // bytes of one TMA box: 128 rows x 64 bf16

__device__ __forceinline__ unsigned char *smem_base(unsigned char *raw, uint32_t *status, bool *ok) {
    // Every tile here needs 1024-byte alignment (128-byte swizzle atoms); the dynamic window is checked
    // rather than padded, because the forward kernel uses all but a few hundred bytes of shared memory.
    *ok = (smem_u32(raw) & 1023u) == 0;
    if (!*ok && threadIdx.x == 0) report(status, 6u, 0xA11Du);
    return raw;
}

// Tile (columns [x, x + 64), rows [row, row + 128)) of one head of an operand.  The kernels come in two
// forms.  FLAT: every operand's batch stride is H times its head stride (contiguous [B,H,N,D] among
// others), the maps are 3-D over {D, N, B H} and a head is its flat index bh = b H + h.  Otherwise the
// maps are 4-D over {D, N, H, B} with the caller's strides ([B,N,H,D], a head slice of a fused QKV
// tensor...).  head_coord turns bh into the coordinates of the form, once per piece.
struct HeadCoord {
    int h, b;
};
template <bool FLAT> __device__ __forceinline__ HeadCoord head_coord(long long bh, int H) {
    if (FLAT) return HeadCoord{(int)bh, 0};
    const unsigned u = (unsigned)bh;  // B H < 2^31
    return HeadCoord{(int)(u % (unsigned)H), (int)(u / (unsigned)H)};
}
template <bool FLAT>
__device__ __forceinline__ void tile_load(void *dst, const CUtensorMap *m, uint64_t *bar, int x, int row,
                                          HeadCoord hc) {
    if constexpr (FLAT) tma_load_3d(dst, m, bar, x, row, hc.h);
    else tma_load_4d(dst, m, bar, x, row, hc.h, hc.b);
}
template <bool FLAT> __device__ __forceinline__ void tile_prefetch(const CUtensorMap *m, int x, int row, HeadCoord hc) {
    if constexpr (FLAT) tma_prefetch_3d(m, x, row, hc.h);
    else tma_prefetch_4d(m, x, row, hc.h, hc.b);
}
template <bool FLAT>
__device__ __forceinline__ void tile_store(const CUtensorMap *m, const void *src, int x, int row, HeadCoord hc) {
    if constexpr (FLAT) tma_store_3d(m, src, x, row, hc.h);
    else tma_store_4d(m, src, x, row, hc.h, hc.b);
}


// Issues the TMA stores of a two-box output tile from shared memory (the boxes that hold the operand's
// columns: nbox of them) and commits them.  One thread.
template <bool FLAT>
__device__ __forceinline__ void store_tile(const CUtensorMap *map, const unsigned char *tile2, int row0, HeadCoord hc,
                                           int nbox) {
    tile_store<FLAT>(map, tile2, 0, row0, hc);
    if (nbox > 1) tile_store<FLAT>(map, tile2 + kBox, 64, row0, hc);
    bulk_commit();
}

constexpr int kEpiThreads = 256;  // eight epilogue warps: two per TMEM lane quarter
__device__ __forceinline__ void epi_sync256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Which of a head's pieces make up the state carried into a piece.
// Half `hf` of the state carried into CTA b's piece of head h, from the piece's own slot ([S (slot_f4
// layout) | z | a], fp32), which tc_combine_kernel has set to the sum over the head's earlier pieces,
// later pieces or all of them.  Row d, columns [64 hf, 64 hf + 64) of S go into TMEM (if to_tmem) and,
// as bf16, into box hf of the operand tile Sb.  Half 0 also writes z[d] to zc (and TMEM column tZ if
// to_tmem && vec_to_tmem), half 1 writes a[d] to ac (and column tA).
static __device__ __forceinline__ void load_carry_half(const float *slots, long long stride, long long h, int b, int d,
                                                int hf, uint32_t tS, uint32_t tZ, uint32_t tA, unsigned char *Sb,
                                                float *zc, float *ac, bool to_tmem, bool vec_to_tmem) {
    constexpr int D = 128;
    const float *slot = slots + slot_of(h, b) * stride;
    const float4 *src = (const float4 *)slot;
    float4 v4[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v4[q] = src[slot_f4(d, hf, q)];  // coalesced over the rows d of a warp
    const float vsum = slot[(size_t)D * D + hf * D + d];
    const float *acc = (const float *)v4;
#pragma unroll
    for (int half32 = 0; half32 < 2; ++half32) {
        const float *a32 = acc + 32 * half32;
        if (to_tmem) {
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(a32[j]);
            tmem_st32(tS + 64 * hf + 32 * half32, r);
        }
        unsigned char *tile = Sb + hf * kBox;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            uint4 w;
            w.x = pack_bf16(a32[8 * g4 + 0], a32[8 * g4 + 1]);
            w.y = pack_bf16(a32[8 * g4 + 2], a32[8 * g4 + 3]);
            w.z = pack_bf16(a32[8 * g4 + 4], a32[8 * g4 + 5]);
            w.w = pack_bf16(a32[8 * g4 + 6], a32[8 * g4 + 7]);
            *(uint4 *)(tile + sw128_off(d, 4 * half32 + g4)) = w;
        }
    }
    (hf == 0 ? zc : ac)[d] = vsum;
    if (to_tmem && vec_to_tmem) tmem_st1(hf == 0 ? tZ : tA, __float_as_uint(vsum));
    if (to_tmem) tmem_st_wait();
}

// Value v of index e (0 <= e < 128) into an N = 16 MMA operand along its K dimension: two 8-row boxes of
// 128-byte rows in the 128-byte swizzle (indices e < 64 in the first box), row 0 = bf16(v), row 1 =
// bf16(v - row 0), rows 2-7 zero (set once by the caller).  An MMA against it puts sum_e v_e x_e, in two
// parts that add up to ~16 significant bits of v, into output columns 0 and 1.
__device__ __forceinline__ void split_tile_put(unsigned char *tile, int e, float v) {
    unsigned char *bx = tile + (e >> 6) * 1024;
    const int r = e & 63;
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    *(__nv_bfloat16 *)(bx + ((r >> 3) << 4) + (r & 7) * 2) = h;              // row 0: 16-byte group r / 8
    *(__nv_bfloat16 *)(bx + 128 + (((r >> 3) ^ 1) << 4) + (r & 7) * 2) = l;  // row 1: group index XOR 1
}

// Multiplies row `row` of box hf of a bf16 tile by s in place.
__device__ __forceinline__ void scale_row_half(unsigned char *tile2, int row, int hf, float s) {
    unsigned char *tile = tile2 + hf * kBox;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        uint4 *p4 = (uint4 *)(tile + sw128_off(row, g8));
        uint4 w = *p4;
        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
        for (int q = 0; q < 4; ++q) wv[q] = pack_bf16(bf16lo(wv[q]) * s, bf16hi(wv[q]) * s);
        *p4 = w;
    }
}

// The same for a piece whose carried state is zero by definition (a causal piece that starts its head
// walking forward, or ends it walking in reverse): zeros instead of a slot read.
static __device__ __forceinline__ void zero_carry_half(int d, int hf, uint32_t tS, unsigned char *Sb, float *zc,
                                                float *ac, bool to_tmem) {
    if (to_tmem) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
        tmem_st32(tS + 64 * hf, r);
        tmem_st32(tS + 64 * hf + 32, r);
    }
    unsigned char *tile = Sb + hf * kBox;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) *(uint4 *)(tile + sw128_off(d, g8)) = make_uint4(0u, 0u, 0u, 0u);
    (hf == 0 ? zc : ac)[d] = 0.f;
    if (to_tmem) tmem_st_wait();
}

// Brings into L2 the carry slot of the piece that follows `pi` in the slice, when `remaining` chunks of
// the current piece are still to be issued (two, or all of a shorter piece).  The slots were written by
// an earlier kernel and the walks stream far more than L2 holds.  One thread (the TMA producer).
// `nfloats`: the slot array's extent (LA_CHECKED: a slot outside it is not prefetched).
template <typename Iter>
__device__ __forceinline__ void prefetch_next_carry(const Iter &pi, int remaining, int piece_len,
                                                    const float *slots, long long stride, int b, long long nfloats,
                                                    uint32_t *status) {
    if (remaining != (piece_len > 2 ? 2 : piece_len - 1)) return;
    Iter pn = pi;
    pn.next();
    if (!pn.valid()) return;
    const long long base = slot_of(pn.get().h, b) * stride;
    if (in_range(base, nfloats, status, 0xB0F1) && in_range(base + kSlotF4 * 4 - 1, nfloats, status, 0xB0F1))
        bulk_prefetch_l2(slots + base, (uint32_t)(kSlotF4 * sizeof(float4)));
}

// Row d's 64 columns [64 hf, 64 hf + 64) of an fp32 TMEM block, rounded into box hf of a bf16 operand tile.
__device__ __forceinline__ void tmem_half_to_tile(uint32_t taddr, unsigned char *tile2, int d, int hf) {
#pragma unroll 1
    for (int half32 = 0; half32 < 2; ++half32) {
        uint32_t v[32];
        tmem_ld32(taddr + 64 * hf + 32 * half32, v);
        tmem_wait_ld(v);
        unsigned char *tile = tile2 + hf * kBox;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[8 * g4 + 0]), __uint_as_float(v[8 * g4 + 1]));
            w.y = pack_bf16(__uint_as_float(v[8 * g4 + 2]), __uint_as_float(v[8 * g4 + 3]));
            w.z = pack_bf16(__uint_as_float(v[8 * g4 + 4]), __uint_as_float(v[8 * g4 + 5]));
            w.w = pack_bf16(__uint_as_float(v[8 * g4 + 6]), __uint_as_float(v[8 * g4 + 7]));
            *(uint4 *)(tile + sw128_off(d, 4 * half32 + g4)) = w;
        }
    }
}

// q_row . z over the 64 entries of box hf, from a bf16 Q tile (two 64-column boxes) and fp32 z.
__device__ __forceinline__ float dot_half(const unsigned char *qtile2, int row, int hf, const float *z) {
    const unsigned char *tile = qtile2 + hf * kBox;
    const float *zz0 = z + 64 * hf;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        const uint4 v = *(const uint4 *)(tile + sw128_off(row, g8));
        const float *zz = zz0 + 8 * g8;
        acc0 = fmaf(bf16lo(v.x), zz[0], acc0);
        acc1 = fmaf(bf16hi(v.x), zz[1], acc1);
        acc0 = fmaf(bf16lo(v.y), zz[2], acc0);
        acc1 = fmaf(bf16hi(v.y), zz[3], acc1);
        acc0 = fmaf(bf16lo(v.z), zz[4], acc0);
        acc1 = fmaf(bf16hi(v.z), zz[5], acc1);
        acc0 = fmaf(bf16lo(v.w), zz[6], acc0);
        acc1 = fmaf(bf16hi(v.w), zz[7], acc1);
    }
    return acc0 + acc1;
}

}  // namespace tc
}  // namespace la
