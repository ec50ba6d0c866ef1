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

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Loads the state carried into a piece (sum of slots b_from..b_to-1 of head h) for TMEM lane / row d:
// row d of the D x D sum into TMEM (if to_tmem) and, rounded to bf16, into row d of the operand tile Sb
// (two 64-column boxes, 128-byte swizzle); the two vector sums into zc[d] and ac[d].
__device__ __forceinline__ void load_carry(const float *slots, long long slot_stride, long long h, int b_from, int b_to, int d,
                                           uint32_t tS, unsigned char *Sb, float *zc, float *ac, bool to_tmem) {
    constexpr int D = 128;
#pragma unroll 1
    for (int c16 = 0; c16 < D / 16; ++c16) {
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
        for (int b = b_from; b < b_to; ++b) {
            const float4 *src = (const float4 *)(slots + slot_of(h, b) * slot_stride + (size_t)d * D + c16 * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = src[q];
                acc[4 * q] += v.x;
                acc[4 * q + 1] += v.y;
                acc[4 * q + 2] += v.z;
                acc[4 * q + 3] += v.w;
            }
        }
        if (to_tmem) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(acc[j]);
            tmem_st16(tS + c16 * 16, r);
        }
        // bf16 copy: row d of an MN-major operand, columns e = c16*16 .. +15 (two 16-byte groups)
        unsigned char *tile = Sb + (c16 / 4) * kBox;
        const int col8 = (c16 % 4) * 2;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
            uint4 v;
            v.x = pack_bf16(acc[8 * g2 + 0], acc[8 * g2 + 1]);
            v.y = pack_bf16(acc[8 * g2 + 2], acc[8 * g2 + 3]);
            v.z = pack_bf16(acc[8 * g2 + 4], acc[8 * g2 + 5]);
            v.w = pack_bf16(acc[8 * g2 + 6], acc[8 * g2 + 7]);
            *(uint4 *)(tile + sw128_off(d, col8 + g2)) = v;
        }
    }
    float z = 0.f, a = 0.f;
    for (int b = b_from; b < b_to; ++b) {
        const float *sl = slots + slot_of(h, b) * slot_stride;
        z += sl[(size_t)D * D + d];
        a += sl[(size_t)D * D + D + d];
    }
    zc[d] = z;
    ac[d] = a;
    if (to_tmem) tmem_st_wait();
}

}  // namespace tc
}  // namespace la
