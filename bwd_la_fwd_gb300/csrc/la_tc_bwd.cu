// la_tc_bwd.cu -- tcgen05 / TMA backward of the bf16 path (D = 128).
//
// Gradients of L = sum_i dO_i . O_i ("Transformer Based Linear Attention with Optimized GPU Kernel
// Implementation", sciencestack.ai page, TL;DR: analytical gradients of the LA head).  With
// dOt_i = dO_i / g_i, dt_i = (dO_i . O_i) / g_i and dW_ij = m_ij (dOt_i . v_j - dt_i):
//   dQ_i = sum_j dW_ij k_j = S_c dOt_i - dt_i z_c + [U K]_i,           U_ij = [j <= i] dW_ij in the chunk
//   dK_j = sum_i dW_ij q_i = P_c v_j - y_c + [U^T Q]_j
//   dV_j = sum_i (1 + q_i . k_j) dOt_i = e_c + P_c^T k_j + [(P/g)^T dO]_j
// where S_c, z_c (earlier rows) are the forward state and P_c = sum q_i dOt_i^T, y_c = sum dt_i q_i,
// e_c = sum dOt_i run over the later rows.  Non-causal: every sum runs over the whole head.
//
// Three launches: the per-piece K^T V sums (shared with the forward), then the dQ walk in chunk order,
// which recomputes O_i (hence g_i and delta_i; the stored O is not read) and also writes each piece's
// reverse sums (P, y, e) and the per-row g_i, dt_i, then the dK / dV walk in reverse chunk order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include "la_internal.h"
#include "la_tc_common.cuh"
#include "la_tc_host.h"
#include "la_tc_kern.cuh"

namespace la {
namespace tc {

using namespace sm100;

// P (or U) in bf16 written over the first 64 columns of a 128-column fp32 TMEM block, in place.
// f(j, x) maps the fp32 value of column j to the bf16 operand value.
template <typename F>
__device__ __forceinline__ void tmem_to_bf16_inplace(uint32_t taddr, F f) {
#pragma unroll 1
    for (int q = 0; q < kC / 32; ++q) {
        uint32_t t0[16], t1[16], pk[16];
        tmem_ld16(taddr + 32 * q, t0);
        tmem_ld16(taddr + 32 * q + 16, t1);
        tmem_ld_wait();
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) {
            const int j = 32 * q + 2 * j2;
            const uint32_t lo = j2 < 8 ? t0[2 * j2] : t1[2 * j2 - 16];
            const uint32_t hi = j2 < 8 ? t0[2 * j2 + 1] : t1[2 * j2 - 15];
            pk[j2] = pack_bf16(f(j, __uint_as_float(lo)), f(j + 1, __uint_as_float(hi)));
        }
        tmem_st16(taddr + 16 * q, pk);
    }
    tmem_st_wait();
}

// Row `row` of the state tile (fp32 TMEM block, 128 columns) rounded into the bf16 operand tile.
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, unsigned char *tile2, int row) {
#pragma unroll 1
    for (int c16 = 0; c16 < 8; ++c16) {
        uint32_t v[16];
        tmem_ld16(taddr + c16 * 16, v);
        tmem_ld_wait();
        unsigned char *tile = tile2 + (c16 / 4) * kBox;
        const int col8 = (c16 % 4) * 2;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[8 * g2 + 0]), __uint_as_float(v[8 * g2 + 1]));
            w.y = pack_bf16(__uint_as_float(v[8 * g2 + 2]), __uint_as_float(v[8 * g2 + 3]));
            w.z = pack_bf16(__uint_as_float(v[8 * g2 + 4]), __uint_as_float(v[8 * g2 + 5]));
            w.w = pack_bf16(__uint_as_float(v[8 * g2 + 6]), __uint_as_float(v[8 * g2 + 7]));
            *(uint4 *)(tile + sw128_off(row, col8 + g2)) = w;
        }
    }
}

// Sum over the chunk's rows r of w[r] * X[r][col..col+1] for a bf16 tile X (two 64-column boxes).
__device__ __forceinline__ float2 weighted_colsum(const unsigned char *tile2, int col, const float *w) {
    const unsigned char *tile = tile2 + (col / 64) * kBox;
    const int cc = col % 64;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int r = 0; r < kC; ++r) {
        const uint32_t v = *(const uint32_t *)(tile + sw128_off(r, cc / 8) + (cc % 8) * 2);
        const float wr = w ? w[r] : 1.f;
        s0 = fmaf(wr, bf16lo(v), s0);
        s1 = fmaf(wr, bf16hi(v), s1);
    }
    return make_float2(s0, s1);
}

// Writes 16 fp32 values (x[c] + add_scale * add[c]) as bf16 into row `row`, columns 16 c16 .. +15, of a
// two-box 128B-swizzled tile (the layout the output TMA map expects).
__device__ __forceinline__ void stage16_bf16(unsigned char *tile2, int row, int c16, const uint32_t (&v)[16],
                                             const float *add, float add_scale) {
    float f[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]) + add_scale * add[j];
    unsigned char *tile = tile2 + (c16 / 4) * kBox;
    const int col8 = (c16 % 4) * 2;
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
        uint4 w;
        w.x = pack_bf16(f[8 * g2 + 0], f[8 * g2 + 1]);
        w.y = pack_bf16(f[8 * g2 + 2], f[8 * g2 + 3]);
        w.z = pack_bf16(f[8 * g2 + 4], f[8 * g2 + 5]);
        w.w = pack_bf16(f[8 * g2 + 6], f[8 * g2 + 7]);
        *(uint4 *)(tile + sw128_off(row, col8 + g2)) = w;
    }
}

// Stores 16 fp32 values (x[c] * scale + add[c]) as bf16 at dst (16-byte aligned).
__device__ __forceinline__ void store16_bf16(__nv_bfloat16 *dst, const uint32_t (&v)[16], const float *add,
                                             float add_scale, float scale) {
    uint4 w0, w1;
    float f[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = (__uint_as_float(v[j]) + add_scale * add[j]) * scale;
    w0.x = pack_bf16(f[0], f[1]);
    w0.y = pack_bf16(f[2], f[3]);
    w0.z = pack_bf16(f[4], f[5]);
    w0.w = pack_bf16(f[6], f[7]);
    w1.x = pack_bf16(f[8], f[9]);
    w1.y = pack_bf16(f[10], f[11]);
    w1.z = pack_bf16(f[12], f[13]);
    w1.w = pack_bf16(f[14], f[15]);
    uint4 *d = (uint4 *)dst;
    d[0] = w0;
    d[1] = w1;
}

// ----------------------------------------------------------------------------------------------------
// dQ walk (chunk order).  Per chunk, causal:
//   T = Q K^T -> P (bf16, TMEM) ; O = P V + Q Sb ; S += K^T V            (the forward, recomputed)
//   epilogue: O_i, g_i, delta_i ; dO tile <- dOt = dO / g (in place) ; g_i, dt_i to the workspace
//   W = dOt V^T -> U = [j <= i](W - dt_i) (bf16, TMEM) ; X = dOt Sb^T + U K ; Ppiece += Q^T dOt
//   epilogue: dQ_i = X_i - dt_i z ; y += sum dt_i q_i, e += sum dOt_i (fp32, CUDA cores)
// Non-causal: O = Q Sb and X = dOt Sb^T with the head's totals; stages hold only Q and dO.
// TMEM: R0 T/P then W/U, R1 O then X, R2 S, R3 the piece's reverse sum P.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL>
__global__ void __launch_bounds__(192, 1) tc_bwd_dq_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr int NST = CAUSAL ? 1 : 2;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = CAUSAL ? 4 * TB : 2 * TB;  // Q, dO (, K, V)
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Sb = sm + NST * STAGE;
    float *zc = (float *)(Sb + TB);
    float *ac = zc + D;
    float *sDt = ac + D;
    uint64_t *full = (uint64_t *)(sDt + kC);
    uint64_t *empty = full + NST;
    uint64_t *bar = empty + NST;
    uint64_t *barT = bar, *barP = bar + 1, *barSb = bar + 2, *barO = bar + 3, *barDt = bar + 4, *barW = bar + 5,
             *barU = bar + 6, *barX = bar + 7, *barS = bar + 8, *barPP = bar + 9, *barPPf = bar + 10,
             *barXf = bar + 11;
    uint32_t *tslot = (uint32_t *)(bar + 12);
    volatile int *abort_flag = (volatile int *)(tslot + 1);
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // MMA commit + the epilogue once its dQ tile has left the Q tile
        }
        const uint32_t counts[12] = {1, 128, 128, 1, 128, 1, 128, 1, 1, 1, 128, 128};
        for (int k = 0; k < 12; ++k) mbar_init(&bar[k], counts[k]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t R0 = tmem, R1 = tmem + 128, R2 = tmem + 256, R3 = tmem + 384;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmdO);
        if (CAUSAL) {
            prefetch_tmap(&P.tmK);
            prefetch_tmap(&P.tmV);
        }
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x301)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tma_load_3d(st + nb * kBox, &P.tmQ, &full[s], nb * 64, c * kC, (int)pc.h);
                    tma_load_3d(st + TB + nb * kBox, &P.tmdO, &full[s], nb * 64, c * kC, (int)pc.h);
                    if (CAUSAL) {
                        tma_load_3d(st + 2 * TB + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, (int)pc.h);
                        tma_load_3d(st + 3 * TB + nb * kBox, &P.tmV, &full[s], nb * 64, c * kC, (int)pc.h);
                    }
                }
            }
        }
        if (!ok) {
            for (int k = it > NST ? it - NST : 0; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKK = idesc_bf16(128, 128, false, false);
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t sb = smem_u32(Sb);
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!CAUSAL && !wait_or_abort(barSb, pno & 1, abort_flag, P.status, 0x302)) break;
            if (pno > 0 && !wait_or_abort(barPPf, (pno - 1) & 1, abort_flag, P.status, 0x303)) break;
            for (int c = pc.a; c < pc.e && ok; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x304);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qb = smem_u32(stages + s * STAGE), ob = qb + TB, kb = qb + 2 * TB, vb = qb + 3 * TB;
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // T = Q K^T
                        mma_ss(R0, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                    mma_commit(barT);
                    ok = wait_or_abort(barP, ph, abort_flag, P.status, 0x305);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // O = P V
                        mma_ts(R1, R0 + 8 * k, sdesc_sw128(vb + 2048 * k, kBox, 1024), idKM, k > 0);
                    ok = wait_or_abort(barSb, ph, abort_flag, P.status, 0x306);
                    if (!ok) break;
                    tc_fence_after();
                } else if (it > 0) {
                    ok = wait_or_abort(barXf, (it - 1) & 1, abort_flag, P.status, 0x307);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)  // O += Q Sb
                    mma_ss(R1, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + 2048 * k, kBox, 1024), idKM, (CAUSAL || k > 0) ? 1u : 0u);
                mma_commit(barO);
                if (CAUSAL && c + 1 < pc.e) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // S += K^T V
                        mma_ss(R2, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024),
                               idMM, 1u);
                }
                ok = wait_or_abort(barDt, ph, abort_flag, P.status, 0x308);  // dOt is in place of dO
                if (!ok) break;
                tc_fence_after();
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // W = dOt V^T
                        mma_ss(R0, sdesc_sw128(ob + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(vb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                    mma_commit(barW);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)  // Ppiece += Q^T dOt
                    mma_ss(R3, sdesc_sw128(qb + 2048 * k, kBox, 1024), sdesc_sw128(ob + 2048 * k, kBox, 1024), idMM,
                           (c > pc.a || k > 0) ? 1u : 0u);
                if (CAUSAL) {
                    ok = wait_or_abort(barU, ph, abort_flag, P.status, 0x309);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)  // X = dOt Sb^T
                    mma_ss(R1, sdesc_sw128(ob + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // X += U K
                        mma_ts(R1, R0 + 8 * k, sdesc_sw128(kb + 2048 * k, kBox, 1024), idKM, 1u);
                }
                mma_commit(barX);
                if (CAUSAL) mma_commit(barS);
                mma_commit(&empty[s]);
                if (c + 1 == pc.e) mma_commit(barPP);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue warps: thread <-> chunk row i (TMEM lane) and state row d (same index)
        const int lb = 32 * (warp & 3);
        const int i = lb + lane;
        const int t = threadIdx.x - 64;
        const int col = 2 * (t & 63);
        const uint32_t lo = (uint32_t)lb << 16;
        __nv_bfloat16 *dQg = (__nv_bfloat16 *)P.dQ;
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            // carried forward state of the piece, combined into its own slot by tc_scan_slots
            if (CAUSAL && it > 0) {
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x30A)) break;
                tc_fence_after();
            }
            load_carry1(P.slots + slot_of(pc.h, blockIdx.x) * P.slot_stride, i, R2 + lo, Sb, zc, ac, CAUSAL);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync();
            mbar_arrive(barSb);
            float2 ye = make_float2(0.f, 0.f);  // y (t < 64) or e (t >= 64) of this piece, two columns
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                unsigned char *qt = st, *ot = st + TB, *kt = st + 2 * TB, *vt = st + 3 * TB;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                const bool row_ok = i < nvalid;
                float r = 0.f;
                if (CAUSAL) {
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x30B);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int q = 0; q < kC / 32; ++q) {  // P = [j <= i](1 + T), r_i = sum_j P_ij (fp32)
                        uint32_t t0[16], t1[16], pk[16];
                        tmem_ld16(R0 + lo + 32 * q, t0);
                        tmem_ld16(R0 + lo + 32 * q + 16, t1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j2 = 0; j2 < 16; ++j2) {
                            const int j = 32 * q + 2 * j2;
                            const uint32_t a0 = j2 < 8 ? t0[2 * j2] : t1[2 * j2 - 16];
                            const uint32_t a1 = j2 < 8 ? t0[2 * j2 + 1] : t1[2 * j2 - 15];
                            const float p0 = j <= i ? 1.f + __uint_as_float(a0) : 0.f;
                            const float p1 = j + 1 <= i ? 1.f + __uint_as_float(a1) : 0.f;
                            pk[j2] = pack_bf16(p0, p1);
                            r += p0 + p1;
                        }
                        tmem_st16(R0 + lo + 16 * q, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP);
                }
                // q_i . z with z before the chunk
                float qz = 0.f;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        const uint4 v = *(const uint4 *)(qt + nb * kBox + sw128_off(i, g8));
                        const float *zz = zc + nb * 64 + g8 * 8;
                        qz += bf16lo(v.x) * zz[0] + bf16hi(v.x) * zz[1] + bf16lo(v.y) * zz[2] + bf16hi(v.y) * zz[3] +
                              bf16lo(v.z) * zz[4] + bf16hi(v.z) * zz[5] + bf16lo(v.w) * zz[6] + bf16hi(v.w) * zz[7];
                    }
                }
                float2 zn = make_float2(0.f, 0.f);  // z (t < 64) or a (t >= 64) after this chunk
                if (CAUSAL) {
                    const float2 cs = weighted_colsum(t < 64 ? kt : vt, col, nullptr);
                    const float *base = t < 64 ? zc : ac;
                    zn = make_float2(base[col] + cs.x, base[col + 1] + cs.y);
                }
                // O_i, g_i, delta_i; dO row -> dOt row in place
                ok = wait_or_abort(barO, ph, abort_flag, P.status, 0x30C);
                if (!ok) break;
                tc_fence_after();
                const float gi = (CAUSAL ? (float)row0 : (float)P.N) + qz + r;
                const float ig = 1.f / gi;
                float delta = 0.f;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t v[16];
                    tmem_ld16(R1 + lo + c16 * 16, v);
                    tmem_ld_wait();
                    unsigned char *tile = ot + (c16 / 4) * kBox;
                    const int col8 = (c16 % 4) * 2;
#pragma unroll
                    for (int g2 = 0; g2 < 2; ++g2) {
                        uint4 *p4 = (uint4 *)(tile + sw128_off(i, col8 + g2));
                        uint4 w = *p4;
                        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int e = c16 * 16 + g2 * 8 + 2 * q;
                            const float o0 = (__uint_as_float(v[g2 * 8 + 2 * q]) + ac[e]) * ig;
                            const float o1 = (__uint_as_float(v[g2 * 8 + 2 * q + 1]) + ac[e + 1]) * ig;
                            const float d0 = bf16lo(wv[q]), d1 = bf16hi(wv[q]);
                            delta = fmaf(d0, o0, fmaf(d1, o1, delta));
                            wv[q] = pack_bf16(d0 * ig, d1 * ig);
                        }
                        *p4 = w;
                    }
                }
                const float dt = delta * ig;
                sDt[i] = dt;
                if (row_ok) {
                    P.rs_g[(size_t)pc.h * P.N + row0 + i] = gi;
                    P.rs_dt[(size_t)pc.h * P.N + row0 + i] = dt;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barDt);
                if (CAUSAL) {  // U = [j <= i](W - dt), bf16, in place of W
                    ok = wait_or_abort(barW, ph, abort_flag, P.status, 0x30D);
                    if (!ok) break;
                    tc_fence_after();
                    tmem_to_bf16_inplace(R0 + lo, [&](int j, float w) { return j <= i ? w - dt : 0.f; });
                    tc_fence_before();
                    mbar_arrive(barU);
                }
                epi_sync();  // every row's dt and dOt are in shared memory
                {
                    const float2 cs = weighted_colsum(t < 64 ? qt : ot, col, t < 64 ? sDt : nullptr);
                    ye.x += cs.x;
                    ye.y += cs.y;
                }
                // dQ_i = X_i - dt_i z, staged in the Q tile (every MMA and column sum that reads Q is done
                // once X is complete and all threads are past this barrier) and stored by TMA
                ok = wait_or_abort(barX, ph, abort_flag, P.status, 0x30E);
                if (!ok) break;
                tc_fence_after();
                epi_sync();
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t v[16];
                    tmem_ld16(R1 + lo + c16 * 16, v);
                    tmem_wait_ld(v);
                    stage16_bf16(qt, i, c16, v, zc + c16 * 16, -dt);
                }
                (void)row_ok;
                (void)dQg;
                fence_proxy_async_smem();
                tc_fence_before();
                epi_sync();
                if (threadIdx.x == 64) {
                    for (int nb = 0; nb < NB; ++nb) tma_store_3d(&P.tmdQ, qt + nb * kBox, nb * 64, (int)row0, (int)pc.h);
                    bulk_commit();
                    bulk_wait_read0();
                    mbar_arrive(&empty[s]);
                }
                if (!CAUSAL) mbar_arrive(barXf);
                if (CAUSAL) {
                    ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x30F);
                    if (!ok) break;
                    tc_fence_after();
                    if (c + 1 < pc.e) {
                        tmem_row_to_tile(R2 + lo, Sb, i);
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(barSb);
                    }
                    epi_sync();  // everyone is done with z and a of this chunk
                    float *base = t < 64 ? zc : ac;
                    base[col] = zn.x;
                    base[col + 1] = zn.y;
                    epi_sync();
                }
            }
            if (!ok) break;
            // the piece's reverse sums -> workspace
            if (!wait_or_abort(barPP, pno & 1, abort_flag, P.status, 0x310)) break;
            tc_fence_after();
            float *slot = P.slots_rev + slot_of(pc.h, blockIdx.x) * P.slot_stride;
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                uint32_t v[16];
                tmem_ld16(R3 + lo + c16 * 16, v);
                tmem_ld_wait();
                float4 *dst = (float4 *)(slot + (size_t)i * D + c16 * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                         __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            slot[(size_t)D * D + (t < 64 ? 0 : D) + col] = ye.x;
            slot[(size_t)D * D + (t < 64 ? 0 : D) + col + 1] = ye.y;
            tc_fence_before();
            mbar_arrive(barPPf);
        }
    }
    if (threadIdx.x == 64) bulk_wait0();  // output stores complete before the CTA exits
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template __global__ void tc_bwd_dq_kernel<true>(const __grid_constant__ TcParams P);
template __global__ void tc_bwd_dq_kernel<false>(const __grid_constant__ TcParams P);

// ----------------------------------------------------------------------------------------------------
// dK / dV walk (reverse chunk order), with lane = key row j of the chunk.  Per chunk, causal:
//   T^T = K Q^T, W^T = V dO^T -> P^T = [i >= j](1 + T^T) / g_i and U^T = [i >= j](W^T / g_i - dt_i)
//   dK = U^T Q + V Pb^T  (then - y)        dV = P^T dO + K Pb  (then + e)
//   dO tile <- dOt in place ; P += Q^T dOt (for the earlier chunks) ; y, e += this chunk's rows
// Pb is the bf16 copy of P (the sum over later rows).  Non-causal: dK = V Pb^T - y, dV = K Pb + e with
// the head's totals; stages hold only K and V.
// TMEM: R0 T^T/P^T, R1 W^T/U^T, R2 dK then dV, R3 P.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL>
__global__ void __launch_bounds__(192, 1) tc_bwd_dkdv_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr int NST = CAUSAL ? 1 : 3;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = CAUSAL ? 4 * TB : 2 * TB;  // causal: Q, dO, K, V; non-causal: K, V
    constexpr uint32_t OFF_K = CAUSAL ? 2 * TB : 0, OFF_V = CAUSAL ? 3 * TB : TB;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Pb = sm + NST * STAGE;
    float *yc = (float *)(Pb + TB);
    float *ec = yc + D;
    float *sIg = ec + D;
    float *sDt = sIg + kC;
    uint64_t *full = (uint64_t *)(sDt + kC);
    uint64_t *empty = full + NST;
    uint64_t *bar = empty + NST;
    uint64_t *barT = bar, *barP = bar + 1, *barPb = bar + 2, *barK = bar + 3, *barKf = bar + 4, *barV = bar + 5,
             *barDt = bar + 6, *barS = bar + 7, *barVf = bar + 8;
    uint32_t *tslot = (uint32_t *)(bar + 9);
    volatile int *abort_flag = (volatile int *)(tslot + 1);
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // MMA commit + the epilogue once its dK, dV tiles have left shared memory
        }
        const uint32_t counts[9] = {1, 128, 128, 1, 128, 1, 128, 1, 128};
        for (int k = 0; k < 9; ++k) mbar_init(&bar[k], counts[k]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t R0 = tmem, R1 = tmem + 128, R2 = tmem + 256, R3 = tmem + 384;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer (chunks of each piece in reverse order)
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        if (CAUSAL) {
            prefetch_tmap(&P.tmQ);
            prefetch_tmap(&P.tmdO);
        }
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x401)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tma_load_3d(st + OFF_K + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, (int)pc.h);
                    tma_load_3d(st + OFF_V + nb * kBox, &P.tmV, &full[s], nb * 64, c * kC, (int)pc.h);
                    if (CAUSAL) {
                        tma_load_3d(st + nb * kBox, &P.tmQ, &full[s], nb * 64, c * kC, (int)pc.h);
                        tma_load_3d(st + TB + nb * kBox, &P.tmdO, &full[s], nb * 64, c * kC, (int)pc.h);
                    }
                }
            }
        }
        if (!ok) {
            for (int k = it > NST ? it - NST : 0; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKK = idesc_bf16(128, 128, false, false);
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t pb = smem_u32(Pb);
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!CAUSAL && !wait_or_abort(barPb, pno & 1, abort_flag, P.status, 0x402)) break;
            for (int c = pc.e - 1; c >= pc.a && ok; --c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x403);
                if (!ok) break;
                tc_fence_after();
                const uint32_t base = smem_u32(stages + s * STAGE);
                const uint32_t qb = base, ob = base + TB, kb = base + OFF_K, vb = base + OFF_V;
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {  // T^T = K Q^T ; W^T = V dO^T
                        const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                        mma_ss(R0, sdesc_sw128(kb + o, 16, 1024), sdesc_sw128(qb + o, 16, 1024), idKK, k > 0);
                        mma_ss(R1, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(ob + o, 16, 1024), idKK, k > 0);
                    }
                    mma_commit(barT);
                    ok = wait_or_abort(barP, ph, abort_flag, P.status, 0x404);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // dK = U^T Q
                        mma_ts(R2, R1 + 8 * k, sdesc_sw128(qb + 2048 * k, kBox, 1024), idKM, k > 0);
                    ok = wait_or_abort(barPb, ph, abort_flag, P.status, 0x405);
                    if (!ok) break;
                    tc_fence_after();
                } else if (it > 0) {
                    ok = wait_or_abort(barVf, (it - 1) & 1, abort_flag, P.status, 0x406);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dK += V Pb^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R2, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(pb + o, 16, 1024), idKK,
                           (CAUSAL || k > 0) ? 1u : 0u);
                }
                mma_commit(barK);
                ok = wait_or_abort(barKf, ph, abort_flag, P.status, 0x407);
                if (!ok) break;
                tc_fence_after();
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // dV = (P/g)^T dO
                        mma_ts(R2, R0 + 8 * k, sdesc_sw128(ob + 2048 * k, kBox, 1024), idKM, k > 0);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)  // dV += K Pb
                    mma_ss(R2, sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(pb + 2048 * k, kBox, 1024), idKM, (CAUSAL || k > 0) ? 1u : 0u);
                mma_commit(barV);
                if (CAUSAL) {
                    ok = wait_or_abort(barDt, ph, abort_flag, P.status, 0x408);  // dOt is in place of dO
                    if (!ok) break;
                    tc_fence_after();
                    if (c > pc.a) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)  // P += Q^T dOt
                            mma_ss(R3, sdesc_sw128(qb + 2048 * k, kBox, 1024), sdesc_sw128(ob + 2048 * k, kBox, 1024),
                                   idMM, 1u);
                    }
                    mma_commit(barS);
                }
                mma_commit(&empty[s]);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue warps: thread <-> key row j (TMEM lane) and state row d (same index)
        const int lb = 32 * (warp & 3);
        const int j = lb + lane;
        const int t = threadIdx.x - 64;
        const int col = 2 * (t & 63);
        const uint32_t lo = (uint32_t)lb << 16;
        __nv_bfloat16 *dKg = (__nv_bfloat16 *)P.dK, *dVg = (__nv_bfloat16 *)P.dV;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // carried reverse sums (causal: the later pieces of the head; non-causal: the whole head),
            // combined into this piece's own slot by tc_scan_slots
            if (CAUSAL && it > 0) {
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x409)) break;
                tc_fence_after();
            }
            load_carry1(P.slots_rev + slot_of(pc.h, blockIdx.x) * P.slot_stride, j, R3 + lo, Pb, yc, ec, CAUSAL);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync();
            mbar_arrive(barPb);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                unsigned char *qt = st, *ot = st + TB;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                const bool row_ok = j < nvalid;
                const size_t grow = (size_t)pc.h * P.N + row0 + j;
                if (CAUSAL) {
                    sIg[j] = row_ok ? 1.f / P.rs_g[grow] : 0.f;
                    sDt[j] = row_ok ? P.rs_dt[grow] : 0.f;
                    epi_sync();
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x40A);
                    if (!ok) break;
                    tc_fence_after();
                    // columns are query rows i of the chunk: keep i >= j
                    tmem_to_bf16_inplace(R0 + lo, [&](int i, float x) { return i >= j ? (1.f + x) * sIg[i] : 0.f; });
                    tmem_to_bf16_inplace(R1 + lo, [&](int i, float x) { return i >= j ? x * sIg[i] - sDt[i] : 0.f; });
                    tc_fence_before();
                    mbar_arrive(barP);
                }
                // dK_j = [dK accumulator]_j - y
                ok = wait_or_abort(barK, ph, abort_flag, P.status, 0x40B);
                if (!ok) break;
                tc_fence_after();
                // dK staged in the V tile (its last reader, dK += V Pb^T, is complete) and stored by TMA
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t v[16];
                    tmem_ld16(R2 + lo + c16 * 16, v);
                    tmem_wait_ld(v);
                    stage16_bf16(st + OFF_V, j, c16, v, yc + c16 * 16, -1.f);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barKf);
                epi_sync();
                if (threadIdx.x == 64) {
                    for (int nb = 0; nb < NB; ++nb)
                        tma_store_3d(&P.tmdK, st + OFF_V + nb * kBox, nb * 64, (int)row0, (int)pc.h);
                    bulk_commit();
                }
                // dV_j = [dV accumulator]_j + e
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x40C);
                if (!ok) break;
                tc_fence_after();
                // dV staged in the K tile (its last reader, dV += K Pb, is complete) and stored by TMA
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t v[16];
                    tmem_ld16(R2 + lo + c16 * 16, v);
                    tmem_wait_ld(v);
                    stage16_bf16(st + OFF_K, j, c16, v, ec + c16 * 16, 1.f);
                }
                (void)row_ok;
                (void)dKg;
                (void)dVg;
                fence_proxy_async_smem();
                tc_fence_before();
                epi_sync();
                if (threadIdx.x == 64) {
                    for (int nb = 0; nb < NB; ++nb)
                        tma_store_3d(&P.tmdV, st + OFF_K + nb * kBox, nb * 64, (int)row0, (int)pc.h);
                    bulk_commit();
                }
                if (!CAUSAL) {
                    mbar_arrive(barVf);
                    if (threadIdx.x == 64) {
                        bulk_wait_read0();
                        mbar_arrive(&empty[s]);
                    }
                    continue;
                }
                // dO row -> dOt row in place; then y and e gain this chunk's rows
                {
                    const float igj = sIg[j];
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                        for (int g8 = 0; g8 < 8; ++g8) {
                            uint4 *p4 = (uint4 *)(ot + nb * kBox + sw128_off(j, g8));
                            uint4 w = *p4;
                            uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                            for (int q = 0; q < 4; ++q) wv[q] = pack_bf16(bf16lo(wv[q]) * igj, bf16hi(wv[q]) * igj);
                            *p4 = w;
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barDt);
                epi_sync();  // every row of dOt is in shared memory
                const float2 cs = weighted_colsum(t < 64 ? qt : ot, col, t < 64 ? sDt : nullptr);
                float *base = t < 64 ? yc : ec;
                const float2 yn = make_float2(base[col] + cs.x, base[col + 1] + cs.y);
                epi_sync();  // every read of the stage by this warp group is done
                if (threadIdx.x == 64) {
                    bulk_wait_read0();  // dK and dV have left the V and K tiles
                    mbar_arrive(&empty[s]);
                }
                ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x40D);
                if (!ok) break;
                tc_fence_after();
                if (c > pc.a) {
                    tmem_row_to_tile(R3 + lo, Pb, j);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(barPb);
                }
                epi_sync();  // everyone is done with y and e of this chunk
                base[col] = yn.x;
                base[col + 1] = yn.y;
                epi_sync();
            }
        }
    }
    if (threadIdx.x == 64) bulk_wait0();  // output stores complete before the CTA exits
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template __global__ void tc_bwd_dkdv_kernel<true>(const __grid_constant__ TcParams P);
template __global__ void tc_bwd_dkdv_kernel<false>(const __grid_constant__ TcParams P);

}  // namespace tc

// ======================================================================================== host ===

namespace {

constexpr size_t kTB = 2 * (size_t)tc::kBox;
constexpr size_t kSmemDq = 4 * kTB + kTB + 3 * 512 + 512;          // causal: 1 stage of Q, dO, K, V
constexpr size_t kSmemDqNc = 2 * 2 * kTB + kTB + 3 * 512 + 512;    // 2 stages of Q, dO
constexpr size_t kSmemDkdv = 4 * kTB + kTB + 4 * 512 + 512;        // 1 stage of Q, dO, K, V
constexpr size_t kSmemDkdvNc = 3 * 2 * kTB + kTB + 4 * 512 + 512;  // 3 stages of K, V
static_assert(kSmemDkdvNc <= 232448, "dK/dV kernel exceeds the shared-memory limit");

bool set_bwd_attrs() {
    static int done = 0;
    if (done) return done > 0;
    const int A = cudaFuncAttributeMaxDynamicSharedMemorySize;
    bool ok = cudaFuncSetAttribute(tc::tc_bwd_dq_kernel<true>, (cudaFuncAttribute)A, (int)kSmemDq) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dq_kernel<false>, (cudaFuncAttribute)A, (int)kSmemDqNc) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel<true>, (cudaFuncAttribute)A, (int)kSmemDkdv) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel<false>, (cudaFuncAttribute)A, (int)kSmemDkdvNc) ==
                  cudaSuccess;
    done = ok ? 1 : -1;
    return ok;
}

}  // namespace

cudaError_t tc_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *dO, void *dQ,
                        void *dK, void *dV, unsigned char *ws, cudaStream_t s) {
    if (!set_bwd_attrs()) return cudaErrorInvalidValue;
    tc::TcParams P;
    memset(&P, 0, sizeof(P));
    if (!tc_host::fill_common(P, p, ws)) return cudaErrorInvalidDevice;
    if (!tc_host::make_map(&P.tmQ, Q, p) || !tc_host::make_map(&P.tmK, K, p) || !tc_host::make_map(&P.tmV, V, p) ||
        !tc_host::make_map(&P.tmdO, dO, p) || !tc_host::make_map(&P.tmdQ, dQ, p) ||
        !tc_host::make_map(&P.tmdK, dK, p) || !tc_host::make_map(&P.tmdV, dV, p))
        return cudaErrorInvalidValue;
    P.slots_rev = (float *)(ws + p.off_states2);
    P.rs_g = (float *)(ws + p.off_rowstats);
    P.rs_dt = P.rs_g + (size_t)p.BH * p.N;
    P.dQ = dQ;
    P.dK = dK;
    P.dV = dV;
    cudaError_t e = tc_host::launch_agg(P, s);
    if (e == cudaSuccess) e = tc_host::launch_scan(P.slots, P, p.BH, p.causal ? 0 : 2, s);
    if (e != cudaSuccess) return e;
    if (p.causal)
        tc::tc_bwd_dq_kernel<true><<<P.sl.G, 192, kSmemDq, s>>>(P);
    else
        tc::tc_bwd_dq_kernel<false><<<P.sl.G, 192, kSmemDqNc, s>>>(P);
    e = tc_host::launch_scan(P.slots_rev, P, p.BH, p.causal ? 1 : 2, s);
    if (e != cudaSuccess) return e;
    if (p.causal)
        tc::tc_bwd_dkdv_kernel<true><<<P.sl.G, 192, kSmemDkdv, s>>>(P);
    else
        tc::tc_bwd_dkdv_kernel<false><<<P.sl.G, 192, kSmemDkdvNc, s>>>(P);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(5);
    return e;
}

}  // namespace la
