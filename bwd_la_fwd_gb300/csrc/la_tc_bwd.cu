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
// Launches: the per-piece K^T V sums and their scan (shared with the forward), the dQ walk in chunk
// order (it recomputes O_i, hence g_i and delta_i; the stored O is not read; it also writes each piece's
// reverse sums P, y, e and the per-row g_i, dt_i), the scan of the reverse sums, and the dK / dV walk in
// reverse chunk order.  Each kernel: warp 0 TMA, warp 1 TMEM + MMA issue, warps 2-9 epilogue (two warps
// per TMEM lane quarter, each owning 64 of the 128 columns).
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

// Reads this half's 64 columns (lane = the thread's row) of a 128-column fp32 TMEM block and maps them
// through f(column, value) to 32 packed bf16 pairs.  The caller writes them back (tmem_st32 at column
// 32 hf) after a barrier, because the two halves' reads and writes overlap.
template <typename F>
__device__ __forceinline__ void tmem_half_to_bf16(uint32_t taddr, int hf, F f, uint32_t (&pk)[32]) {
    uint32_t t0[32], t1[32];
    tmem_ld32(taddr + 64 * hf, t0);
    tmem_ld32(taddr + 64 * hf + 32, t1);
    tmem_wait_ld(t0);
    tmem_wait_ld(t1);
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        const int c = 64 * hf + 2 * m;
        const uint32_t a0 = m < 16 ? t0[2 * m] : t1[2 * m - 32];
        const uint32_t a1 = m < 16 ? t0[2 * m + 1] : t1[2 * m - 31];
        pk[m] = pack_bf16(f(c, __uint_as_float(a0)), f(c + 1, __uint_as_float(a1)));
    }
}

// Sum over rows [64 rh, 64 rh + 64) of w[r] * X[r][2 cp .. 2 cp + 1] for a bf16 tile X (two 64-column
// boxes, 128-byte swizzle); w == nullptr means weights of one.
__device__ __forceinline__ float2 colsum_half(const unsigned char *tile2, int cp, int rh, const float *w) {
    const int col = 2 * cp;
    const unsigned char *tile = tile2 + (col / 64) * kBox;
    const int cc = col % 64;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
    for (int r = 64 * rh; r < 64 * rh + 64; ++r) {
        const uint32_t v = *(const uint32_t *)(tile + sw128_off(r, cc / 8) + (cc % 8) * 2);
        const float wr = w ? w[r] : 1.f;
        s0 = fmaf(wr, bf16lo(v), s0);
        s1 = fmaf(wr, bf16hi(v), s1);
    }
    return make_float2(s0, s1);
}

// Reads this half's 64 columns of an fp32 TMEM block, adds add_scale * add[c] (c = column), rounds to
// bf16 and writes them into row `row`, box hf of a two-box 128B-swizzled tile (the layout of the output
// TMA maps).
__device__ __forceinline__ void tmem_half_to_out(uint32_t taddr, int hf, const float *add, float add_scale,
                                                 unsigned char *tile2, int row) {
    unsigned char *tile = tile2 + hf * kBox;
#pragma unroll 1
    for (int half32 = 0; half32 < 2; ++half32) {
        uint32_t v[32];
        tmem_ld32(taddr + 64 * hf + 32 * half32, v);
        tmem_wait_ld(v);
        const float *aa = add + 64 * hf + 32 * half32;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            uint4 w;
            uint32_t *wv = (uint32_t *)&w;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int m = 8 * g4 + 2 * q;
                wv[q] = pack_bf16(__uint_as_float(v[m]) + add_scale * aa[m],
                                  __uint_as_float(v[m + 1]) + add_scale * aa[m + 1]);
            }
            *(uint4 *)(tile + sw128_off(row, 4 * half32 + g4)) = w;
        }
    }
}

// Issues the TMA stores of a two-box output tile from shared memory and commits them.  One thread.
__device__ __forceinline__ void store_tile(const CUtensorMap *map, const unsigned char *tile2, int row0, int h) {
    tma_store_3d(map, tile2, 0, row0, h);
    tma_store_3d(map, tile2 + kBox, 64, row0, h);
    bulk_commit();
}

// ----------------------------------------------------------------------------------------------------
// dQ walk (chunk order).  The forward output is not recomputed: with W' = dO V^T and Y = dO Sb^T (Sb =
// bf16 state before the chunk),
//   delta_i g_i = dO_i . a + sum_j P_ij W'_ij + q_i . Y_i,      P_ij = [j <= i](1 + q_i . k_j)
//   dQ_i = (Y_i + [U' K]_i) / g_i - dt_i z,                     U'_ij = [j <= i](W'_ij - delta_i)
// Per chunk, causal: T = Q K^T and W' (R0, R1); S += K^T V (R2); the epilogue forms P, r_i and
// sum_j P_ij W'_ij from T and W' in registers; Y into R0; the epilogue forms g_i, delta_i, dt_i and U'
// (bf16, in place of W'); X = Y + U' K in R0; dO -> dO / g in place; Ppiece += Q^T (dO / g) (R3).
// Non-causal: only Y (R0, the head's totals) and Ppiece; stages hold only Q and dO.
// Epilogue thread u = threadIdx.x - 64: row i = 32 (warp % 4) + lane, column half hf = u / 128; for the
// column sums it owns column pair cp = u % 64 of tensor u / 128 over row half (u / 64) % 2.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dq_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr int NST = CAUSAL ? 1 : 2;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = CAUSAL ? 4 * TB : 2 * TB;  // Q, dO (, K, V)
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Sb = sm + NST * STAGE;
    float *zc = (float *)(Sb + TB);  // z before the chunk (fp32, D)
    float *ac = zc + D;              // a before the chunk
    float *sDt = ac + D;             // dt_i of the chunk's rows
    float *xg = sDt + kC;            // [2][128] row partials of g (per column half)
    float *xd = xg + 2 * kC;         // [2][128] row partials of delta g
    float *cs = xd + 2 * kC;         // [2 tensors][2 row halves][128 columns] column-sum partials
    uint64_t *full = (uint64_t *)(cs + 4 * D);
    uint64_t *empty = full + NST;
    uint64_t *bar = empty + NST;
    uint64_t *barT = bar, *barTr = bar + 1, *barSb = bar + 2, *barY = bar + 3, *barDt = bar + 4, *barU = bar + 5,
             *barX = bar + 6, *barS = bar + 7, *barPP = bar + 8, *barPPf = bar + 9, *barXf = bar + 10;
    uint32_t *tslot = (uint32_t *)(bar + 11);
    volatile int *abort_flag = (volatile int *)(tslot + 1);
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // MMA commit + the epilogue once its dQ tile has left shared memory
        }
        const uint32_t E = kEpiThreads;
        const uint32_t counts[11] = {1, E, E, 1, E, E, 1, 1, 1, E, E};
        for (int k = 0; k < 11; ++k) mbar_init(&bar[k], counts[k]);
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
                    for (int k = 0; k < 8; ++k) {  // T = Q K^T ; W' = dO V^T
                        const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                        mma_ss(R0, sdesc_sw128(qb + o, 16, 1024), sdesc_sw128(kb + o, 16, 1024), idKK, k > 0);
                        mma_ss(R1, sdesc_sw128(ob + o, 16, 1024), sdesc_sw128(vb + o, 16, 1024), idKK, k > 0);
                    }
                    mma_commit(barT);
                    ok = wait_or_abort(barTr, ph, abort_flag, P.status, 0x305);  // T has been read out of R0
                    if (!ok) break;
                    ok = wait_or_abort(barSb, ph, abort_flag, P.status, 0x306);
                    if (!ok) break;
                    tc_fence_after();
                } else if (it > 0) {
                    ok = wait_or_abort(barXf, (it - 1) & 1, abort_flag, P.status, 0x307);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)  // Y = dO Sb^T
                    mma_ss(R0, sdesc_sw128(ob + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                mma_commit(barY);
                if (CAUSAL) {
                    if (c + 1 < pc.e) {  // S += K^T V, once the epilogue has copied S into Sb (barSb above)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mma_ss(R2, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024),
                                   idMM, 1u);
                    }
                    ok = wait_or_abort(barU, ph, abort_flag, P.status, 0x308);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // X = Y + U' K
                        mma_ts(R0, R1 + 8 * k, sdesc_sw128(kb + 2048 * k, kBox, 1024), idKM, 1u);
                }
                ok = wait_or_abort(barDt, ph, abort_flag, P.status, 0x309);  // dO / g is in place of dO
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // Ppiece += Q^T (dO / g)
                    mma_ss(R3, sdesc_sw128(qb + 2048 * k, kBox, 1024), sdesc_sw128(ob + 2048 * k, kBox, 1024), idMM,
                           (c > pc.a || k > 0) ? 1u : 0u);
                mma_commit(barX);
                mma_commit(barS);
                mma_commit(&empty[s]);
                if (c + 1 == pc.e) mma_commit(barPP);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const int which = u >> 7, cp = u & 63, rh = (u >> 6) & 1;  // column-sum role
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            // carried forward state of the piece, combined into its own slot by tc_scan_slots
            if (CAUSAL && it > 0) {
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x30A)) break;
                tc_fence_after();
            }
            load_carry_half(P.slots + slot_of(pc.h, blockIdx.x) * P.slot_stride, i, hf, R2 + lo, 0u, 0u, Sb, zc,
                            ac, CAUSAL, /*vec_to_tmem=*/false);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barSb);
            float2 ye = make_float2(0.f, 0.f);  // this thread's part of y (which 0) or e (which 1)
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                unsigned char *qt = st, *ot = st + TB, *kt = st + 2 * TB, *vt = st + 3 * TB;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                float gpart = 0.f, dpart = 0.f;  // partial g_i and partial delta_i g_i over this half
                if (CAUSAL) {  // P, r_i and sum_j P_ij W'_ij over this half's columns j (fp32)
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x30B);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t t0[32], w0[32];
#pragma unroll 1
                    for (int half32 = 0; half32 < 2; ++half32) {
                        tmem_ld32(R0 + lo + 64 * hf + 32 * half32, t0);
                        tmem_ld32(R1 + lo + 64 * hf + 32 * half32, w0);
                        tmem_wait_ld(t0);
                        tmem_wait_ld(w0);
#pragma unroll
                        for (int m = 0; m < 32; ++m) {
                            const int j = 64 * hf + 32 * half32 + m;
                            const float pij = j <= i ? 1.f + __uint_as_float(t0[m]) : 0.f;
                            gpart += pij;
                            dpart = fmaf(pij, __uint_as_float(w0[m]), dpart);
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(barTr);
                }
                gpart += dot_half(qt, i, hf, zc);  // q_i . z, z before the chunk
                dpart += dot_half(ot, i, hf, ac);  // dO_i . a, a before the chunk
                xg[hf * kC + i] = gpart;
                float2 zn = make_float2(0.f, 0.f);
                if (CAUSAL) {  // column sums of K (which 0) and V (which 1) over this thread's row half
                    const float2 v = colsum_half(which == 0 ? kt : vt, cp, rh, nullptr);
                    cs[(which * 2 + rh) * D + 2 * cp] = v.x;
                    cs[(which * 2 + rh) * D + 2 * cp + 1] = v.y;
                }
                epi_sync256();
                const float gi = (CAUSAL ? (float)row0 : (float)P.N) + xg[i] + xg[kC + i];
                const float ig = 1.f / gi;
                if (CAUSAL && rh == 0) {
                    const float *base = which == 0 ? zc : ac;
                    const float *c0 = cs + (which * 2) * D, *c1 = c0 + D;
                    zn = make_float2(base[2 * cp] + c0[2 * cp] + c1[2 * cp], base[2 * cp + 1] + c0[2 * cp + 1] + c1[2 * cp + 1]);
                }
                // q_i . Y_i over this half's d (Y = dO Sb^T)
                ok = wait_or_abort(barY, ph, abort_flag, P.status, 0x30C);
                if (!ok) break;
                tc_fence_after();
                uint32_t y0[32], y1[32];
                tmem_ld32(R0 + lo + 64 * hf, y0);
                tmem_ld32(R0 + lo + 64 * hf + 32, y1);
                tmem_wait_ld(y0);
                tmem_wait_ld(y1);
                {
                    const unsigned char *tile = qt + hf * kBox;
                    float acc = 0.f;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        const uint4 v = *(const uint4 *)(tile + sw128_off(i, g8));
                        const uint32_t *yy = g8 < 4 ? y0 + 8 * g8 : y1 + 8 * (g8 - 4);
                        acc = fmaf(bf16lo(v.x), __uint_as_float(yy[0]), acc);
                        acc = fmaf(bf16hi(v.x), __uint_as_float(yy[1]), acc);
                        acc = fmaf(bf16lo(v.y), __uint_as_float(yy[2]), acc);
                        acc = fmaf(bf16hi(v.y), __uint_as_float(yy[3]), acc);
                        acc = fmaf(bf16lo(v.z), __uint_as_float(yy[4]), acc);
                        acc = fmaf(bf16hi(v.z), __uint_as_float(yy[5]), acc);
                        acc = fmaf(bf16lo(v.w), __uint_as_float(yy[6]), acc);
                        acc = fmaf(bf16hi(v.w), __uint_as_float(yy[7]), acc);
                    }
                    dpart += acc;
                }
                xd[hf * kC + i] = dpart;
                tc_fence_before();
                epi_sync256();
                tc_fence_after();
                const float delta = (xd[i] + xd[kC + i]) * ig;
                const float dt = delta * ig;
                if (hf == 0) {
                    sDt[i] = dt;
                    if (i < nvalid) {
                        P.rs_g[(size_t)pc.h * P.N + row0 + i] = gi;
                        P.rs_dt[(size_t)pc.h * P.N + row0 + i] = dt;
                    }
                }
                if (CAUSAL) {  // U' = [j <= i](W' - delta), bf16, in place of W'
                    uint32_t pk[32];
                    tmem_half_to_bf16(R1 + lo, hf, [&](int j, float w) { return j <= i ? w - delta : 0.f; }, pk);
                    tc_fence_before();
                    epi_sync256();  // both halves have read W' before U' overwrites it
                    tc_fence_after();
                    tmem_st32(R1 + lo + 32 * hf, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barU);
                }
                {  // dO -> dO / g in place (W' and Y, its unscaled readers, are done)
                    unsigned char *tile = ot + hf * kBox;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        uint4 *p4 = (uint4 *)(tile + sw128_off(i, g8));
                        uint4 w = *p4;
                        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                        for (int q = 0; q < 4; ++q) wv[q] = pack_bf16(bf16lo(wv[q]) * ig, bf16hi(wv[q]) * ig);
                        *p4 = w;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barDt);
                epi_sync256();  // every row of dO / g and every dt_i is in shared memory
                {  // y += sum_i dt_i q_i (which 0), e += sum_i dO_i / g_i (which 1), over this thread's row half
                    const float2 v = colsum_half(which == 0 ? qt : ot, cp, rh, which == 0 ? sDt : nullptr);
                    ye.x += v.x;
                    ye.y += v.y;
                }
                // dQ_i = X_i / g_i - dt_i z (X = Y + U' K; non-causal X = Y), staged in a tile whose readers
                // are done (causal: V; non-causal: Q, once Ppiece is complete)
                ok = wait_or_abort(barX, ph, abort_flag, P.status, 0x30E);
                if (!ok) break;
                tc_fence_after();
                unsigned char *dqt = CAUSAL ? vt : qt;
                if (!CAUSAL) epi_sync256();  // every read of the Q tile (y sums) is done
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(R0 + lo + 64 * hf, v0);
                    tmem_ld32(R0 + lo + 64 * hf + 32, v1);
                    tmem_wait_ld(v0);
                    tmem_wait_ld(v1);
                    unsigned char *tile = dqt + hf * kBox;
                    const float *zz = zc + 64 * hf;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        const uint32_t *xx = g8 < 4 ? v0 + 8 * g8 : v1 + 8 * (g8 - 4);
                        uint4 w;
                        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int m = 8 * g8 + 2 * q;
                            wv[q] = pack_bf16(__uint_as_float(xx[2 * q]) * ig - dt * zz[m],
                                              __uint_as_float(xx[2 * q + 1]) * ig - dt * zz[m + 1]);
                        }
                        *(uint4 *)(tile + sw128_off(i, g8)) = w;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                if (!CAUSAL) mbar_arrive(barXf);
                epi_sync256();
                if (u == 0) {
                    store_tile(&P.tmdQ, dqt, (int)row0, (int)pc.h);
                    bulk_wait_read0();
                    mbar_arrive(&empty[s]);
                }
                if (CAUSAL) {
                    ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x30F);
                    if (!ok) break;
                    tc_fence_after();
                    if (c + 1 < pc.e) {
                        tmem_half_to_tile(R2 + lo, Sb, i, hf);
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(barSb);
                    }
                    // z (which 0) and a (which 1) after this chunk
                    if (rh == 0) {
                        float *base = which == 0 ? zc : ac;
                        base[2 * cp] = zn.x;
                        base[2 * cp + 1] = zn.y;
                    }
                    epi_sync256();
                }
            }
            if (!ok) break;
            // the piece's reverse sums -> workspace
            if (!wait_or_abort(barPP, pno & 1, abort_flag, P.status, 0x310)) break;
            tc_fence_after();
            float *slot = P.slots_rev + slot_of(pc.h, blockIdx.x) * P.slot_stride;
#pragma unroll 1
            for (int half32 = 0; half32 < 2; ++half32) {
                uint32_t v[32];
                tmem_ld32(R3 + lo + 64 * hf + 32 * half32, v);
                tmem_wait_ld(v);
                float4 *dst = (float4 *)(slot + (size_t)i * D + 64 * hf + 32 * half32);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                         __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            // y, e: add the two row halves
            cs[(which * 2 + rh) * D + 2 * cp] = ye.x;
            cs[(which * 2 + rh) * D + 2 * cp + 1] = ye.y;
            tc_fence_before();
            epi_sync256();
            if (rh == 0) {
                const float *c0 = cs + (which * 2) * D, *c1 = c0 + D;
                slot[(size_t)D * D + which * D + 2 * cp] = c0[2 * cp] + c1[2 * cp];
                slot[(size_t)D * D + which * D + 2 * cp + 1] = c0[2 * cp + 1] + c1[2 * cp + 1];
            }
            mbar_arrive(barPPf);
            epi_sync256();  // cs is reused by the next piece
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
// the head's totals; stages hold only K and V.  dK leaves through the V tile and dV through the K tile.
// TMEM: R0 T^T/P^T, R1 W^T/U^T, R2 dK then dV, R3 P.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dkdv_kernel(const __grid_constant__ TcParams P) {
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
    float *sIg = ec + D;                  // causal only: 1/g_i and dt_i of the chunk's rows
    float *sDt = sIg + (CAUSAL ? kC : 0);
    float *cs = sDt + (CAUSAL ? kC : 0);  // causal only: [2][2][128] column-sum partials
    uint64_t *full = (uint64_t *)(cs + (CAUSAL ? 4 * D : 0));
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
        const uint32_t E = kEpiThreads;
        const uint32_t counts[9] = {1, E, E, 1, E, 1, E, 1, E};
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
        // ---- epilogue: thread <-> key row j (TMEM lane) and column half hf
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int j = 32 * q4 + lane;
        const int which = u >> 7, cp = u & 63, rh = (u >> 6) & 1;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // carried reverse sums (causal: later pieces of the head; non-causal: the whole head), combined
            // into this piece's own slot by tc_scan_slots
            if (CAUSAL && it > 0) {
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x409)) break;
                tc_fence_after();
            }
            load_carry_half(P.slots_rev + slot_of(pc.h, blockIdx.x) * P.slot_stride, j, hf, R3 + lo, 0u, 0u, Pb, yc,
                            ec, CAUSAL, /*vec_to_tmem=*/false);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barPb);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                unsigned char *qt = st, *ot = st + TB;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                if (CAUSAL) {
                    if (hf == 0) {
                        const bool ok_row = j < nvalid;
                        const size_t grow = (size_t)pc.h * P.N + row0 + j;
                        sIg[j] = ok_row ? 1.f / P.rs_g[grow] : 0.f;
                        sDt[j] = ok_row ? P.rs_dt[grow] : 0.f;
                    }
                    epi_sync256();
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x40A);
                    if (!ok) break;
                    tc_fence_after();
                    // columns are query rows i of the chunk: keep i >= j
                    uint32_t pk0[32], pk1[32];
                    tmem_half_to_bf16(R0 + lo, hf, [&](int i, float x) { return i >= j ? (1.f + x) * sIg[i] : 0.f; }, pk0);
                    tmem_half_to_bf16(R1 + lo, hf, [&](int i, float x) { return i >= j ? x * sIg[i] - sDt[i] : 0.f; }, pk1);
                    tc_fence_before();
                    epi_sync256();
                    tc_fence_after();
                    tmem_st32(R0 + lo + 32 * hf, pk0);
                    tmem_st32(R1 + lo + 32 * hf, pk1);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP);
                }
                // dK_j = [accumulator]_j - y, staged in the V tile (its last reader, dK += V Pb^T, is done)
                ok = wait_or_abort(barK, ph, abort_flag, P.status, 0x40B);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R2 + lo, hf, yc, -1.f, st + OFF_V, j);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barKf);
                epi_sync256();
                if (u == 0) store_tile(&P.tmdK, st + OFF_V, (int)row0, (int)pc.h);
                // dV_j = [accumulator]_j + e, staged in the K tile (its last reader, dV += K Pb, is done)
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x40C);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R2 + lo, hf, ec, 1.f, st + OFF_K, j);
                fence_proxy_async_smem();
                tc_fence_before();
                if (!CAUSAL) mbar_arrive(barVf);
                epi_sync256();
                if (u == 0) store_tile(&P.tmdV, st + OFF_K, (int)row0, (int)pc.h);
                if (!CAUSAL) {
                    if (u == 0) {
                        bulk_wait_read0();
                        mbar_arrive(&empty[s]);
                    }
                    continue;
                }
                // dO row -> dOt row in place, for P += Q^T dOt and the e sums
                {
                    const float igj = sIg[j];
                    unsigned char *tile = ot + hf * kBox;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        uint4 *p4 = (uint4 *)(tile + sw128_off(j, g8));
                        uint4 w = *p4;
                        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
                        for (int q = 0; q < 4; ++q) wv[q] = pack_bf16(bf16lo(wv[q]) * igj, bf16hi(wv[q]) * igj);
                        *p4 = w;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barDt);
                epi_sync256();  // every row of dOt is in shared memory
                {  // this chunk's rows: y += sum dt_i q_i (which 0), e += sum dOt_i (which 1)
                    const float2 v = colsum_half(which == 0 ? qt : ot, cp, rh, which == 0 ? sDt : nullptr);
                    cs[(which * 2 + rh) * D + 2 * cp] = v.x;
                    cs[(which * 2 + rh) * D + 2 * cp + 1] = v.y;
                }
                epi_sync256();
                float2 yn = make_float2(0.f, 0.f);
                if (rh == 0) {
                    const float *base = which == 0 ? yc : ec;
                    const float *c0 = cs + (which * 2) * D, *c1 = c0 + D;
                    yn = make_float2(base[2 * cp] + c0[2 * cp] + c1[2 * cp], base[2 * cp + 1] + c0[2 * cp + 1] + c1[2 * cp + 1]);
                }
                if (u == 0) {
                    bulk_wait_read0();  // dK and dV have left the V and K tiles
                    mbar_arrive(&empty[s]);
                }
                ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x40D);
                if (!ok) break;
                tc_fence_after();
                if (c > pc.a) {
                    tmem_half_to_tile(R3 + lo, Pb, j, hf);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(barPb);
                }
                if (rh == 0) {
                    float *base = which == 0 ? yc : ec;
                    base[2 * cp] = yn.x;
                    base[2 * cp + 1] = yn.y;
                }
                epi_sync256();
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
constexpr size_t kEpiSmemDq = 2 * 128 * 4 + 128 * 4 + 4 * 128 * 4 + 4 * 128 * 4;  // z, a, dt, 2 x-arrays, cs
constexpr size_t kSmemDq = 4 * kTB + kTB + kEpiSmemDq + 512;         // causal: 1 stage of Q, dO, K, V
constexpr size_t kSmemDqNc = 2 * 2 * kTB + kTB + kEpiSmemDq + 512;   // 2 stages of Q, dO
constexpr size_t kSmemDkdv = 4 * kTB + kTB + 4 * 128 * 4 + 4 * 128 * 4 + 512;  // y, e, 1/g, dt, cs
constexpr size_t kSmemDkdvNc = 3 * 2 * kTB + kTB + 2 * 128 * 4 + 512;         // 3 stages of K, V
static_assert(kSmemDkdvNc <= 232448 && kSmemDq <= 232448, "backward kernel exceeds the shared-memory limit");

bool set_bwd_attrs() {
    static int done = 0;
    if (done) return done > 0;
    const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
    bool ok = cudaFuncSetAttribute(tc::tc_bwd_dq_kernel<true>, A, (int)kSmemDq) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dq_kernel<false>, A, (int)kSmemDqNc) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel<true>, A, (int)kSmemDkdv) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_bwd_dkdv_kernel<false>, A, (int)kSmemDkdvNc) == cudaSuccess;
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
    const unsigned nthr = 64 + tc::kEpiThreads;
    cudaError_t e = tc_host::launch_agg(P, s);
    if (e == cudaSuccess) e = tc_host::launch_scan(P.slots, P, p.BH, p.causal ? 0 : 2, s);
    if (e != cudaSuccess) return e;
    if (p.causal)
        tc::tc_bwd_dq_kernel<true><<<P.sl.G, nthr, kSmemDq, s>>>(P);
    else
        tc::tc_bwd_dq_kernel<false><<<P.sl.G, nthr, kSmemDqNc, s>>>(P);
    e = tc_host::launch_scan(P.slots_rev, P, p.BH, p.causal ? 1 : 2, s);
    if (e != cudaSuccess) return e;
    if (p.causal)
        tc::tc_bwd_dkdv_kernel<true><<<P.sl.G, nthr, kSmemDkdv, s>>>(P);
    else
        tc::tc_bwd_dkdv_kernel<false><<<P.sl.G, nthr, kSmemDkdvNc, s>>>(P);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(5);
    return e;
}

}  // namespace la
