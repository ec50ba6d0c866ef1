// la_tc_wide.cu -- tcgen05 / TMA kernels for bf16 heads of D = 256: the forward and the backward.
//
// Method ("Transformer Based Linear Attention with Optimized GPU Kernel Implementation", sciencestack.ai
// page, TL;DR: forward/backward formulation, normalisation scheme, analytical gradients, O(N D^2) time,
// O(N D) memory; the D = 256 head is the widest of the head-size sweep, Figures 2 and 3).
//
// A D = 256 state (256 x 256 fp32) alone fills a CTA's tensor memory, so one CTA here computes one
// 128-column half of an output, with 256-deep contractions: TMEM holds the chunk's T = X Y^T (128
// columns), the output half (128) and the state half S = sum_j y_j w_j^T (256 rows of d, two 128-lane
// blocks: 256 columns).  The forward and the three gradients are all the same computation -- a linear
// attention without normalisation over query rows x, key rows y and value rows w,
//     out_i = sum_{j in m(i)} (c_ij + x_i . y_j) w_j,
// with the mask m and the constant c chosen per pass (dOt_i = dO_i / g_i, dt_i = dO_i . O_i / g_i):
//     forward  x = q,   y = k,   w = v,   c = 1,       j <= i,  then divided by g_i = sum_j (1 + q_i . k_j)
//     dQ       x = dOt, y = v,   w = k,   c = -dt_i,   j <= i   (per query row)
//     dK       x = v,   y = dOt, w = q,   c = -dt_j,   j >= i   (per key row)
//     dV       x = k,   y = q,   w = dOt, c = 1,       j >= i
// (dK_j = sum_{i >= j} dW_ij q_i and dV_j = sum_{i >= j} (W_ij / g_i) dO_i with dW_ij = dOt_i . v_j - dt_i).
// Per 128-row chunk (causal): out = X Sb + P W + c a, P_ij = m_ij (c_ij + T_ij) (bf16 in TMEM), Sb the
// bf16 state of the earlier chunks (later chunks, walking in reverse), a = sum c_j w_j over them; X Sb and
// S += Y^T W are issued while the epilogue forms P.  Non-causal: S, a (and z) over the whole head first, then out = X Sb + c a for every chunk.
// The normaliser g_i = n_i + q_i . z + r_i (z = sum k_j, r_i = sum_j P_ij) is formed by the forward and by
// a g-only pass of the same kernel that the backward runs first.
//
// Work split: CTA b computes column half b & 1 of heads b / 2, b / 2 + G / 2, ... from a zero state, so no
// state is carried between CTAs (B H = 64 heads give 128 CTAs).  The g-only pass has no halves.
// Roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2-9 epilogue (thread = chunk row i
// = TMEM lane, half hf = 64 of the 128 output columns).  Every barrier wait is bounded (AbortState).
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

enum : int { kWFwd = 0, kWG = 1, kWDq = 2, kWDk = 3, kWDv = 4 };

struct WideParams {
    CUtensorMap tmX, tmY, tmW, tmOut;  // bf16, 256 columns, boxes of 64 columns x 128 rows of one head
    int H;                             // heads per batch entry (map coordinates of a head)
    int BH;                            // heads
    long long N;                       // rows per head
    int nchunk;                        // chunks of kC rows per head
    uint32_t *status;                  // workspace status word
    float *g_out;                      // forward, g-only pass: g_i [BH, N] (forward: may be null)
    float *g_ws;                       // forward: also keep g_i here for the backward (may be null)
    const float *rs_dt;                // dQ, dK passes: dt_i [BH, N]
    const uint32_t *skip;              // dQ, dK, dV passes: skip everything when *skip (may be null)
    uint64_t tag[7];                   // forward with g_ws: the record of what g belongs to
    uint64_t wait_ns;                  // bound on one barrier wait (0: kWaitNs)
};

// The record a forward that keeps g in the workspace writes into the header's tag words, and that a
// reusing backward checks: Q's and K's addresses and strides, the shape and the mask.
__host__ __device__ inline void wide_g_tag(const void *Q, const void *K, uint64_t qk_layout, long long BH,
                                           long long N, int causal, uint64_t *t) {
    t[0] = 0x4C415F5749444547ull ^ qk_layout;  // "LA_WIDEG"
    t[1] = (uint64_t)(uintptr_t)Q;
    t[2] = (uint64_t)(uintptr_t)K;
    t[3] = (uint64_t)BH;
    t[4] = (uint64_t)N;
    t[5] = (uint64_t)causal;
    t[6] = 4;  // form: g of the D = 256 forward
}

// Thread 0 of a walk: whether the backward's row kernel found no matching record (then nothing is done).
__device__ __forceinline__ bool wide_skipped(const WideParams &P) {
    return P.skip != nullptr && *(volatile const uint32_t *)P.skip != 0u;
}

// Key row j's weight in an N = 16 MMA operand (8-row boxes of 128-byte rows, 128-byte swizzle, rows
// j < 64 in the first box): row 0 holds bf16(w), row 1 bf16(w - row 0); rows 2-7 stay zero.  An MMA of
// W^T against it puts sum_j w_j w_row_j, in two parts, into output columns 0 and 1.
__device__ __forceinline__ void weight_put(unsigned char *t, int j, float w) {
    unsigned char *bx = t + (j >> 6) * 1024;
    const int e = j & 63;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    *(__nv_bfloat16 *)(bx + ((e >> 3) << 4) + (e & 7) * 2) = hi;
    *(__nv_bfloat16 *)(bx + 128 + (((e >> 3) ^ 1) << 4) + (e & 7) * 2) = lo;
}
__device__ __forceinline__ float weight_get(const unsigned char *t, int j) {
    const unsigned char *bx = t + (j >> 6) * 1024;
    const int e = j & 63;
    return __bfloat162float(*(const __nv_bfloat16 *)(bx + ((e >> 3) << 4) + (e & 7) * 2)) +
           __bfloat162float(*(const __nv_bfloat16 *)(bx + 128 + (((e >> 3) ^ 1) << 4) + (e & 7) * 2));
}

// q_row . z over d in [128 hf, 128 hf + 128): boxes 2 hf and 2 hf + 1 of a four-box bf16 tile.
__device__ __forceinline__ float dot_quarter2(const unsigned char *xt, int row, int hf, const float *z) {
    return dot_half(xt + 2 * hf * kBox, row, 0, z + 128 * hf) + dot_half(xt + 2 * hf * kBox, row, 1, z + 128 * hf);
}

// Zeroes row `row` of the two boxes (row blocks 0 and 1) of column box hf of the bf16 state tile.
__device__ __forceinline__ void zero_state_rows(unsigned char *Sb, int row, int hf) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int rb = 0; rb < 2; ++rb) {
        unsigned char *box = Sb + (2 * rb + hf) * kBox;
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) *(uint4 *)(box + sw128_off(row, g8)) = z;
    }
}

// The value-side constant of an output row: u_i a (forward, dV: u = 1; dQ: u = -dt_i), or a^w itself (dK,
// where the weight sits inside the sum).  With the accumulator value v of output column e.
template <int MODE> __device__ __forceinline__ float with_const(float v, float a, float u) {
    if constexpr (MODE == kWDq) return fmaf(u, a, v);
    return v + a;
}

// ----------------------------------------------------------------------------------------------------
// Causal walk (forward or reverse chunk order).  TMEM: T 0-127 (P packed into 0-63 once read; the chunk's
// column sums z 64-95 and a 96-111 after that; the row-sum exchange 112-115), out 128-255, S 256-511.
// One stage of tiles, filled in three parts so that the next chunk's first T steps start while this
// chunk's out tile is still leaving: the low and high 128 columns of X and Y, and W.
// ----------------------------------------------------------------------------------------------------
template <int MODE, bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_wide_kernel(const __grid_constant__ WideParams P) {
    constexpr bool REV = MODE == kWDk || MODE == kWDv;
    constexpr bool HAS_W = MODE != kWG;
    constexpr bool NORM = MODE == kWFwd || MODE == kWG;
    constexpr bool KCONST = MODE == kWDk;
    constexpr uint32_t XB = 4 * kBox;  // an X or Y tile: 128 rows x 256 columns
    constexpr uint32_t WB = 2 * kBox;  // a W (or out) tile: 128 rows x 128 columns
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *xt = sm, *yt = sm + XB, *wt = sm + 2 * XB;
    unsigned char *Sb = sm + 2 * XB + WB;    // bf16 state [d][e]: box (row block rb, column box cb) at (2 rb + cb) kBox
    unsigned char *area = Sb + 4 * kBox;     // 2 KB: z (fp32, 256) + ones (forward, g-only); ones (dQ, dV); weights (dK)
    float *zc = (float *)area;
    unsigned char *ones = NORM ? area + 1024 : area;
    unsigned char *wtile = area;
    float *ac = (float *)(area + 2048);      // a (fp32, 128): the constant-weighted sum of the earlier w rows
    // The stage is filled and released in three parts: lo = columns 0-127 of X and Y, hi = columns 128-255
    // of X and Y, and W.  lo and W are free once the state update has read them; hi also holds the out tile.
    uint64_t *fullLo = (uint64_t *)(ac + 128);
    uint64_t *fullHi = fullLo + 1, *fullW = fullLo + 2, *emptyLW = fullLo + 3, *emptyHi = fullLo + 4;
    uint64_t *barT = fullLo + 5, *barP = fullLo + 6, *barSb = fullLo + 7, *barO = fullLo + 8, *barS = fullLo + 9;
    uint32_t *tslot = (uint32_t *)(fullLo + 10);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(fullLo, 1);
        mbar_init(fullHi, 1);
        mbar_init(fullW, 1);
        mbar_init(emptyLW, 1);  // the chunk's last MMA commit (the state update)
        mbar_init(emptyHi, 2);  // the last MMA commit + the epilogue once the out tile has left X's high half
        mbar_init(barT, 1);
        mbar_init(barP, kEpiThreads);
        mbar_init(barSb, kEpiThreads);
        mbar_init(barO, 1);
        mbar_init(barS, 1);
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    if (KCONST) {
        for (int k = threadIdx.x; k < 512; k += blockDim.x) ((uint32_t *)wtile)[k] = 0u;
    } else {
        for (int k = threadIdx.x; k < 256; k += blockDim.x) ((uint32_t *)ones)[k] = 0x3F803F80u;
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    griddep_launch_dependents();
    if (MODE == kWFwd && P.g_ws && blockIdx.x == 0 && threadIdx.x == 0) {  // g is kept: record for what
        volatile uint64_t *w = (volatile uint64_t *)((unsigned char *)P.status + 128);
        for (int k = 0; k < 7; ++k) w[k] = P.tag[k];
    }
    if (MODE >= kWDq) {  // the backward's row kernel may have found no forward state to use
        if (threadIdx.x == 0 && wide_skipped(P)) *abort_flag = 1;
        __syncthreads();
    }
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t tT = tmem, tO = tmem + 128, tS0 = tmem + 256, tS1 = tmem + 384;
    const uint32_t tZ0 = tT + 64, tZ1 = tT + 80, tA = tT + 96, tX = tT + 112;
    const int half = MODE == kWG ? 0 : (int)(blockIdx.x & 1);
    const int h0 = MODE == kWG ? (int)blockIdx.x : (int)(blockIdx.x >> 1);
    const int hstep = MODE == kWG ? (int)gridDim.x : (int)(gridDim.x >> 1);
    const int nch = P.nchunk;

    if (skip) {
        // no forward state to use: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer: X, Y (256 columns) and W (this CTA's half) of each chunk, one stage in three parts
        prefetch_tmap(&P.tmX);
        prefetch_tmap(&P.tmY);
        if (HAS_W) prefetch_tmap(&P.tmW);
        int it = 0, nlo = 0, nhi = 0, nw = 0;  // parts issued
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep) {
            const HeadCoord hc = head_coord<FLAT>(h, P.H);
            for (int k = 0; k < nch; ++k, ++it) {
                const int c = REV ? nch - 1 - k : k;
                if (it > 0 && !wait_or_abort(emptyLW, (it - 1) & 1, abort_flag, P.status, 0x501)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fullLo, 2 * WB);
                for (int nb = 0; nb < 2; ++nb) {
                    tile_load<FLAT>(xt + nb * kBox, &P.tmX, fullLo, nb * 64, c * kC, hc);
                    tile_load<FLAT>(yt + nb * kBox, &P.tmY, fullLo, nb * 64, c * kC, hc);
                }
                ++nlo;
                if (HAS_W) {
                    mbar_arrive_expect_tx(fullW, WB);
                    for (int nb = 0; nb < 2; ++nb)
                        tile_load<FLAT>(wt + nb * kBox, &P.tmW, fullW, 128 * half + 64 * nb, c * kC, hc);
                    ++nw;
                }
                if (it > 0 && !wait_or_abort(emptyHi, (it - 1) & 1, abort_flag, P.status, 0x505)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fullHi, 2 * WB);
                for (int nb = 2; nb < 4; ++nb) {
                    tile_load<FLAT>(xt + nb * kBox, &P.tmX, fullHi, nb * 64, c * kC, hc);
                    tile_load<FLAT>(yt + nb * kBox, &P.tmY, fullHi, nb * 64, c * kC, hc);
                }
                ++nhi;
                // the CTA's next chunk into L2 while this one is processed
                int nh = h, nk = k + 1;
                if (nk == nch) {
                    nh = h + hstep;
                    nk = 0;
                }
                if (nh < P.BH) {
                    const int nc = REV ? nch - 1 - nk : nk;
                    const HeadCoord hn = head_coord<FLAT>(nh, P.H);
                    for (int nb = 0; nb < 4; ++nb) {
                        tile_prefetch<FLAT>(&P.tmX, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmY, nb * 64, nc * kC, hn);
                    }
                    if (HAS_W)
                        for (int nb = 0; nb < 2; ++nb) tile_prefetch<FLAT>(&P.tmW, 128 * half + 64 * nb, nc * kC, hn);
                }
            }
        }
        if (!ok || *abort_flag) {  // issued copies land before the CTA exits
            if (nlo > 0) mbar_wait(fullLo, (nlo - 1) & 1, 50000000ull);
            if (nhi > 0) mbar_wait(fullHi, (nhi - 1) & 1, 50000000ull);
            if (nw > 0) mbar_wait(fullW, (nw - 1) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKK = idesc_bf16(128, 128, false, false);
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t idZ = idesc_bf16(128, 16, true, false);
        const uint32_t xb = smem_u32(xt), yb = smem_u32(yt), wb = smem_u32(wt), sb = smem_u32(Sb);
        const uint32_t cb = smem_u32(KCONST ? wtile : ones);
        int it = 0;
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep) {
            for (int k = 0; k < nch && ok; ++k, ++it) {
                const uint32_t ph = it & 1;
                ok = wait_or_abort(fullLo, ph, abort_flag, P.status, 0x502);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s) {  // T = X Y^T over columns 0-127 ...
                    const uint32_t o = (s >> 2) * kBox + 32 * (s & 3);
                    mma_ss(tT, sdesc_sw128(xb + o, 16, 1024), sdesc_sw128(yb + o, 16, 1024), idKK, s > 0);
                }
                ok = wait_or_abort(fullHi, ph, abort_flag, P.status, 0x506);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int s = 8; s < 16; ++s) {  // ... and 128-255
                    const uint32_t o = (s >> 2) * kBox + 32 * (s & 3);
                    mma_ss(tT, sdesc_sw128(xb + o, 16, 1024), sdesc_sw128(yb + o, 16, 1024), idKK, 1u);
                }
                mma_commit(barT);
                if (HAS_W) {
                    // once the epilogue has copied the state into Sb (and read the previous out): out = X Sb
                    // and S += Y^T W while the epilogue forms P
                    ok = wait_or_abort(barSb, ph, abort_flag, P.status, 0x504);
                    if (ok) ok = wait_or_abort(fullW, ph, abort_flag, P.status, 0x507);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int s = 0; s < 16; ++s)  // out = X Sb over the 256 rows d of the state
                        mma_ss(tO, sdesc_sw128(xb + (s >> 2) * kBox + 32 * (s & 3), 16, 1024),
                               sdesc_sw128(sb + (s >> 3) * 2 * kBox + 2048 * (s & 7), kBox, 1024), idKM, s > 0);
                    if (k + 1 < nch) {
#pragma unroll
                        for (int s = 0; s < 8; ++s) {  // S += Y^T W, rows d of the two 128-column blocks of Y
                            const uint32_t acc = (k > 0 || s > 0) ? 1u : 0u;
                            mma_ss(tS0, sdesc_sw128(yb + 2048 * s, kBox, 1024), sdesc_sw128(wb + 2048 * s, kBox, 1024),
                                   idMM, acc);
                            mma_ss(tS1, sdesc_sw128(yb + 2 * kBox + 2048 * s, kBox, 1024),
                                   sdesc_sw128(wb + 2048 * s, kBox, 1024), idMM, acc);
                        }
                    }
                }
                mma_commit(barS);  // also: X Sb, Sb's reader, is complete
                ok = wait_or_abort(barP, ph, abort_flag, P.status, 0x503);  // T read out; P in TMEM
                if (!ok) break;
                tc_fence_after();
                if (HAS_W) {
#pragma unroll
                    for (int s = 0; s < 8; ++s)  // out += P W (P in TMEM, 16 rows j per step)
                        mma_ts(tO, tT + 8 * s, sdesc_sw128(wb + 2048 * s, kBox, 1024), idKM, 1u);
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {  // the chunk's column sums: z = Y^T 1, a = W^T c
                    const uint64_t cd = KCONST ? sdesc_sw128(cb + (s >> 2) * 1024 + 32 * (s & 3), 16, 0)
                                               : sdesc_sw128(cb + 32 * (s & 3), 16, 0);
                    if (NORM) {
                        mma_ss(tZ0, sdesc_sw128(yb + 2048 * s, kBox, 1024), cd, idZ, s > 0);
                        mma_ss(tZ1, sdesc_sw128(yb + 2 * kBox + 2048 * s, kBox, 1024), cd, idZ, s > 0);
                    }
                    if (HAS_W) mma_ss(tA, sdesc_sw128(wb + 2048 * s, kBox, 1024), cd, idZ, s > 0);
                }
                mma_commit(barO);
                mma_commit(emptyLW);
                mma_commit(emptyHi);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread <-> chunk row i (TMEM lane) and output column half hf
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0;
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep) {
            const HeadCoord hc = head_coord<FLAT>(h, P.H);
            // a zero state at the head's start (the previous head's last MMAs on Sb are done: its barO)
            if (HAS_W) {
                zero_state_rows(Sb, i, hf);
                fence_proxy_async_smem();
                if (hf == 1) ac[i] = 0.f;
            }
            if (NORM && hf == 0) {
                zc[i] = 0.f;
                zc[128 + i] = 0.f;
            }
            epi_sync256();
            if (HAS_W) mbar_arrive(barSb);
            for (int k = 0; k < nch; ++k, ++it) {
                const int c = REV ? nch - 1 - k : k;
                const uint32_t ph = it & 1;
                const long long row0 = (long long)c * kC;
                const bool row_ok = row0 + i < P.N;
                const size_t rix = (size_t)h * P.N + (row_ok ? row0 + i : 0);
                const bool rix_ok = in_range((long long)rix, (long long)P.BH * P.N, P.status, 0xB010);
                float u = 1.f;  // query-side constant of row i
                if (MODE == kWDq) u = row_ok && rix_ok ? -P.rs_dt[rix] : 0.f;
                if (KCONST) {  // key-side constants of the chunk's rows (the previous chunk's MMAs read theirs: barO)
                    if (hf == 0) weight_put(wtile, i, row_ok && rix_ok ? -P.rs_dt[rix] : 0.f);
                    fence_proxy_async_smem();
                    epi_sync256();
                }
                ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x510);
                if (!ok) break;
                tc_fence_after();
                float part = 0.f;
                {  // P = m(c + T) over this half's columns j; r_i partial (fp32, before rounding)
                    uint32_t t0[32], t1[32], pk[32];
                    tmem_ld32(tT + lo + 64 * hf, t0);
                    tmem_ld32(tT + lo + 64 * hf + 32, t1);
                    tmem_wait_ld(t0);
                    tmem_wait_ld(t1);
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int j = 64 * hf + 2 * m;
                        const uint32_t a0 = m < 16 ? t0[2 * m] : t1[2 * m - 32];
                        const uint32_t a1 = m < 16 ? t0[2 * m + 1] : t1[2 * m - 31];
                        const bool in0 = REV ? j >= i : j <= i, in1 = REV ? j + 1 >= i : j + 1 <= i;
                        const float c0 = KCONST ? weight_get(wtile, j) : u;
                        const float c1 = KCONST ? weight_get(wtile, j + 1) : u;
                        const float p0 = in0 ? c0 + __uint_as_float(a0) : 0.f;
                        const float p1 = in1 ? c1 + __uint_as_float(a1) : 0.f;
                        pk[m] = pack_bf16(p0, p1);
                        if (NORM) part += p0 + p1;
                    }
                    tc_fence_before();
                    epi_sync256();  // both halves have read T before P and the exchange overwrite it
                    tc_fence_after();
                    if (HAS_W) tmem_st32(tT + lo + 32 * hf, pk);
                }
                const uint32_t tXc = tX + lo + 2 * (it & 1);
                if (NORM) {
                    part += dot_quarter2(xt, i, hf, zc);  // q_i . z over this half's 128 entries of d
                    tmem_st1(tXc + hf, __float_as_uint(part));
                }
                if (HAS_W || NORM) tmem_st_wait();
                tc_fence_before();
                mbar_arrive(barP);
                float gi = 0.f, inv = 1.f;
                if (NORM) {  // g_i = n + q_i . z + r_i from both halves
                    epi_sync256();
                    tc_fence_after();
                    uint32_t x0, x1;
                    tmem_ld2(tXc, x0, x1);
                    tmem_wait_ld(x0, x1);
                    gi = (float)row0 + __uint_as_float(x0) + __uint_as_float(x1);
                    inv = 1.f / gi;
                    if (row_ok && hf == 0) {
                        if (P.g_out && rix_ok) P.g_out[rix] = gi;
                        if (MODE == kWFwd && P.g_ws && rix_ok) P.g_ws[rix] = gi;
                    }
                }
                ok = wait_or_abort(barO, ph, abort_flag, P.status, 0x511);
                if (!ok) break;
                tc_fence_after();
                float zn0 = 0.f, zn1 = 0.f, an = 0.f;  // z (hf 0: rows d = i, 128 + i) and a (hf 1: e = i) after the chunk
                if (NORM && hf == 0) {
                    uint32_t v0, v1, w0, w1;
                    tmem_ld2(tZ0 + lo, v0, v1);
                    tmem_ld2(tZ1 + lo, w0, w1);
                    tmem_wait_ld(v0, v1);
                    tmem_wait_ld(w0, w1);
                    zn0 = zc[i] + __uint_as_float(v0);
                    zn1 = zc[128 + i] + __uint_as_float(w0);
                }
                if (HAS_W && hf == 1) {
                    uint32_t v0, v1;
                    tmem_ld2(tA + lo, v0, v1);
                    tmem_wait_ld(v0, v1);
                    an = ac[i] + __uint_as_float(v0) + (KCONST ? __uint_as_float(v1) : 0.f);
                }
                if (HAS_W) {
                    // out_i = [P W + X Sb]_i + constant (forward: / g_i), staged in X's high half (its readers,
                    // the MMAs and this row's q . z, are done)
                    unsigned char *otile = xt + (2 + hf) * kBox;
#pragma unroll 1
                    for (int half32 = 0; half32 < 2; ++half32) {
                        uint32_t v[32];
                        tmem_ld32(tO + lo + 64 * hf + 32 * half32, v);
                        tmem_wait_ld(v);
                        const float *aa = ac + 64 * hf + 32 * half32;
                        uint4 w4[4];
                        uint32_t *wv = (uint32_t *)w4;
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const float e0 = with_const<MODE>(__uint_as_float(v[2 * m]), aa[2 * m], u) * inv;
                            const float e1 = with_const<MODE>(__uint_as_float(v[2 * m + 1]), aa[2 * m + 1], u) * inv;
                            wv[m] = pack_bf16(e0, e1);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) *(uint4 *)(otile + sw128_off(i, 4 * half32 + q)) = w4[q];
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                epi_sync256();  // the out tile is complete; every read of z, a and the exchange is done
                if (threadIdx.x == 64 && HAS_W) {
                    for (int nb = 0; nb < 2; ++nb)
                        tile_store<FLAT>(&P.tmOut, xt + (2 + nb) * kBox, 128 * half + 64 * nb, (int)row0, hc);
                    bulk_commit();
                }
                if (NORM && hf == 0) {
                    zc[i] = zn0;
                    zc[128 + i] = zn1;
                }
                if (HAS_W && hf == 1) ac[i] = an;
                ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x512);
                if (!ok) break;
                tc_fence_after();
                if (HAS_W && k + 1 < nch) {  // S after this chunk -> Sb for the next (X Sb of this chunk is done)
                    tmem_half_to_tile(tS0 + lo, Sb, i, hf);
                    tmem_half_to_tile(tS1 + lo, Sb + 2 * kBox, i, hf);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(barSb);
                }
                if (threadIdx.x == 64) {  // after the copy the next chunk's MMAs wait for
                    if (HAS_W) bulk_wait_read0();  // the out tile has left X's high half
                    mbar_arrive(emptyHi);
                }
                epi_sync256();  // z, a of the next chunk are in place
            }
        }
    }
    if (threadIdx.x == 64) bulk_wait0();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------------------------------
// Non-causal: per head, phase A sums S = Y^T W, z = Y^T 1 and a = W^T c over every chunk (one stage of Y,
// W); the epilogue turns them into Sb, z, a; phase B forms out = X Sb + constant for every chunk (two
// stages of X, two TMEM output buffers).  TMEM: output buffers 0-127 and 128-255 (phase A's column sums
// in 0-47), S 256-511 (its first columns hold the row-sum exchange once Sb is made).
// ----------------------------------------------------------------------------------------------------
template <int MODE, bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_wide_nc_kernel(const __grid_constant__ WideParams P) {
    constexpr bool HAS_W = MODE != kWG;
    constexpr bool NORM = MODE == kWFwd || MODE == kWG;
    constexpr bool KCONST = MODE == kWDk;
    constexpr uint32_t XB = 4 * kBox, WB = 2 * kBox;
    constexpr uint32_t STAGE_A = XB + (HAS_W ? WB : 0);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *region = sm;           // phase A: Y at +0, W at +XB; phase B: X stages at +0 and +XB
    unsigned char *Sb = sm + 2 * XB;
    unsigned char *area = Sb + 4 * kBox;  // as in the causal kernel
    float *zc = (float *)area;
    unsigned char *ones = NORM ? area + 1024 : area;
    unsigned char *wtile = area;
    float *ac = (float *)(area + 2048);
    uint64_t *fullA = (uint64_t *)(ac + 128);
    uint64_t *emptyA = fullA + 1, *barW = fullA + 2, *barA = fullA + 3, *barSb = fullA + 4;
    uint64_t *fullB = fullA + 5, *emptyB = fullA + 7, *barOB = fullA + 9, *barOf = fullA + 11;  // [2] each
    uint32_t *tslot = (uint32_t *)(fullA + 13);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(fullA, 1);
        mbar_init(emptyA, 1);
        mbar_init(barW, kEpiThreads);
        mbar_init(barA, 1);
        mbar_init(barSb, kEpiThreads);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&fullB[b], 1);
            mbar_init(&emptyB[b], HAS_W ? 2 : 1);  // (the MMA commit +) the epilogue once it is done with X
            mbar_init(&barOB[b], 1);
            mbar_init(&barOf[b], kEpiThreads);
        }
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    if (KCONST) {
        for (int k = threadIdx.x; k < 512; k += blockDim.x) ((uint32_t *)wtile)[k] = 0u;
    } else {
        for (int k = threadIdx.x; k < 256; k += blockDim.x) ((uint32_t *)ones)[k] = 0x3F803F80u;
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    griddep_launch_dependents();
    if (MODE == kWFwd && P.g_ws && blockIdx.x == 0 && threadIdx.x == 0) {  // g is kept: record for what
        volatile uint64_t *w = (volatile uint64_t *)((unsigned char *)P.status + 128);
        for (int k = 0; k < 7; ++k) w[k] = P.tag[k];
    }
    if (MODE >= kWDq) {  // the backward's row kernel may have found no forward state to use
        if (threadIdx.x == 0 && wide_skipped(P)) *abort_flag = 1;
        __syncthreads();
    }
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t tS0 = tmem + 256, tS1 = tmem + 384;
    const uint32_t tZ0 = tmem, tZ1 = tmem + 16, tA = tmem + 32, tX = tS0;
    const int half = MODE == kWG ? 0 : (int)(blockIdx.x & 1);
    const int h0 = MODE == kWG ? (int)blockIdx.x : (int)(blockIdx.x >> 1);
    const int hstep = MODE == kWG ? (int)gridDim.x : (int)(gridDim.x >> 1);
    const int nch = P.nchunk;

    if (skip) {
        // no forward state to use: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmX);
        prefetch_tmap(&P.tmY);
        if (HAS_W) prefetch_tmap(&P.tmW);
        int nA = 0, nB[2] = {0, 0};  // loads issued per barrier
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep) {
            const HeadCoord hc = head_coord<FLAT>(h, P.H);
            // phase A overwrites both X stages of the previous head's phase B: let their outputs leave first
            for (int b = 0; b < 2 && ok; ++b)
                if (nB[b] > 0) ok = wait_or_abort(&emptyB[b], (nB[b] - 1) & 1, abort_flag, P.status, 0x521);
            for (int k = 0; k < nch && ok; ++k) {
                if (nA > 0 && !wait_or_abort(emptyA, (nA - 1) & 1, abort_flag, P.status, 0x522)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(fullA, STAGE_A);
                for (int nb = 0; nb < 4; ++nb) tile_load<FLAT>(region + nb * kBox, &P.tmY, fullA, nb * 64, k * kC, hc);
                if (HAS_W)
                    for (int nb = 0; nb < 2; ++nb)
                        tile_load<FLAT>(region + XB + nb * kBox, &P.tmW, fullA, 128 * half + 64 * nb, k * kC, hc);
                ++nA;
            }
            if (ok && nA > 0) ok = wait_or_abort(emptyA, (nA - 1) & 1, abort_flag, P.status, 0x523);  // Y, W read
            for (int k = 0; k < nch && ok; ++k) {
                const int s = k & 1;  // phase B's loads alternate stages within each head
                if (nB[s] > 0 && !wait_or_abort(&emptyB[s], (nB[s] - 1) & 1, abort_flag, P.status, 0x524)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&fullB[s], XB);
                for (int nb = 0; nb < 4; ++nb)
                    tile_load<FLAT>(region + s * XB + nb * kBox, &P.tmX, &fullB[s], nb * 64, k * kC, hc);
                ++nB[s];
            }
        }
        if (!ok || *abort_flag) {  // let the copies already issued land before the CTA exits
            if (nA > 0) mbar_wait(fullA, (nA - 1) & 1, 50000000ull);
            for (int b = 0; b < 2; ++b)
                if (nB[b] > 0) mbar_wait(&fullB[b], (nB[b] - 1) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t idZ = idesc_bf16(128, 16, true, false);
        const uint32_t rb = smem_u32(region), sb = smem_u32(Sb);
        const uint32_t cb = smem_u32(KCONST ? wtile : ones);
        int nA = 0, nB[2] = {0, 0}, hn = 0;
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep, ++hn) {
            // phase A writes the column sums into output buffer 0: the previous head's outputs are read
            for (int b = 0; b < 2 && ok && HAS_W; ++b)
                if (nB[b] > 0) ok = wait_or_abort(&barOf[b], (nB[b] - 1) & 1, abort_flag, P.status, 0x531);
            for (int k = 0; k < nch && ok; ++k, ++nA) {
                ok = wait_or_abort(fullA, nA & 1, abort_flag, P.status, 0x532);
                if (ok && KCONST) ok = wait_or_abort(barW, nA & 1, abort_flag, P.status, 0x533);
                if (!ok) break;
                tc_fence_after();
                const uint32_t yb = rb, wb = rb + XB;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t acc = (k > 0 || s > 0) ? 1u : 0u;
                    const uint64_t cd = KCONST ? sdesc_sw128(cb + (s >> 2) * 1024 + 32 * (s & 3), 16, 0)
                                               : sdesc_sw128(cb + 32 * (s & 3), 16, 0);
                    if (HAS_W) {  // S += Y^T W ; a += W^T c
                        mma_ss(tS0, sdesc_sw128(yb + 2048 * s, kBox, 1024), sdesc_sw128(wb + 2048 * s, kBox, 1024),
                               idMM, acc);
                        mma_ss(tS1, sdesc_sw128(yb + 2 * kBox + 2048 * s, kBox, 1024),
                               sdesc_sw128(wb + 2048 * s, kBox, 1024), idMM, acc);
                        mma_ss(tA, sdesc_sw128(wb + 2048 * s, kBox, 1024), cd, idZ, acc);
                    }
                    if (NORM) {  // z += Y^T 1
                        mma_ss(tZ0, sdesc_sw128(yb + 2048 * s, kBox, 1024), cd, idZ, acc);
                        mma_ss(tZ1, sdesc_sw128(yb + 2 * kBox + 2048 * s, kBox, 1024), cd, idZ, acc);
                    }
                }
                mma_commit(emptyA);
            }
            if (!ok) break;
            mma_commit(barA);
            if (!HAS_W) continue;  // the g-only pass needs no MMA in phase B
            ok = wait_or_abort(barSb, hn & 1, abort_flag, P.status, 0x534);  // Sb, z, a are ready
            if (!ok) break;
            for (int k = 0; k < nch && ok; ++k) {
                const int s = k & 1;
                ok = wait_or_abort(&fullB[s], nB[s] & 1, abort_flag, P.status, 0x535);
                if (ok && nB[s] > 0) ok = wait_or_abort(&barOf[s], (nB[s] - 1) & 1, abort_flag, P.status, 0x536);
                if (!ok) break;
                tc_fence_after();
                const uint32_t xb = rb + s * XB;
#pragma unroll
                for (int t = 0; t < 16; ++t)  // out = X Sb over the 256 rows d of the state
                    mma_ss(tmem + 128 * s, sdesc_sw128(xb + (t >> 2) * kBox + 32 * (t & 3), 16, 1024),
                           sdesc_sw128(sb + (t >> 3) * 2 * kBox + 2048 * (t & 7), kBox, 1024), idKM, t > 0);
                mma_commit(&barOB[s]);
                mma_commit(&emptyB[s]);
                ++nB[s];
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int nA = 0, nB[2] = {0, 0}, hn = 0;
        bool ok = true;
        for (int h = h0; h < P.BH && ok; h += hstep, ++hn) {
            const HeadCoord hc = head_coord<FLAT>(h, P.H);
            if (KCONST) {  // each chunk's key weights, before phase A's MMA of that chunk
                for (int k = 0; k < nch && ok; ++k, ++nA) {
                    if (nA > 0) ok = wait_or_abort(emptyA, (nA - 1) & 1, abort_flag, P.status, 0x541);
                    if (!ok) break;
                    const long long r = (long long)k * kC + i;
                    if (hf == 0) {
                        const long long x = (long long)h * P.N + r;
                        weight_put(wtile, i, r < P.N && in_range(x, (long long)P.BH * P.N, P.status, 0xB011)
                                                 ? -P.rs_dt[x] : 0.f);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(barW);
                }
                if (!ok) break;
            }
            ok = wait_or_abort(barA, hn & 1, abort_flag, P.status, 0x542);
            if (!ok) break;
            tc_fence_after();
            // the head's sums -> Sb (bf16), z, a
            if (HAS_W) {
                tmem_half_to_tile(tS0 + lo, Sb, i, hf);
                tmem_half_to_tile(tS1 + lo, Sb + 2 * kBox, i, hf);
                if (hf == 1) {
                    uint32_t v0, v1;
                    tmem_ld2(tA + lo, v0, v1);
                    tmem_wait_ld(v0, v1);
                    ac[i] = __uint_as_float(v0) + (KCONST ? __uint_as_float(v1) : 0.f);
                }
                fence_proxy_async_smem();
            }
            if (NORM && hf == 0) {
                uint32_t v0, v1, w0, w1;
                tmem_ld2(tZ0 + lo, v0, v1);
                tmem_ld2(tZ1 + lo, w0, w1);
                tmem_wait_ld(v0, v1);
                tmem_wait_ld(w0, w1);
                zc[i] = __uint_as_float(v0);
                zc[128 + i] = __uint_as_float(w0);
            }
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barSb);
            for (int k = 0; k < nch; ++k) {
                const int s = k & 1;
                const uint32_t phs = nB[s] & 1;
                const long long row0 = (long long)k * kC;
                const bool row_ok = row0 + i < P.N;
                const size_t rix = (size_t)h * P.N + (row_ok ? row0 + i : 0);
                const bool rix_ok = in_range((long long)rix, (long long)P.BH * P.N, P.status, 0xB010);
                unsigned char *xs = region + s * XB;
                float u = 1.f;
                if (MODE == kWDq) u = row_ok && rix_ok ? -P.rs_dt[rix] : 0.f;
                float inv = 1.f;
                if (NORM) {  // g_i = N + q_i . z, halves exchanged through two TMEM columns
                    ok = wait_or_abort(&fullB[s], phs, abort_flag, P.status, 0x543);
                    if (!ok) break;
                    const float part = dot_quarter2(xs, i, hf, zc);
                    const uint32_t tXc = tX + lo + 2 * (k & 1);
                    tmem_st1(tXc + hf, __float_as_uint(part));
                    tmem_st_wait();
                    tc_fence_before();
                    epi_sync256();
                    tc_fence_after();
                    uint32_t x0, x1;
                    tmem_ld2(tXc, x0, x1);
                    tmem_wait_ld(x0, x1);
                    const float gi = (float)P.N + __uint_as_float(x0) + __uint_as_float(x1);
                    inv = 1.f / gi;
                    if (row_ok && hf == 0) {
                        if (P.g_out && rix_ok) P.g_out[rix] = gi;
                        if (MODE == kWFwd && P.g_ws && rix_ok) P.g_ws[rix] = gi;
                    }
                }
                if (HAS_W) {
                    ok = wait_or_abort(&barOB[s], phs, abort_flag, P.status, 0x544);
                    if (!ok) break;
                    tc_fence_after();
                    unsigned char *otile = xs + hf * kBox;  // X is read (X Sb done, q . z done before the sync)
#pragma unroll 1
                    for (int half32 = 0; half32 < 2; ++half32) {
                        uint32_t v[32];
                        tmem_ld32(tmem + 128 * s + lo + 64 * hf + 32 * half32, v);
                        tmem_wait_ld(v);
                        const float *aa = ac + 64 * hf + 32 * half32;
                        uint4 w4[4];
                        uint32_t *wv = (uint32_t *)w4;
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const float e0 = with_const<MODE>(__uint_as_float(v[2 * m]), aa[2 * m], u) * inv;
                            const float e1 = with_const<MODE>(__uint_as_float(v[2 * m + 1]), aa[2 * m + 1], u) * inv;
                            wv[m] = pack_bf16(e0, e1);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) *(uint4 *)(otile + sw128_off(i, 4 * half32 + q)) = w4[q];
                    }
                    tc_fence_before();
                    mbar_arrive(&barOf[s]);
                    fence_proxy_async_smem();
                }
                epi_sync256();  // the out tile is complete (every read of X, the exchange, z and a is done)
                if (threadIdx.x == 64) {
                    if (HAS_W) {
                        for (int nb = 0; nb < 2; ++nb)
                            tile_store<FLAT>(&P.tmOut, xs + nb * kBox, 128 * half + 64 * nb, (int)row0, hc);
                        bulk_commit();
                        bulk_wait_read0();
                    }
                    mbar_arrive(&emptyB[s]);
                }
                ++nB[s];
            }
            epi_sync256();  // Sb, z and a of this head are no longer read
        }
    }
    if (threadIdx.x == 64) bulk_wait0();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------------------------------
// Row terms of the backward: dt_i = (dO_i . O_i) / g_i and dOt_i = dO_i / g_i (bf16, contiguous
// [B H, N, 256]).  A warp takes kRowsPerWarp rows, a lane 8 consecutive columns of each; every load of
// the warp's rows is issued before the first is used, so that enough bytes are in flight.
// ----------------------------------------------------------------------------------------------------
constexpr int kRowsPerWarp = 4;

struct WideTag {
    uint64_t t[7];
};

// With `check`, g comes from the forward: every block first compares the workspace record with `expect`;
// on a mismatch nothing is computed, block 0 reports LA_ERR_STATE and tells the walks to skip.
__global__ void __launch_bounds__(256) wide_rowstats_kernel(const __nv_bfloat16 *__restrict__ dO, Layout ldo,
                                                            const __nv_bfloat16 *__restrict__ O, Layout lo,
                                                            const float *__restrict__ g, float *__restrict__ dt,
                                                            __nv_bfloat16 *__restrict__ dOt, int H, long long N,
                                                            long long rows, uint32_t *status, int check,
                                                            WideTag expect) {
    __shared__ int bad;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        bool match = true;
        if (check) {
            const volatile uint64_t *w = (const volatile uint64_t *)((const unsigned char *)status + 128);
            for (int k = 0; k < 7; ++k) match = match && w[k] == expect.t[k];
        }
        bad = match ? 0 : 1;
        if (blockIdx.x == 0) {
            ((WsHeader *)status)->wide_skip = match ? 0u : 1u;
            if (!match) report(status, kDevState, 0x5A7Fu);
        }
    }
    __syncthreads();
    if (bad) return;
    const int lane = threadIdx.x & 31;
    const long long r0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRowsPerWarp;
    uint4 a[kRowsPerWarp], o[kRowsPerWarp];
    float gi[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        const long long r = r0 + k < rows ? r0 + k : rows - 1;  // rows past the end repeat the last (not stored)
        const long long bh = r / N, n = r - bh * N;
        const long long b = bh / H, h = bh - b * H;
        a[k] = *(const uint4 *)(dO + b * ldo.sb + h * ldo.sh + n * ldo.sn + 8 * lane);
        o[k] = *(const uint4 *)(O + b * lo.sb + h * lo.sh + n * lo.sn + 8 * lane);
        gi[k] = in_range(r, rows, status, 0xB012) ? g[r] : 1.f;
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        const uint32_t av[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, ov[4] = {o[k].x, o[k].y, o[k].z, o[k].w};
        float d = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            d = fmaf(bf16lo(av[q]), bf16lo(ov[q]), d);
            d = fmaf(bf16hi(av[q]), bf16hi(ov[q]), d);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (r0 + k >= rows || !in_range(r0 + k, rows, status, 0xB012)) continue;
        const float ig = 1.f / gi[k];
        if (lane == 0) dt[r0 + k] = d * ig;
        uint4 sc;
        uint32_t *sv = (uint32_t *)&sc;
#pragma unroll
        for (int q = 0; q < 4; ++q) sv[q] = pack_bf16(bf16lo(av[q]) * ig, bf16hi(av[q]) * ig);
        *(uint4 *)(dOt + (r0 + k) * 256 + 8 * lane) = sc;
    }
}

}  // namespace tc

// ======================================================================================== host ===

namespace {

using tc::WideParams;
typedef void (*WideKernel)(const WideParams);

constexpr size_t kSmemWide = 2 * 4 * (size_t)tc::kBox + 2 * (size_t)tc::kBox + 4 * (size_t)tc::kBox + 2048 + 512 + 256;
constexpr size_t kSmemWideNc = 2 * 4 * (size_t)tc::kBox + 4 * (size_t)tc::kBox + 2048 + 512 + 256;
static_assert(kSmemWide <= 232448 && kSmemWideNc <= 232448, "wide kernels exceed the shared-memory limit");

template <int MODE, bool FLAT> WideKernel wide_kernel(bool causal) {
    return causal ? tc::tc_wide_kernel<MODE, FLAT> : tc::tc_wide_nc_kernel<MODE, FLAT>;
}

WideKernel pick(int mode, bool causal, bool flat) {
    switch (mode) {
        case tc::kWFwd: return flat ? wide_kernel<tc::kWFwd, true>(causal) : wide_kernel<tc::kWFwd, false>(causal);
        case tc::kWG: return flat ? wide_kernel<tc::kWG, true>(causal) : wide_kernel<tc::kWG, false>(causal);
        case tc::kWDq: return flat ? wide_kernel<tc::kWDq, true>(causal) : wide_kernel<tc::kWDq, false>(causal);
        case tc::kWDk: return flat ? wide_kernel<tc::kWDk, true>(causal) : wide_kernel<tc::kWDk, false>(causal);
        default: return flat ? wide_kernel<tc::kWDv, true>(causal) : wide_kernel<tc::kWDv, false>(causal);
    }
}

bool set_wide_attrs() {
    static std::atomic<int> state[kMaxDevices];
    return once_per_device(state, [] {
        const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
        for (int mode = 0; mode < 5; ++mode)
            for (int c = 0; c < 2; ++c)
                for (int f = 0; f < 2; ++f)
                    if (cudaFuncSetAttribute(pick(mode, c != 0, f != 0), A, (int)(c ? kSmemWide : kSmemWideNc)) !=
                        cudaSuccess)
                        return false;
        return true;
    });
}

cudaError_t launch_wide(int mode, bool causal, bool flat, const WideParams &P, int nsm, cudaStream_t s) {
    // one CTA per (head, output half); the g-only pass has no halves
    int cap = nsm;
    // Test hook: fewer CTAs, so that small problems also exercise several heads per CTA.
    if (const char *env = getenv("LA_TC_MAX_CTAS")) {
        const long long c = atoll(env);
        if (c >= 2 && c < cap) cap = (int)c;
    }
    int G = mode == tc::kWG ? (P.BH < cap ? P.BH : cap) : 2 * (P.BH < cap / 2 ? P.BH : cap / 2);
    if (G < 1) G = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(64 + tc::kEpiThreads);
    cfg.dynamicSmemBytes = causal ? kSmemWide : kSmemWideNc;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pick(mode, causal, flat), P);
}

bool wide_common(WideParams &P, const Plan &p) {
    memset(&P, 0, sizeof(P));
    P.H = p.H;
    P.BH = p.BH;
    P.N = p.N;
    P.nchunk = (p.N + tc::kC - 1) / tc::kC;
    P.wait_ns = 0;
    if (const char *env = getenv("LA_TEST_WAIT_NS")) {
        const long long ns = atoll(env);
        if (ns >= 1000000) P.wait_ns = (uint64_t)ns;
    }
    return true;
}

}  // namespace

bool wide_supported(const Plan &p) { return p.dtype == 1 && p.D == 256; }

uint64_t qk_layout(const Plan &p) {  // FNV-1a over Q's and K's strides
    uint64_t hsh = 0xcbf29ce484222325ull;
    for (int op : {kOpQ, kOpK})
        for (long long v : {p.lay[op].sb, p.lay[op].sh, p.lay[op].sn}) hsh = (hsh ^ (uint64_t)v) * 0x100000001b3ull;
    return hsh;
}

cudaError_t wide_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                         unsigned char *ws, cudaStream_t s, bool keep_g) {
    if (!set_wide_attrs()) return cudaErrorInvalidValue;
    const int nsm = tc_host::sm_count();
    if (nsm <= 1) return cudaErrorInvalidDevice;
    WideParams P;
    wide_common(P, p);
    const int ops[4] = {kOpQ, kOpK, kOpV, kOpO};
    const bool flat = tc_host::flat_heads(p, ops, 4);
    if (!tc_host::make_map(&P.tmX, Q, p, kOpQ, flat) || !tc_host::make_map(&P.tmY, K, p, kOpK, flat) ||
        !tc_host::make_map(&P.tmW, V, p, kOpV, flat) || !tc_host::make_map(&P.tmOut, O, p, kOpO, flat))
        return cudaErrorInvalidValue;
    P.status = (uint32_t *)ws;
    P.g_out = g;
    if (keep_g) {  // the workspace has room for the backward's row terms: keep g there for it
        P.g_ws = (float *)(ws + p.off_rowstats);
        tc::wide_g_tag(Q, K, qk_layout(p), p.BH, p.N, p.causal, P.tag);
    }
    const cudaError_t e = launch_wide(tc::kWFwd, p.causal != 0, flat, P, nsm, s);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t wide_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O,
                          const void *dO, void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s,
                          bool reuse_g) {
    if (!set_wide_attrs()) return cudaErrorInvalidValue;
    const int nsm = tc_host::sm_count();
    if (nsm <= 1) return cudaErrorInvalidDevice;
    const bool causal = p.causal != 0;
    float *rs_g = (float *)(ws + p.off_rowstats);
    float *rs_dt = rs_g + (size_t)p.BH * p.N;
    __nv_bfloat16 *dOt = (__nv_bfloat16 *)(ws + p.off_states);
    // dOt is a contiguous [B, H, N, D] operand: its map takes the place of dO's
    Plan q = p;
    q.lay[kOpdO] = Layout{(long long)p.H * p.N * p.D, (long long)p.N * p.D, (long long)p.D};
    const int ops[8] = {kOpQ, kOpK, kOpV, kOpO, kOpdO, kOpdQ, kOpdK, kOpdV};
    const bool flat = tc_host::flat_heads(p, ops, 8);
    unsigned launches = 0;
    WideParams P;
    wide_common(P, p);
    P.status = (uint32_t *)ws;
    // 1. g_i (the forward's normaliser) from Q and K, unless the forward kept it in the workspace
    cudaError_t e = cudaSuccess;
    if (!reuse_g) {
        if (!tc_host::make_map(&P.tmX, Q, p, kOpQ, flat) || !tc_host::make_map(&P.tmY, K, p, kOpK, flat))
            return cudaErrorInvalidValue;
        P.g_out = rs_g;
        if ((e = launch_wide(tc::kWG, causal, flat, P, nsm, s)) != cudaSuccess) return e;
        ++launches;
    }
    // 2. dt_i and dOt = dO / g (checking, when g is reused, that it belongs to these Q, K and shape)
    {
        tc::WideTag expect;
        tc::wide_g_tag(Q, K, qk_layout(p), p.BH, p.N, p.causal, expect.t);
        const long long rows = (long long)p.BH * p.N;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((rows + 8 * tc::kRowsPerWarp - 1) / (8 * tc::kRowsPerWarp)));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc::wide_rowstats_kernel, (const __nv_bfloat16 *)dO, p.lay[kOpdO],
                               (const __nv_bfloat16 *)O, p.lay[kOpO], (const float *)rs_g, rs_dt, dOt, p.H,
                               (long long)p.N, rows, (uint32_t *)ws, reuse_g ? 1 : 0, expect);
        if (e != cudaSuccess) return e;
        ++launches;
    }
    P.g_out = nullptr;
    P.rs_dt = rs_dt;
    P.skip = &((const WsHeader *)ws)->wide_skip;
    // 3. dQ: x = dOt, y = V, w = K
    if (!tc_host::make_map(&P.tmX, dOt, q, kOpdO, flat) || !tc_host::make_map(&P.tmY, V, p, kOpV, flat) ||
        !tc_host::make_map(&P.tmW, K, p, kOpK, flat) || !tc_host::make_map(&P.tmOut, dQ, p, kOpdQ, flat))
        return cudaErrorInvalidValue;
    if ((e = launch_wide(tc::kWDq, causal, flat, P, nsm, s)) != cudaSuccess) return e;
    ++launches;
    // 4. dK: x = V, y = dOt, w = Q (reverse)
    if (!tc_host::make_map(&P.tmX, V, p, kOpV, flat) || !tc_host::make_map(&P.tmY, dOt, q, kOpdO, flat) ||
        !tc_host::make_map(&P.tmW, Q, p, kOpQ, flat) || !tc_host::make_map(&P.tmOut, dK, p, kOpdK, flat))
        return cudaErrorInvalidValue;
    if ((e = launch_wide(tc::kWDk, causal, flat, P, nsm, s)) != cudaSuccess) return e;
    ++launches;
    // 5. dV: x = K, y = Q, w = dOt (reverse)
    if (!tc_host::make_map(&P.tmX, K, p, kOpK, flat) || !tc_host::make_map(&P.tmY, Q, p, kOpQ, flat) ||
        !tc_host::make_map(&P.tmW, dOt, q, kOpdO, flat) || !tc_host::make_map(&P.tmOut, dV, p, kOpdV, flat))
        return cudaErrorInvalidValue;
    if ((e = launch_wide(tc::kWDv, causal, flat, P, nsm, s)) != cudaSuccess) return e;
    ++launches;
    count_launches(launches);
    return cudaSuccess;
}

}  // namespace la
