// la_tc_sweep.cu -- the causal backward as one reverse sweep per head (tcgen05 / TMA, bf16, D = 128).
//
// The two-walk backward (la_tc_bwd.cu) reads Q, K, V and dO twice: its dQ walk walks each piece forward
// and leaves the piece's reverse sums for the dK / dV walk, which walks it back.  The sweep takes g_i
// from the forward (kept in the workspace) and delta_i = dO_i . O_i from the forward's output, and walks
// each head once, last chunk first, forming dQ, dK and dV of a chunk together: the gradient's
// eight tensor volumes (Q, K, V, O, dO in, dQ, dK, dV out) move once ("Transformer Based Linear Attention
// with Optimized GPU Kernel Implementation", sciencestack.ai page, TL;DR: analytical gradients and
// minimal data movement).  With dOt_i = dO_i / g_i, dt_i = (dO_i . O_i) / g_i and, within chunk c,
// U_ij = [j <= i] (dOt_i . v_j - dt_i) and P_ij = [j <= i] (1 + q_i . k_j):
//   dQ = dOt Sb^T - dt z^T + U K            Sb, z: state before the chunk (S = sum k v^T, z = sum k)
//   dK = U^T Q + V Pb^T - y                 Pb, y, e: sums over the head's later rows,
//   dV = P^T dOt + K Pb + e                   P = sum q_i dOt_i^T, y = sum dt_i q_i, e = sum dOt_i
// Walking backwards, S before chunk c is the head's total (kept by the forward's combine) minus the
// chunks at and after c; TMEM holds its negative, -S, to which each chunk adds K_c^T V_c.  z before the
// chunk comes from the forward's per-chunk column sums z_c.  P grows by Q_c^T dOt_c per chunk (TMEM);
// y and e grow by column sums that the epilogue forms on the CUDA cores.
//
// One CTA per head, heads beyond the grid looping (the walk needs no carries between CTAs, so neither
// the forward's piece sums nor a combine).  One TMA stage (Q, dO, K, V: 128 KB), the bf16 copies Sb and
// Pb and the tile U^T (32 KB each) fill shared memory.  The outputs leave by TMA from tiles whose
// operands are spent by then: dV from Pb (once dK, Pb's last reader, is done), dK from U^T and dQ from Sb
// (once dQ is done); the next chunk's O tile comes by TMA into Pb as soon as the dV store has read it, and
// after the dots dO_i . O_i Pb takes that chunk's P.  TMEM:
// -S (columns 0-127), P (128-255) and two blocks that each chunk uses in turn:
//   R0: T^T = K Q^T -> P^T (bf16, the dV operand) -> dK accumulator
//   R1: Wt^T = V dOt^T -> dV accumulator -> dQ accumulator
// Per chunk the MMA issuer runs -S += K^T V; T^T; (dOt in place) Wt^T; P += Q^T dOt; (P^T, U^T, Sb
// formed) dV = P^T dOt + K Pb into R1; (dV's MMAs done) dK = U^T Q + V Pb^T into R0; (dV read out)
// dQ = dOt Sb^T + U K into R1.  U^T is one shared-memory tile, read K-major for dK and MN-major (as U)
// for dQ.  Warp 0 TMA, warp 1 TMEM + MMA issue, warps 2-9 epilogue (TMEM lane quarter = warp % 4,
// column half = (warp - 2) / 4).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "la_internal.h"
#include "la_tc_common.cuh"
#include "la_tc_host.h"
#include "la_tc_kern.cuh"

namespace la {
namespace tc {

using namespace sm100;

namespace {

// This half's 64 columns of an fp32 TMEM block (lane = the thread's row) mapped through f(column, value),
// rounded to bf16, into row `row`, box hf of a two-box 128B-swizzled tile.
template <typename F>
__device__ __forceinline__ void tmem_half_map_to_tile(uint32_t taddr, int hf, F f, unsigned char *tile2, int row) {
    unsigned char *tile = tile2 + hf * kBox;
#pragma unroll 1
    for (int half32 = 0; half32 < 2; ++half32) {
        uint32_t v[32];
        tmem_ld32(taddr + 64 * hf + 32 * half32, v);
        tmem_wait_ld(v);
        const int c0 = 64 * hf + 32 * half32;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            uint4 w;
            uint32_t *wv = (uint32_t *)&w;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int m = 8 * g4 + 2 * q;
                wv[q] = pack_bf16(f(c0 + m, __uint_as_float(v[m])), f(c0 + m + 1, __uint_as_float(v[m + 1])));
            }
            *(uint4 *)(tile + sw128_off(row, 4 * half32 + g4)) = w;
        }
    }
}

}  // namespace

template <bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_sweep_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = 4 * TB;  // Q, dO, K, V
    constexpr uint32_t E = kEpiThreads;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stage = sm;
    unsigned char *Sb = sm + STAGE;    // bf16 S before the chunk, rows d
    unsigned char *Pb = Sb + TB;       // bf16 P over the later rows, rows d
    unsigned char *Ut = Pb + TB;       // bf16 U^T of the chunk, rows j
    float *yv = (float *)(Ut + TB);    // y over the later rows (fp32, D)
    float *ev = yv + D;                // e over the later rows
    float *zv = ev + D;                // z: after the chunk until the epilogue steps it back, then before it
    float *dtv = zv + D;               // dt_i of the chunk's rows (first the half-row dots of half 1)
    float *dpart = dtv + kC;           // the half-row dots dO_i . O_i of half 0
    uint64_t *full = (uint64_t *)(dpart + kC);
    uint64_t *empty = full + 1;
    uint64_t *bar = empty + 1;
    uint64_t *barS = bar, *barSr = bar + 1, *barT = bar + 2, *barO = bar + 3, *barW = bar + 4, *barPb = bar + 5,
             *barP = bar + 6, *barE1 = bar + 7, *barV = bar + 8, *barVr = bar + 9, *barK = bar + 10,
             *barQ = bar + 11, *barR = bar + 12;
    uint64_t *fullO = bar + 13;  // the chunk's O tile has landed in Pb
    uint32_t *tslot = (uint32_t *)(bar + 14);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(empty, 1);  // the chunk's last MMA commit: every epilogue read of the stage precedes barVr
        //                              S  Sr  T  O  W  Pb P  E1 V  Vr K  Q  R  fullO
        const uint32_t counts[14] = {1, E, 1, E, 1, E, 1, E, 1, E, 1, 1, E, 1};
        for (int k = 0; k < 14; ++k) mbar_init(&bar[k], counts[k]);
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Everything above touches only this CTA's shared memory and TMEM; every global access comes after
    // the previous kernel of the stream has completed.
    griddep_wait();
    griddep_launch_dependents();
    // The forward must have kept g and the heads' totals beside its sums, for these K and V, and no other
    // backward may have used its record: like the two walks, this backward uses it up (each backward needs
    // a forward of its own).  Every CTA claims the record with this launch's token; the first finds it
    // unused, the others find the token.
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicCAS((uint32_t *)fwd_sums_used(P), 0u, P.use_token);
        if (!state_tag_matches(P, (uint64_t)P.check_tag - 1) || !*fwd_terms_kept(P) ||
            (prev != 0u && prev != P.use_token)) {
            *abort_flag = 1;
            report(P.status, kDevState, 0x5A7Eu);
        }
    }
    __syncthreads();
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t TS = tmem, TP = tmem + 128, R0 = tmem + 256, R1 = tmem + 384;
    const long long BH = P.sl.T / P.sl.nchunk;
    const int nchunk = P.sl.nchunk;
    int o_issued = -1;  // thread 64: the step whose O load it issued and that no wait has seen land yet

    if (skip) {
        // the state this call relies on is not in the workspace: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer: each head's chunks, last first
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmdO);
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        prefetch_tmap(&P.tmO);
        int it = 0;
        bool ok = true;
        for (long long bh = blockIdx.x; bh < BH && ok; bh += gridDim.x) {
            const HeadCoord hc = head_coord<FLAT>(bh, P.H);
            for (int c = nchunk - 1; c >= 0; --c, ++it) {
                if (it > 0 && !wait_or_abort(empty, (it - 1) & 1, abort_flag, P.status, 0x501)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full, STAGE);
                for (int nb = 0; nb < NB; ++nb) {
                    tile_load<FLAT>(stage + nb * kBox, &P.tmQ, full, nb * 64, c * kC, hc);
                    tile_load<FLAT>(stage + TB + nb * kBox, &P.tmdO, full, nb * 64, c * kC, hc);
                    tile_load<FLAT>(stage + 2 * TB + nb * kBox, &P.tmK, full, nb * 64, c * kC, hc);
                    tile_load<FLAT>(stage + 3 * TB + nb * kBox, &P.tmV, full, nb * 64, c * kC, hc);
                }
                // the next chunk to be walked, into L2 (with its rows of O, which the epilogue reads itself)
                const long long nh = c > 0 ? bh : bh + gridDim.x;
                const int nc = c > 0 ? c - 1 : nchunk - 1;
                if (nh < BH) {
                    const HeadCoord hn = head_coord<FLAT>(nh, P.H);
                    for (int nb = 0; nb < NB; ++nb) {
                        tile_prefetch<FLAT>(&P.tmQ, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmdO, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmK, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmV, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmO, nb * 64, nc * kC, hn);
                    }
                }
            }
        }
        if (!ok && it > 0) mbar_wait(full, (it - 1) & 1, 50000000ull);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKK = idesc_bf16(128, 128, false, false);
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t qb = smem_u32(stage), ob = qb + TB, kb = qb + 2 * TB, vb = qb + 3 * TB;
        const uint32_t sb = smem_u32(Sb), pb = smem_u32(Pb), ub = smem_u32(Ut);
        int it = 0;
        bool ok = true;
        for (long long bh = blockIdx.x; bh < BH && ok; bh += gridDim.x) {
            for (int c = nchunk - 1; c >= 0 && ok; --c, ++it) {
                const uint32_t ph = it & 1;
                ok = wait_or_abort(full, ph, abort_flag, P.status, 0x502);
                if (ok) ok = wait_or_abort(barSr, ph, abort_flag, P.status, 0x503);  // -S read into Sb
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // -S += K^T V: -S before this chunk
                    mma_ss(TS, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024), idMM, 1u);
                mma_commit(barS);
                if (it > 0 && !(ok = wait_or_abort(barR, ph ^ 1, abort_flag, P.status, 0x504))) break;  // R0, R1 read
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // T^T = K Q^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R0, sdesc_sw128(kb + o, 16, 1024), sdesc_sw128(qb + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barT);
                ok = wait_or_abort(barO, ph, abort_flag, P.status, 0x505);  // dOt is in place of dO
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // Wt^T = V dOt^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R1, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(ob + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barW);
                ok = wait_or_abort(barPb, ph, abort_flag, P.status, 0x506);  // P read into Pb (or zero)
                if (!ok) break;
                tc_fence_after();
                const bool first = c == nchunk - 1;
#pragma unroll
                for (int k = 0; k < 8; ++k)  // P += Q^T dOt: the later rows of the next chunk to be walked
                    mma_ss(TP, sdesc_sw128(qb + 2048 * k, kBox, 1024), sdesc_sw128(ob + 2048 * k, kBox, 1024), idMM,
                           (!first || k > 0) ? 1u : 0u);
                mma_commit(barP);
                ok = wait_or_abort(barE1, ph, abort_flag, P.status, 0x507);  // P^T, U^T formed; R1 read
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dV = P^T dOt + K Pb
                    mma_ts(R1, R0 + 64 * (k >> 2) + 8 * (k & 3), sdesc_sw128(ob + 2048 * k, kBox, 1024), idKM, k > 0);
                    mma_ss(R1, sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(pb + 2048 * k, kBox, 1024), idKM, 1u);
                }
                mma_commit(barV);
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x508);  // dV's reads of P^T in R0 are done
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dK = U^T Q + V Pb^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R0, sdesc_sw128(ub + o, 16, 1024), sdesc_sw128(qb + 2048 * k, kBox, 1024), idKM, k > 0);
                    mma_ss(R0, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(pb + o, 16, 1024), idKK, 1u);
                }
                mma_commit(barK);
                ok = wait_or_abort(barVr, ph, abort_flag, P.status, 0x509);  // dV read out of R1
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dQ = dOt Sb^T + U K
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R1, sdesc_sw128(ob + o, 16, 1024), sdesc_sw128(sb + o, 16, 1024), idKK, k > 0);
                    mma_ss(R1, sdesc_sw128(ub + 2048 * k, kBox, 1024), sdesc_sw128(kb + 2048 * k, kBox, 1024), idMM, 1u);
                }
                mma_commit(barQ);
                mma_commit(empty);  // dK and dQ were the last MMAs to read the stage
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread <-> TMEM lane r (row i, j or d) and column half hf
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        unsigned char *qt = stage, *ot = stage + TB;
        // column sums: this thread's column pair (2 cp, 2 cp + 1) over rows 8 k + 2 rq + {0, 1}
        const int cp = u >> 2, rq = u & 3;
        const int cbox = cp >> 5, cc = 2 * (cp & 31);
        int it = 0;
        bool ok = true;
        for (long long bh = blockIdx.x; bh < BH && ok; bh += gridDim.x) {
            // head start: -S and z of the whole head, y = e = 0 (P = 0: the first chunk zeroes Pb)
            {
                const long long base = bh * P.slot_stride;
                if (in_range(base + (long long)D * D + D, n_htot_floats(P), P.status, 0xB00D)) {
                    const float4 *src = (const float4 *)(P.htot + base);
                    float4 v4[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) v4[q] = src[slot_f4(r, hf, q)];
                    const float *acc = (const float *)v4;
                    uint32_t neg[32];
#pragma unroll
                    for (int m = 0; m < 32; ++m) neg[m] = __float_as_uint(-acc[m]);
                    tmem_st32(TS + lo + 64 * hf, neg);
#pragma unroll
                    for (int m = 0; m < 32; ++m) neg[m] = __float_as_uint(-acc[32 + m]);
                    tmem_st32(TS + lo + 64 * hf + 32, neg);
                    if (hf == 0) zv[r] = P.htot[base + (long long)D * D + r];
                    tmem_st_wait();
                }
                (hf == 0 ? yv : ev)[r] = 0.f;
                tc_fence_before();
                mbar_arrive(barSr);
            }
            const HeadCoord hc = head_coord<FLAT>(bh, P.H);
            // g_r and component r of z_c (half 0) of chunk c, loaded one chunk ahead
            auto row_terms = [&](int c, float *g, float *z) {
                const long long row = (long long)c * kC + r;
                *g = 1.f;
                if (row < P.N) {
                    const long long gix = bh * P.N + row;
                    if (in_range(gix, n_row_floats(P), P.status, 0xB00E)) *g = P.rs_g[gix];
                }
                *z = 0.f;
                const long long zi = (bh * nchunk + c) * 256 + r;
                if (hf == 0 && in_range(zi, n_chunk_floats(P), P.status, 0xB00F)) *z = P.chunk_za[zi];
            };
            float gnext, znext;
            row_terms(nchunk - 1, &gnext, &znext);
            // thread 64: the O tile of chunk c2 of head bh2 into Pb (step it2 of the walk)
            auto load_o = [&](long long bh2, int c2, int it2) {
                const HeadCoord h2 = head_coord<FLAT>(bh2, P.H);
                mbar_arrive_expect_tx(fullO, TB);
                tile_load<FLAT>(Pb, &P.tmO, fullO, 0, c2 * kC, h2);
                tile_load<FLAT>(Pb + kBox, &P.tmO, fullO, 64, c2 * kC, h2);
                o_issued = it2;
            };
            for (int c = nchunk - 1; c >= 0; --c, ++it) {
                const uint32_t ph = it & 1;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)(P.N - row0 < kC ? P.N - row0 : kC);
                const bool rv = r < nvalid;
                const float gi = gnext, zc = znext;
                // E0: the chunk's O tile into Pb (issued with the previous chunk's dV store, but for the first)
                if (u == 0 && it == 0) load_o(bh, c, it);
                if (c > 0) row_terms(c - 1, &gnext, &znext);
                if (hf == 0) zv[r] -= zc;  // z before this chunk
                const float ig = rv ? 1.f / gi : 0.f;
                ok = wait_or_abort(full, ph, abort_flag, P.status, 0x50A);
                if (ok) ok = wait_or_abort(fullO, ph, abort_flag, P.status, 0x512);
                if (!ok) break;
                if (u == 0) o_issued = -1;
                // half-row dots dO_r . O_r (before dO is scaled)
                {
                    const unsigned char *dt2 = ot + hf * kBox, *ot2 = Pb + hf * kBox;
                    float d0 = 0.f, d1 = 0.f;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        const uint4 dv = *(const uint4 *)(dt2 + sw128_off(r, g8));
                        const uint4 ov = *(const uint4 *)(ot2 + sw128_off(r, g8));
                        const uint32_t w[4] = {dv.x, dv.y, dv.z, dv.w}, x[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            d0 = fmaf(bf16lo(w[q]), bf16lo(x[q]), d0);
                            d1 = fmaf(bf16hi(w[q]), bf16hi(x[q]), d1);
                        }
                    }
                    (hf == 0 ? dpart : dtv)[r] = d0 + d1;
                }
                epi_sync256();
                if (hf == 0) dtv[r] = rv ? (dpart[r] + dtv[r]) * ig : 0.f;
                scale_row_half(ot, r, hf, ig);  // dO row -> dOt row in place
                // Pb for this chunk in place of O: P over the later rows (the previous chunk's update), zero at
                // the head's last chunk
                if (c == nchunk - 1) {
                    unsigned char *tile = Pb + hf * kBox;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) *(uint4 *)(tile + sw128_off(r, g8)) = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    ok = wait_or_abort(barP, (it - 1) & 1, abort_flag, P.status, 0x511);
                    if (!ok) break;
                    tc_fence_after();
                    tmem_half_to_tile(TP + lo, Pb, r, hf);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barPb);
                mbar_arrive(barO);
                if (u == 0) bulk_wait_read0();  // the previous chunk's dK and dQ have left U^T and Sb
                epi_sync256();  // every dt_i is in dtv
                // E1: P^T = [i >= j, i valid] (1 + T^T) into R0 + 64 hf + [0, 32) (the columns this half has
                // read), then U^T = [i >= j, i valid] (Wt^T - dt_i) -> Ut row j: the operands of dV and dK
                ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x50C);
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t t0[32], t1[32], pk[32];
                    tmem_ld32(R0 + lo + 64 * hf, t0);
                    tmem_ld32(R0 + lo + 64 * hf + 32, t1);
                    tmem_wait_ld(t0);
                    tmem_wait_ld(t1);
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int i = 64 * hf + 2 * m;
                        const uint32_t a0 = m < 16 ? t0[2 * m] : t1[2 * m - 32];
                        const uint32_t a1 = m < 16 ? t0[2 * m + 1] : t1[2 * m - 31];
                        pk[m] = pack_bf16(i >= r && i < nvalid ? 1.f + __uint_as_float(a0) : 0.f,
                                          i + 1 >= r && i + 1 < nvalid ? 1.f + __uint_as_float(a1) : 0.f);
                    }
                    tmem_st32(R0 + lo + 64 * hf, pk);
                    tmem_st_wait();
                }
                ok = wait_or_abort(barW, ph, abort_flag, P.status, 0x50D);
                if (!ok) break;
                tc_fence_after();
                tmem_half_map_to_tile(
                    R1 + lo, hf, [&](int i, float x) { return i >= r && i < nvalid ? x - dtv[i] : 0.f; }, Ut, r);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barE1);
                // while dV and dK run: -S before the chunk -> Sb (dQ's operand; then -S may take the next
                // chunk's K^T V), and this chunk's column sums y_c = sum_i dt_i q_i, e_c = sum_i dOt_i (two
                // columns a thread), read before the stage is released (after dQ, which waits for E2)
                ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x50B);
                if (!ok) break;
                tc_fence_after();
                tmem_half_map_to_tile(TS + lo, hf, [](int, float x) { return -x; }, Sb, r);
                tc_fence_before();
                if (c > 0) mbar_arrive(barSr);  // at the head's first chunk the next head's start arrives
                float y0 = 0.f, y1 = 0.f, e0 = 0.f, e1 = 0.f;
                {
                    const unsigned char *qbx = qt + cbox * kBox, *obx = ot + cbox * kBox;
                    const uint32_t cb = (uint32_t)(cc & 7) * 2;
#pragma unroll 4
                    for (int k = 0; k < 16; ++k)
#pragma unroll
                        for (int s = 0; s < 2; ++s) {
                            const int row = 8 * k + 2 * rq + s;
                            const uint32_t off = sw128_off(row, cc >> 3) + cb;
                            const uint32_t qv = *(const uint32_t *)(qbx + off), ov2 = *(const uint32_t *)(obx + off);
                            const float dt = dtv[row];
                            y0 = fmaf(dt, bf16lo(qv), y0);
                            y1 = fmaf(dt, bf16hi(qv), y1);
                            e0 += bf16lo(ov2);
                            e1 += bf16hi(ov2);
                        }
#pragma unroll
                    for (int m = 1; m <= 2; m <<= 1) {
                        y0 += __shfl_xor_sync(0xffffffffu, y0, m);
                        y1 += __shfl_xor_sync(0xffffffffu, y1, m);
                        e0 += __shfl_xor_sync(0xffffffffu, e0, m);
                        e1 += __shfl_xor_sync(0xffffffffu, e1, m);
                    }
                }
                // E2: dV_j = [R1]_j + e, staged in Pb once dK (Pb's last reader) is done, then R1 is free for dQ
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x50E);
                if (ok) ok = wait_or_abort(barK, ph, abort_flag, P.status, 0x50F);
                if (!ok) break;
                tc_fence_after();
                tmem_half_map_to_tile(R1 + lo, hf, [&](int e, float x) { return x + ev[e]; }, Pb, r);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barVr);
                epi_sync256();  // dV staged
                if (u == 0) {
                    store_tile<FLAT>(&P.tmdV, Pb, (int)row0, hc, NB);
                    // once the store has read Pb (the older groups are done), the next chunk's O into Pb
                    const long long nbh = c > 0 ? bh : bh + gridDim.x;
                    if (nbh < BH) {
                        bulk_wait_read0();
                        load_o(nbh, c > 0 ? c - 1 : nchunk - 1, it + 1);
                    }
                }
                // E3: dK_j = [R0]_j - y into U^T, dQ_i = [R1]_i - dt_i z into Sb (both spent once dQ is done)
                ok = wait_or_abort(barQ, ph, abort_flag, P.status, 0x510);
                if (!ok) break;
                tc_fence_after();
                tmem_half_map_to_tile(R0 + lo, hf, [&](int d, float x) { return x - yv[d]; }, Ut, r);
                {
                    const float dti = dtv[r];
                    tmem_half_map_to_tile(R1 + lo, hf, [&](int d, float x) { return x - dti * zv[d]; }, Sb, r);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barR);
                epi_sync256();  // dK and dQ staged
                if (u == 0) {
                    tile_store<FLAT>(&P.tmdK, Ut, 0, (int)row0, hc);
                    tile_store<FLAT>(&P.tmdK, Ut + kBox, 64, (int)row0, hc);
                    tile_store<FLAT>(&P.tmdQ, Sb, 0, (int)row0, hc);
                    tile_store<FLAT>(&P.tmdQ, Sb + kBox, 64, (int)row0, hc);
                    bulk_commit();
                }
                if (rq == 0) {  // this chunk's rows join the later ones
                    const int col = 64 * cbox + cc;
                    yv[col] += y0;
                    yv[col + 1] += y1;
                    ev[col] += e0;
                    ev[col + 1] += e1;
                }
                epi_sync256();  // yv, ev, zv and dtv are rewritten for the next chunk
            }
        }
    }
    if (threadIdx.x == 64) {
        bulk_wait0();  // output stores complete before the CTA exits
        if (o_issued >= 0) mbar_wait(fullO, o_issued & 1, 50000000ull);  // an O load left by an abort lands
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template __global__ void tc_bwd_sweep_kernel<true>(const __grid_constant__ TcParams P);
template __global__ void tc_bwd_sweep_kernel<false>(const __grid_constant__ TcParams P);

}  // namespace tc

namespace {

constexpr size_t kTB = 2 * (size_t)tc::kBox;
// stage (Q, dO, K, V), Sb, Pb, U^T; y, e, z, dt, dots; 16 barriers, TMEM slot, abort state
constexpr size_t kSmemSweep = 4 * kTB + 3 * kTB + 5 * 128 * 4 + 18 * 8 + 32;
static_assert(kSmemSweep <= 232448, "sweep kernel exceeds the shared-memory limit");

bool set_sweep_attrs() {
    static std::atomic<int> state[kMaxDevices];
    return once_per_device(state, [] {
        const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
        return cudaFuncSetAttribute(tc::tc_bwd_sweep_kernel<true>, A, (int)kSmemSweep) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_bwd_sweep_kernel<false>, A, (int)kSmemSweep) == cudaSuccess;
    });
}

}  // namespace

bool tc_sweep_chosen(const Plan &p, int nsm) {
    if (!p.causal || p.D != 128 || nsm <= 0) return false;
    if (const char *env = getenv("LA_TC_SWEEP")) {
        if (env[0] == '0') return false;
        if (env[0] == '1') return true;
    }
    // Times fitted to measurements on one GB300 (152 SMs; B = 4, 8, 16, H = 16, N = 1024 ... 4096): the
    // sweep ~8.0 us per chunk a CTA walks (one CTA per head) + 20 us; the two walks ~10.1 us per chunk a CTA
    // walks (all SMs) + 38.5 us (two combines, two ramps).  The sweep wins once the heads fill the GPU
    // (B H >~ 100 at these lengths).
    const double nchunk = (double)(((long long)p.N + tc::kC - 1) / tc::kC);
    const double heads_per_cta = (double)((p.BH + nsm - 1) / nsm);
    const double sweep = 8.0 * heads_per_cta * nchunk + 20.0;
    const double walks = 10.1 * (double)p.BH * nchunk / (double)nsm + 38.5;
    return sweep < walks;
}

cudaError_t tc_backward_sweep(const Plan &p, tc::TcParams &P, const void *O, void *dQ, void *dK, void *dV,
                              unsigned char *ws, cudaStream_t s) {
    if (!set_sweep_attrs()) return cudaErrorInvalidValue;
    P.O = const_cast<void *>(O);
    P.dQ = dQ;
    P.dK = dK;
    P.dV = dV;
    P.rs_g = (float *)(ws + p.off_rowstats);
    P.htot = (float *)(ws + p.off_htot);
    P.check_tag = (int)tc::kTagPrefix + 1;
    // a token of this launch, for claiming the forward's record (0: unused, 1: the two walks' mark)
    static std::atomic<uint32_t> next_token{2};
    uint32_t tok = next_token.fetch_add(1);
    while (tok < 2) tok = next_token.fetch_add(1);
    P.use_token = tok;
    const int nsm = tc_host::sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    long long grid = p.BH < nsm ? p.BH : nsm;
    // Test hook (as for the other kernels): fewer CTAs, so that small problems also walk several heads
    // per CTA.
    if (const char *env = getenv("LA_TC_MAX_CTAS")) {
        const long long cap = atoll(env);
        if (cap >= 1 && cap < grid) grid = cap;
    }
    cudaError_t e = tc_host::launch_tc(P.flat ? tc::tc_bwd_sweep_kernel<true> : tc::tc_bwd_sweep_kernel<false>, (unsigned)grid,
                                       64 + tc::kEpiThreads, kSmemSweep, s, P);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace la
