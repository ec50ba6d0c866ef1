// la_tc_bwd.cu -- tcgen05 / TMA backward of the bf16 path (kernels on 128 columns; D = 32, 64 zero-extended).
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
// Launches: the per-piece K^T V sums (shared with the forward, so the backward that reuses the forward's
// workspace skips them), a combine that turns the piece slots into the carries of each piece, the dQ walk
// in chunk order (it forms g_i and delta_i from the chunk's own products and the carried state, so the
// stored O is not read -- except in its ROWS form, for the causal backward that reuses a forward given a
// backward-sized workspace: g_i from the forward and delta_i = dO_i . O_i; it also writes each piece's
// reverse sums P, y, e and, causal, the per-row g_i, dt_i), a combine of those reverse sums, and the
// dK / dV walk in reverse chunk order.  Each kernel: warp 0 TMA, warp 1 TMEM + MMA issue, warps 2-9
// epilogue (two warps per TMEM lane quarter, each owning 64 of the 128 columns).
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
// through f(column, value) to 32 packed bf16 pairs.  Callers write them back into TMEM columns this
// thread has itself read, so that no other thread's pending reads are overwritten.
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

// Row `row` of dQ over columns [64 hf, 64 hf + 64): x * ig - dt * z, rounded to bf16 into box hf of the
// staging tile (x: the 64 fp32 values of this half, as bit patterns).
__device__ __forceinline__ void regs_half_to_dq(const uint32_t (&x0)[32], const uint32_t (&x1)[32], int hf, float ig,
                                                float dt, const float *z, unsigned char *tile2, int row) {
    unsigned char *tile = tile2 + hf * kBox;
    const float *zz = z + 64 * hf;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        const uint32_t *xx = g8 < 4 ? x0 + 8 * g8 : x1 + 8 * (g8 - 4);
        uint4 w;
        uint32_t *wv = (uint32_t *)&w;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int m = 8 * g8 + 2 * q;
            wv[q] = pack_bf16(__uint_as_float(xx[2 * q]) * ig - dt * zz[m],
                              __uint_as_float(xx[2 * q + 1]) * ig - dt * zz[m + 1]);
        }
        *(uint4 *)(tile + sw128_off(row, g8)) = w;
    }
}

// The same from this half's 64 columns of an fp32 TMEM block (lane = row).
__device__ __forceinline__ void tmem_half_to_dq(uint32_t taddr, int hf, float ig, float dt, const float *z,
                                                unsigned char *tile2, int row) {
    uint32_t x0[32], x1[32];
    tmem_ld32(taddr + 64 * hf, x0);
    tmem_ld32(taddr + 64 * hf + 32, x1);
    tmem_wait_ld(x0);
    tmem_wait_ld(x1);
    regs_half_to_dq(x0, x1, hf, ig, dt, z, tile2, row);
}

// End of a dQ-walk piece: its reverse sums into its workspace slot.  Ppiece = sum_i q_i (dO_i / g_i)^T
// from TMEM (row i, this half's 64 columns); half 1 also writes component i of y and of e.
__device__ __forceinline__ void piece_rev_sums(const TcParams &P, const Piece &pc, uint32_t taddr, int i, int hf,
                                               float y, float e) {
    constexpr int D = 128;
    float *slot = P.slots_rev + slot_of(pc.h, blockIdx.x) * P.slot_stride;
    const bool sok = slot_ok(P, pc.h, blockIdx.x, 0xB007);  // the same for the whole CTA
#pragma unroll 1
    for (int half32 = 0; half32 < 2; ++half32) {
        uint32_t v[32];
        tmem_ld32(taddr + 64 * hf + 32 * half32, v);
        tmem_wait_ld(v);
        float4 *dst = (float4 *)slot;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (sok) dst[slot_f4(i, hf, 8 * half32 + q)] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                              __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    }
    if (hf == 1 && sok) {
        slot[(size_t)D * D + i] = y;
        slot[(size_t)D * D + D + i] = e;
    }
}

// q_row . z and q_row . y over box hf of a bf16 tile in one pass over the row: z fp32 (shared memory), y the
// 64 fp32 values of this half (bit patterns).
__device__ __forceinline__ float2 dot2_half(const unsigned char *tile2, int row, int hf, const float *z,
                                            const uint32_t (&y0)[32], const uint32_t (&y1)[32]) {
    const unsigned char *tile = tile2 + hf * kBox;
    const float *zz0 = z + 64 * hf;
    float az = 0.f, bz = 0.f, ay = 0.f, by = 0.f;
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        const uint4 v = *(const uint4 *)(tile + sw128_off(row, g8));
        const float *zz = zz0 + 8 * g8;
        const uint32_t *yy = g8 < 4 ? y0 + 8 * g8 : y1 + 8 * (g8 - 4);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = bf16lo(w[q]), hi = bf16hi(w[q]);
            az = fmaf(lo, zz[2 * q], az);
            bz = fmaf(hi, zz[2 * q + 1], bz);
            ay = fmaf(lo, __uint_as_float(yy[2 * q]), ay);
            by = fmaf(hi, __uint_as_float(yy[2 * q + 1]), by);
        }
    }
    return make_float2(az + bz, ay + by);
}


// The chunk walked after chunk c of piece pc when each piece is walked in reverse: c - 1 in the piece,
// else the last chunk of the piece that `pi` yields next.  False when c is the last chunk walked.
template <typename Iter>
__device__ __forceinline__ bool next_rev_chunk(const Iter &pi, const Piece &pc, int c, long long *h, int *cn) {
    if (c > pc.a) {
        *h = pc.h;
        *cn = c - 1;
        return true;
    }
    Iter pn = pi;
    pn.next();
    if (!pn.valid()) return false;
    const Piece q = pn.get();
    *h = q.h;
    *cn = q.e - 1;
    return true;
}

// g_j and dt_j of row j of chunk c of head h, from the dQ walk's row statistics (0 past the end of the
// head), and component j of that chunk's column sum y_c (hf 0) or e_c (hf 1).  Loads only: the values are
// used one chunk later.
__device__ __forceinline__ void load_chunk_stats(const TcParams &P, long long h, int c, int j, int hf, float *g,
                                                 float *dt, float *ye) {
    const long long r = (long long)c * kC + j;
    const long long x = h * P.N + r;
    const bool in = r < P.N && in_range(x, n_row_floats(P), P.status, 0xB008);
    *g = in ? P.rs_g[x] : 0.f;
    *dt = in ? P.rs_dt[x] : 0.f;
    const long long yi = (h * P.sl.nchunk + c) * 256 + hf * 128 + j;
    *ye = in_range(yi, n_chunk_floats(P), P.status, 0xB008) ? P.chunk_ye[yi] : 0.f;
}

// ----------------------------------------------------------------------------------------------------
// dQ walk (chunk order), causal.  The forward output is not recomputed: with W' = dO V^T and Y = dO Sb^T
// (Sb = bf16 state before the chunk),
//   delta_i g_i = dO_i . a + sum_j P_ij W'_ij + q_i . Y_i,      P_ij = [j <= i](1 + q_i . k_j)
//   dQ_i = (Y_i + [U' K]_i) / g_i - dt_i z,                     U'_ij = [j <= i](W'_ij - delta_i)
// Per chunk: T = Q K^T and W' (R0, R1); the epilogue forms P, r_i and sum_j P_ij W'_ij from T and W' in
// registers; Y into R0; S += K^T V (R2); the epilogue forms g_i, delta_i, dt_i and U' (bf16, in place of
// W'); X = Y + U' K in R0; dO -> dO / g in place; Ppiece += Q^T (dO / g) (R3).  The column sums the
// state and the reverse sums need (z += sum k_j, a += sum v_j, y += sum dt_i q_i, e += sum dO_i / g_i)
// are N = 16 MMAs against a tile of ones or of dt_i, into the columns of R1 that U' leaves free; the
// epilogue drains them with the dQ row.  One TMA stage (Q, dO, K, V); the next chunk's tiles are
// prefetched into L2 meanwhile, and dQ leaves through its own staging tile.
// ROWS (the backward that reuses a forward given a backward-sized workspace): g_i is the forward's, kept
// in the workspace, and delta_i = dO_i . O_i from the stored O, whose tile comes by TMA into the dQ
// staging tile between two dQ stores; T, the P sums and the q . z, q . Y dots are not needed.
// Epilogue thread u = threadIdx.x - 64: row i = 32 (warp % 4) + lane, column half hf = u / 128.
// ----------------------------------------------------------------------------------------------------
template <bool FLAT, bool ROWS>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dq_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = 4 * TB;  // Q, dO, K, V
    constexpr uint32_t E = kEpiThreads;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stage = sm;
    unsigned char *Sb = sm + STAGE;
    unsigned char *dqt = Sb + TB;        // dQ staging tile
    unsigned char *ones = dqt + TB;      // 8 rows x 128 B of bf16 1.0 (N = 16 operand, rows repeated)
    unsigned char *dtt = ones + 1024;    // dt_i of the chunk's rows, as an N = 16 operand (split_tile_put)
    float *zc = (float *)(dtt + 2048);   // z before the chunk (fp32, D)
    float *ac = zc + D;                  // a before the chunk
    float *xg = ac + D;                  // [2][128] row partials of g (per column half)
    float *xd = xg + 2 * kC;             // [2][128] row partials of delta g
    uint64_t *full = (uint64_t *)(xd + 2 * kC);
    uint64_t *empty = full + 1;
    uint64_t *bar = empty + 1;
    uint64_t *barT = bar, *barTr = bar + 1, *barSb = bar + 2, *barY = bar + 3, *barU = bar + 4, *barDt = bar + 5,
             *barX = bar + 6, *barR = bar + 7, *barPPf = bar + 8, *barC = bar + 9;
    uint64_t *fullO = bar + 10;  // ROWS: the chunk's O tile has landed in the staging tile
    uint32_t *tslot = (uint32_t *)(bar + 11);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(empty, 1);  // the chunk's last MMA commit: every epilogue read of the stage precedes barDt
        const uint32_t counts[11] = {1, E, E, 1, E, E, 1, E, E, 1, 1};
        for (int k = 0; k < 11; ++k) mbar_init(&bar[k], counts[k]);
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    for (int k = threadIdx.x; k < 256; k += blockDim.x) ((uint32_t *)ones)[k] = 0x3F803F80u;
    for (int k = threadIdx.x; k < 512; k += blockDim.x) ((uint32_t *)dtt)[k] = 0u;
    fence_proxy_async_smem();
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
    if (P.check_tag) {  // the forward's per-piece sums (ROWS: and g) are reused: in the workspace, unused?
        if (threadIdx.x == 0 && (!state_tag_matches(P, (uint64_t)P.check_tag - 1) || *fwd_sums_used(P) ||
                                 (ROWS && !*fwd_terms_kept(P)))) {
            *abort_flag = 1;
            report(P.status, kDevState, 0x5A7Eu);
        }
        __syncthreads();
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *bwd_skip(P) = *abort_flag ? 1u : 0u;  // for the dK / dV walk
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t R0 = tmem, R1 = tmem + 128, R2 = tmem + 256, R3 = tmem + 384;
    int o_issued = -1;  // ROWS, thread 64: the step whose O load it issued and that no wait has seen land
    // column sums of the chunk (N = 16 each; column 0 of each holds the sum, column 1 of cY the dt remainder),
    // in the R1 columns that U' (R1 + [0, 32) and R1 + [64, 96)) leaves free
    const uint32_t cY = R1 + 96, cE = R1 + 112;

    if (skip) {
        // the state this call relies on is not in the workspace: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmdO);
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        const long long hi = slice_lo(P.sl, blockIdx.x + 1);
        {  // the first piece's carry slot
            PieceIter p0(P.sl, blockIdx.x);
            if (p0.valid() && slot_ok(P, p0.get().h, blockIdx.x, 0xB0F0))
                bulk_prefetch_l2(P.slots + slot_of(p0.get().h, blockIdx.x) * P.slot_stride,
                                 (uint32_t)(kSlotF4 * sizeof(float4)));
        }
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            const HeadCoord hc = head_coord<FLAT>(pc.h, P.H);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                prefetch_next_carry(pi, pc.e - 1 - c, pc.e - pc.a, P.slots, P.slot_stride, blockIdx.x, n_slot_floats(P), P.status);
                if (it > 0 && !wait_or_abort(empty, (it - 1) & 1, abort_flag, P.status, 0x301)) {
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
                const long long nx = pc.h * P.sl.nchunk + c + 1;  // the slice's next chunk, into L2
                if (nx < hi) {
                    const int nh = (int)(nx / P.sl.nchunk), nrow = (int)(nx % P.sl.nchunk) * kC;
                    const HeadCoord hn = head_coord<FLAT>(nh, P.H);
                    for (int nb = 0; nb < NB; ++nb) if (nb == 0 || P.nbox > 1) {
                        tile_prefetch<FLAT>(&P.tmQ, nb * 64, nrow, hn);
                        tile_prefetch<FLAT>(&P.tmdO, nb * 64, nrow, hn);
                        tile_prefetch<FLAT>(&P.tmK, nb * 64, nrow, hn);
                        tile_prefetch<FLAT>(&P.tmV, nb * 64, nrow, hn);
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
        const uint32_t idZ = idesc_bf16(128, 16, true, false);
        const uint32_t sb = smem_u32(Sb), on = smem_u32(ones), dtb = smem_u32(dtt);
        const uint32_t qb = smem_u32(stage), ob = qb + TB, kb = qb + 2 * TB, vb = qb + 3 * TB;
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            for (int c = pc.a; c < pc.e && ok; ++c, ++it) {
                const uint32_t ph = it & 1;
                ok = wait_or_abort(full, ph, abort_flag, P.status, 0x304);
                if (ok && it > 0) ok = wait_or_abort(barR, ph ^ 1, abort_flag, P.status, 0x307);  // R0, R1 drained
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // T = Q K^T (not with ROWS) ; W' = dO V^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    if (!ROWS) mma_ss(R0, sdesc_sw128(qb + o, 16, 1024), sdesc_sw128(kb + o, 16, 1024), idKK, k > 0);
                    mma_ss(R1, sdesc_sw128(ob + o, 16, 1024), sdesc_sw128(vb + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barT);
                if (!ROWS) ok = wait_or_abort(barTr, ph, abort_flag, P.status, 0x305);  // T has been read out of R0
                if (!ok) break;
                ok = wait_or_abort(barSb, ph, abort_flag, P.status, 0x306);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // Y = dO Sb^T
                    mma_ss(R0, sdesc_sw128(ob + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                mma_commit(barY);
                if (c + 1 < pc.e) {  // S += K^T V, once the epilogue has copied S into Sb (barSb above)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ss(R2, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024),
                               idMM, 1u);
                }
                ok = wait_or_abort(barU, ph, abort_flag, P.status, 0x308);  // U' written, W' no longer needed
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // X = Y + U' K
                    mma_ts(R0, R1 + 64 * (k >> 2) + 8 * (k & 3), sdesc_sw128(kb + 2048 * k, kBox, 1024), idKM, 1u);
                mma_commit(barX);
                ok = wait_or_abort(barDt, ph, abort_flag, P.status, 0x309);  // dO / g in place, dt_i in dtt
                if (!ok) break;
                if (c == pc.a && pno > 0) ok = wait_or_abort(barPPf, (pno - 1) & 1, abort_flag, P.status, 0x303);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // Ppiece += Q^T (dO / g) ; y_c = Q^T dt ; e_c = (dO / g)^T 1
                    const uint64_t qa = sdesc_sw128(qb + 2048 * k, kBox, 1024);
                    const uint64_t oa = sdesc_sw128(ob + 2048 * k, kBox, 1024);
                    mma_ss(R3, qa, oa, idMM, (c > pc.a || k > 0) ? 1u : 0u);
                    mma_ss(cY, qa, sdesc_sw128(dtb + (k >> 2) * 1024 + 32 * (k & 3), 16, 0), idZ, k > 0);
                    mma_ss(cE, oa, sdesc_sw128(on + 32 * (k & 3), 16, 0), idZ, k > 0);
                }
                mma_commit(barC);
                mma_commit(empty);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        unsigned char *qt = stage, *ot = stage + TB;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // forward state carried into the piece, from the head's earlier pieces (the previous
            // piece's MMAs on R2 are complete: its last barX has been waited for)
            if (pc.a == 0)  // the head's first piece: nothing before it
                zero_carry_half(i, hf, R2 + lo, Sb, zc, ac, true);
            else if (slot_ok(P, pc.h, blockIdx.x, 0xB003))
                load_carry_half(P.slots, P.slot_stride, pc.h, blockIdx.x, i, hf, R2 + lo, 0u, 0u,
                                Sb, zc, ac, true, false);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barSb);
            float yacc = 0.f, eacc = 0.f;  // half 1: y_i and e_i of the piece (row i = component d)
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const uint32_t ph = it & 1;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                // this chunk's z_c[i] (half 0) or a_c[i] (half 1), from the sums kernel; used at the chunk's end
                const long long zi = ((long long)pc.h * P.sl.nchunk + c) * 256 + hf * 128 + i;
                const float zav = in_range(zi, n_chunk_floats(P), P.status, 0xB009) ? P.chunk_za[zi] : 0.f;
                float gi, delta;
                if (ROWS) {
                    // g_i from the forward; delta_i = dO_i . O_i, O's tile in the staging tile (the first
                    // chunk's load issued here, the others' after the previous dQ store)
                    const HeadCoord hcur = head_coord<FLAT>(pc.h, P.H);
                    if (u == 0 && it == 0) {
                        mbar_arrive_expect_tx(fullO, TB);
                        tile_load<FLAT>(dqt, &P.tmO, fullO, 0, (int)row0, hcur);
                        tile_load<FLAT>(dqt + kBox, &P.tmO, fullO, 64, (int)row0, hcur);
                        o_issued = it;
                    }
                    gi = 1.f;
                    if (i < nvalid) {
                        const long long x = (long long)pc.h * P.N + row0 + i;
                        if (in_range(x, n_row_floats(P), P.status, 0xB00A)) gi = P.rs_g[x];
                    }
                    ok = wait_or_abort(full, ph, abort_flag, P.status, 0x310);  // dO has landed
                    if (ok) ok = wait_or_abort(fullO, ph, abort_flag, P.status, 0x30F);
                    if (!ok) break;
                    if (u == 0) o_issued = -1;
                    {
                        const unsigned char *dt2 = ot + hf * kBox, *ot2 = dqt + hf * kBox;
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int g8 = 0; g8 < 8; ++g8) {
                            const uint4 dv = *(const uint4 *)(dt2 + sw128_off(i, g8));
                            const uint4 ov = *(const uint4 *)(ot2 + sw128_off(i, g8));
                            const uint32_t w[4] = {dv.x, dv.y, dv.z, dv.w}, x[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                d0 = fmaf(bf16lo(w[q]), bf16lo(x[q]), d0);
                                d1 = fmaf(bf16hi(w[q]), bf16hi(x[q]), d1);
                            }
                        }
                        xd[hf * kC + i] = d0 + d1;
                    }
                    tc_fence_before();
                    epi_sync256();
                    tc_fence_after();
                    delta = xd[i] + xd[kC + i];
                    // W' (for U') and Y (the last reader of dO before it is scaled) are complete
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x30B);
                    if (ok) ok = wait_or_abort(barY, ph, abort_flag, P.status, 0x30C);
                    if (!ok) break;
                    tc_fence_after();
                } else {
                float gpart = 0.f, dpart = 0.f;  // partial g_i and partial delta_i g_i over this half
                {  // P, r_i and sum_j P_ij W'_ij over this half's columns j (fp32)
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
                dpart += dot_half(ot, i, hf, ac);  // dO_i . a, a before the chunk
                // q_i . z and q_i . Y_i over this half's d (Y = dO Sb^T), one pass over the Q row
                ok = wait_or_abort(barY, ph, abort_flag, P.status, 0x30C);
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t y0[32], y1[32];
                    tmem_ld32(R0 + lo + 64 * hf, y0);
                    tmem_ld32(R0 + lo + 64 * hf + 32, y1);
                    tmem_wait_ld(y0);
                    tmem_wait_ld(y1);
                    const float2 qq = dot2_half(qt, i, hf, zc, y0, y1);
                    gpart += qq.x;
                    dpart += qq.y;
                }
                xg[hf * kC + i] = gpart;
                xd[hf * kC + i] = dpart;
                if (u == 0) bulk_wait_read0();  // the previous chunk's dQ has left the staging tile
                tc_fence_before();
                epi_sync256();
                tc_fence_after();
                gi = (float)row0 + xg[i] + xg[kC + i];
                delta = (xd[i] + xd[kC + i]) * (1.f / gi);
                }
                const float ig = 1.f / gi;
                const float dt = delta * ig;
                if (hf == 0 && i < nvalid) {
                    const long long x = (long long)pc.h * P.N + row0 + i;
                    if (in_range(x, n_row_floats(P), P.status, 0xB00A)) {
                        P.rs_g[x] = gi;
                        P.rs_dt[x] = dt;
                    }
                }
                {  // U' = [j <= i](W' - delta), bf16, over the R1 columns this half has read: R1 + 64 hf + [0, 32)
                    uint32_t pk[32];
                    tmem_half_to_bf16(R1 + lo, hf, [&](int j, float w) { return j <= i ? w - delta : 0.f; }, pk);
                    tmem_st32(R1 + lo + 64 * hf, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barU);
                }
                scale_row_half(ot, i, hf, ig);  // dO -> dO / g in place (W' and Y, its unscaled readers, are done)
                if (hf == 0) split_tile_put(dtt, i, dt);
                fence_proxy_async_smem();
                mbar_arrive(barDt);
                // dQ_i = X_i / g_i - dt_i z (X = Y + U' K), and the chunk's column sums
                ok = wait_or_abort(barX, ph, abort_flag, P.status, 0x30E);  // X = Y + U' K
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_dq(R0 + lo, hf, ig, dt, zc, dqt, i);
                fence_proxy_async_smem();
                epi_sync256();  // dQ rows are staged, every read of zc for this chunk is done
                if (u == 0) {
                    store_tile<FLAT>(&P.tmdQ, dqt, (int)row0, head_coord<FLAT>(pc.h, P.H), P.nbox);
                    // ROWS: once the store has read the staging tile, the next chunk's O tile into it
                    const long long nx = pc.h * P.sl.nchunk + c + 1;
                    if (ROWS && nx < slice_lo(P.sl, blockIdx.x + 1)) {
                        bulk_wait_read0();
                        mbar_arrive_expect_tx(fullO, TB);
                        const HeadCoord hn = head_coord<FLAT>(nx / P.sl.nchunk, P.H);
                        const int nrow = (int)(nx % P.sl.nchunk) * kC;
                        tile_load<FLAT>(dqt, &P.tmO, fullO, 0, nrow, hn);
                        tile_load<FLAT>(dqt + kBox, &P.tmO, fullO, 64, nrow, hn);
                        o_issued = it + 1;
                    }
                }
                if (c + 1 < pc.e) {
                    tmem_half_to_tile(R2 + lo, Sb, i, hf);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(barSb);
                }
                (hf == 0 ? zc : ac)[i] += zav;  // z and a after this chunk
                ok = wait_or_abort(barC, ph, abort_flag, P.status, 0x30D);  // Ppiece, y_c, e_c
                if (!ok) break;
                tc_fence_after();
                uint32_t s0, s1, s2, s3;
                if (hf == 1) {  // y_c, e_c (component i): into the piece sums, and kept per chunk for the dK / dV walk
                    tmem_ld2(cY + lo, s0, s1);
                    tmem_ld2(cE + lo, s2, s3);
                    tmem_wait_ld(s0, s1);
                    tmem_wait_ld(s2, s3);
                    const float yv = __uint_as_float(s0) + __uint_as_float(s1), ev = __uint_as_float(s2);
                    const long long ci = ((long long)pc.h * P.sl.nchunk + c) * 256;
                    if (in_range(ci + i, n_chunk_floats(P), P.status, 0xB00B) &&
                        in_range(ci + 128 + i, n_chunk_floats(P), P.status, 0xB00B)) {
                        P.chunk_ye[ci + i] = yv;
                        P.chunk_ye[ci + 128 + i] = ev;
                    }
                    yacc += yv;
                    eacc += ev;
                }
                tc_fence_before();
                mbar_arrive(barR);
                epi_sync256();
            }
            if (!ok) break;
            piece_rev_sums(P, pc, R3 + lo, i, hf, yacc, eacc);  // Ppiece is complete (last barC)
            tc_fence_before();
            mbar_arrive(barPPf);
        }
    }
    if (threadIdx.x == 64) {
        bulk_wait0();  // output stores complete before the CTA exits
        if (ROWS && o_issued >= 0) mbar_wait(fullO, o_issued & 1, 50000000ull);  // an O load left by an abort lands
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------------------------------
// dQ walk, non-causal.  Every row sees the head's totals S, z, a (all its pieces' slots), so the chunks
// of a piece are independent apart from the piece sums Ppiece = sum_i q_i (dO_i / g_i)^T, y and e:
//   g_i = N + q_i . z,   delta_i g_i = dO_i . a + q_i . Y_i,   dQ_i = Y_i / g_i - dt_i z,   Y = dO Sb^T.
// Two TMA stages of (Q, dO).  Y alternates between TMEM blocks R0 and R1, so that the MMA of the next
// chunk runs while the epilogue works on this one; Ppiece (R3) and the column sums y, e (N = 16 MMAs
// into R2) are issued one chunk behind, once the epilogue has rewritten dO as dO / g in place; dQ leaves
// through its own staging tile.
// ----------------------------------------------------------------------------------------------------
template <bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dq_nc_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64, NST = 2;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = 2 * TB;  // Q, dO
    constexpr uint32_t E = kEpiThreads;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Sb = sm + NST * STAGE;
    unsigned char *dqt = Sb + TB;      // dQ staging tile
    unsigned char *ones = dqt + TB;    // 8 rows x 128 B of bf16 1.0
    unsigned char *dtt = ones + 1024;  // [2 chunk parities] dt_i as an N = 16 operand (split_tile_put)
    float *zc = (float *)(dtt + 4096); // the head's z
    float *ac = zc + D;                // the head's a
    float *xg = ac + D;                // [2][128] row partials of g
    float *xd = xg + 2 * kC;           // [2][128] row partials of delta g
    uint64_t *full = (uint64_t *)(xd + 2 * kC);
    uint64_t *empty = full + NST;
    uint64_t *barY = empty + NST;  // [2]: Y of the chunk is in R0 / R1
    uint64_t *barYf = barY + 2;    // [2]: the epilogue has read Y out of R0 / R1
    uint64_t *barDt = barYf + 2, *barX = barDt + 1, *barSb = barDt + 2, *barPP = barDt + 3, *barPPf = barDt + 4;
    uint32_t *tslot = (uint32_t *)(barDt + 5);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // the Ppiece MMA commit: every epilogue read of the stage precedes barDt
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&barY[b], 1);
            mbar_init(&barYf[b], E);
        }
        mbar_init(barDt, E);
        mbar_init(barX, 1);
        mbar_init(barSb, E);
        mbar_init(barPP, 1);
        mbar_init(barPPf, E);
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    for (int k = threadIdx.x; k < 256; k += blockDim.x) ((uint32_t *)ones)[k] = 0x3F803F80u;
    for (int k = threadIdx.x; k < 1024; k += blockDim.x) ((uint32_t *)dtt)[k] = 0u;
    fence_proxy_async_smem();
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
    if (P.check_tag) {  // the forward's per-piece sums are reused: are they in the workspace (and unused)?
        if (threadIdx.x == 0 && (!state_tag_matches(P, (uint64_t)P.check_tag - 1) || *fwd_sums_used(P))) {
            *abort_flag = 1;
            report(P.status, kDevState, 0x5A7Eu);
        }
        __syncthreads();
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *bwd_skip(P) = *abort_flag ? 1u : 0u;  // for the dK / dV walk
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t R2 = tmem + 256, R3 = tmem + 384;
    const uint32_t cY = R2, cE = R2 + 16;  // piece sums y (columns 0, 1: two parts) and e (column 0)

    if (skip) {
        // the state this call relies on is not in the workspace: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmdO);
        {  // the first piece's carry slot
            PieceIter p0(P.sl, blockIdx.x);
            if (p0.valid() && slot_ok(P, p0.get().h, blockIdx.x, 0xB0F0))
                bulk_prefetch_l2(P.slots + slot_of(p0.get().h, blockIdx.x) * P.slot_stride,
                                 (uint32_t)(kSlotF4 * sizeof(float4)));
        }
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            const HeadCoord hc = head_coord<FLAT>(pc.h, P.H);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                prefetch_next_carry(pi, pc.e - 1 - c, pc.e - pc.a, P.slots, P.slot_stride, blockIdx.x, n_slot_floats(P), P.status);
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x321)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tile_load<FLAT>(st + nb * kBox, &P.tmQ, &full[s], nb * 64, c * kC, hc);
                    tile_load<FLAT>(st + TB + nb * kBox, &P.tmdO, &full[s], nb * 64, c * kC, hc);
                }
                // the chunk that will next refill this stage, into L2 (within the slice)
                const long long nx = pc.h * P.sl.nchunk + c + NST;
                if (nx < slice_lo(P.sl, blockIdx.x + 1)) {
                    const int nrow = (int)(nx % P.sl.nchunk) * kC;
                    const HeadCoord hn = head_coord<FLAT>(nx / P.sl.nchunk, P.H);
                    for (int nb = 0; nb < NB; ++nb) if (nb == 0 || P.nbox > 1) {
                        tile_prefetch<FLAT>(&P.tmQ, nb * 64, nrow, hn);
                        tile_prefetch<FLAT>(&P.tmdO, nb * 64, nrow, hn);
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
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t idZ = idesc_bf16(128, 16, true, false);
        const uint32_t sb = smem_u32(Sb), on = smem_u32(ones), dtb = smem_u32(dtt);
        // Ppiece += Q^T (dO / g), y += Q^T dt, e += (dO / g)^T 1 for flat chunk index itp
        auto ppiece = [&](int itp, bool first) -> bool {
            if (!wait_or_abort(barDt, itp & 1, abort_flag, P.status, 0x322)) return false;
            tc_fence_after();
            const uint32_t qb = smem_u32(stages + (itp % NST) * STAGE), ob = qb + TB;
            const uint32_t db = dtb + (itp & 1) * 2048;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t acc = (!first || k > 0) ? 1u : 0u;
                const uint64_t qa = sdesc_sw128(qb + 2048 * k, kBox, 1024);
                const uint64_t oa = sdesc_sw128(ob + 2048 * k, kBox, 1024);
                mma_ss(R3, qa, oa, idMM, acc);
                mma_ss(cY, qa, sdesc_sw128(db + (k >> 2) * 1024 + 32 * (k & 3), 16, 0), idZ, acc);
                mma_ss(cE, oa, sdesc_sw128(on + 32 * (k & 3), 16, 0), idZ, acc);
            }
            mma_commit(barX);
            mma_commit(&empty[itp % NST]);
            return true;
        };
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!wait_or_abort(barSb, pno & 1, abort_flag, P.status, 0x323)) break;
            if (pno > 0 && !wait_or_abort(barPPf, (pno - 1) & 1, abort_flag, P.status, 0x324)) break;
            for (int c = pc.a; c < pc.e && ok; ++c, ++it) {
                const int s = it % NST, b = it & 1;
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x325);
                if (ok && it >= 2) ok = wait_or_abort(&barYf[b], ((it >> 1) - 1) & 1, abort_flag, P.status, 0x326);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ob = smem_u32(stages + s * STAGE) + TB;
#pragma unroll
                for (int k = 0; k < 8; ++k)  // Y = dO Sb^T
                    mma_ss(tmem + 128 * b, sdesc_sw128(ob + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                mma_commit(&barY[b]);
                if (c > pc.a) ok = ppiece(it - 1, c - 1 == pc.a);
            }
            if (!ok || !ppiece(it - 1, pc.e - 1 == pc.a)) break;
            mma_commit(barPP);
        }
    } else if (warp >= 2) {
        // ---- epilogue
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (slot_ok(P, pc.h, blockIdx.x, 0xB003))
                load_carry_half(P.slots, P.slot_stride, pc.h, blockIdx.x, i, hf, 0u, 0u, 0u, Sb, zc,
                                ac, false, false);
            fence_proxy_async_smem();
            epi_sync256();
            mbar_arrive(barSb);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST, b = it & 1;
                unsigned char *qt = stages + s * STAGE, *ot = qt + TB;
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x327);
                if (!ok) break;
                const float dpart = dot_half(ot, i, hf, ac);  // dO_i . a
                ok = wait_or_abort(&barY[b], (it >> 1) & 1, abort_flag, P.status, 0x328);
                if (!ok) break;
                tc_fence_after();
                uint32_t y0[32], y1[32];
                tmem_ld32(tmem + 128 * b + lo + 64 * hf, y0);
                tmem_ld32(tmem + 128 * b + lo + 64 * hf + 32, y1);
                tmem_wait_ld(y0);
                tmem_wait_ld(y1);
                tc_fence_before();
                mbar_arrive(&barYf[b]);
                const float2 qq = dot2_half(qt, i, hf, zc, y0, y1);  // q_i . z, q_i . Y_i
                xg[hf * kC + i] = qq.x;
                xd[hf * kC + i] = dpart + qq.y;
                if (u == 0) bulk_wait_read0();  // the previous chunk's dQ has left the staging tile
                epi_sync256();
                const float gi = (float)P.N + xg[i] + xg[kC + i];
                const float ig = 1.f / gi;
                const float dt = (xd[i] + xd[kC + i]) * ig * ig;
                regs_half_to_dq(y0, y1, hf, ig, dt, zc, dqt, i);
                scale_row_half(ot, i, hf, ig);  // dO -> dO / g in place (Y, its unscaled reader, is done)
                if (hf == 0) split_tile_put(dtt + (it & 1) * 2048, i, dt);
                fence_proxy_async_smem();
                if (it > 0) {  // keeps barDt one phase ahead of the MMA issuer at most
                    ok = wait_or_abort(barX, (it - 1) & 1, abort_flag, P.status, 0x329);
                    if (!ok) break;
                }
                mbar_arrive(barDt);
                epi_sync256();  // dQ of every row is staged
                if (u == 0) store_tile<FLAT>(&P.tmdQ, dqt, c * kC, head_coord<FLAT>(pc.h, P.H), P.nbox);
            }
            if (!ok) break;
            ok = wait_or_abort(barPP, pno & 1, abort_flag, P.status, 0x32A);
            if (!ok) break;
            tc_fence_after();
            uint32_t s0, s1, s2, s3;
            tmem_ld2(cY + lo, s0, s1);
            tmem_ld2(cE + lo, s2, s3);
            tmem_wait_ld(s0, s1);
            tmem_wait_ld(s2, s3);
            piece_rev_sums(P, pc, R3 + lo, i, hf, __uint_as_float(s0) + __uint_as_float(s1), __uint_as_float(s2));
            tc_fence_before();
            mbar_arrive(barPPf);
            epi_sync256();  // zc, ac and Sb are rewritten by the next piece
        }
    }
    if (threadIdx.x == 64) bulk_wait0();  // output stores complete before the CTA exits
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------------------------------------
// dK / dV walk (reverse chunk order: the slice's pieces last first, each piece's chunks last first),
// causal, with lane = key row j of the chunk.  Per chunk:
//   the epilogue first rewrites dO as dOt = dO / g in place (g_i, dt_i and the chunk's column sums
//   y_c, e_c come from the dQ walk and are loaded one chunk ahead); T^T = K Q^T (R0) and
//   Wt^T = V dOt^T (R1); P^T = [i >= j](1 + T^T) as soon as T^T is in, and U^T = [i >= j](Wt^T - dt_i)
//   once Wt^T is, both bf16 into R0 (per 64 rows i: P^T in the first 32 columns of the 64, U^T in the
//   next 32); dV = P^T dOt + K Pb (R2, then + e) while U^T is formed, then dK = U^T Q + V Pb^T (R1,
//   over the consumed Wt^T, then - y); P += Q^T dOt (R3: the sum over later rows, for the earlier
//   chunks); then y += y_c, e += e_c.
// Pb is the bf16 copy of P.  Wt^T takes dOt rounded to bf16, so U^T = Wt^T - dt carries ~2^-9 of
// |dO . v| / g where the two terms cancel (a single row: dK is then 0 by the definition); the dQ walk
// forms W' from dO itself.  dK and dV leave through staging tiles of their own, so the stage is released
// as soon as dK, the last MMA reading it, is done.  One TMA stage (Q, dO, K, V); the next chunk's tiles
// are prefetched into L2 meanwhile.
// ----------------------------------------------------------------------------------------------------
template <bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dkdv_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = 4 * TB;  // Q, dO, K, V
    constexpr uint32_t E = kEpiThreads;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stage = sm;
    unsigned char *Pb = sm + STAGE;
    unsigned char *dvt = Pb + TB;     // dV staging tile
    unsigned char *dkt = dvt + TB;    // dK staging tile
    float *yc = (float *)(dkt + TB);  // y over the later rows (fp32, D)
    float *ec = yc + D;               // e over the later rows
    float *sDt = ec + D;              // dt_i of the chunk's rows
    uint64_t *full = (uint64_t *)(sDt + kC);
    uint64_t *empty = full + 1;
    uint64_t *bar = empty + 1;
    uint64_t *barO = bar, *barT1 = bar + 1, *barT2 = bar + 2, *barP1 = bar + 3, *barP2 = bar + 4, *barPb = bar + 5,
             *barK = bar + 6, *barV = bar + 7, *barR = bar + 8;
    uint32_t *tslot = (uint32_t *)(bar + 9);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(empty, 1);  // the chunk's last MMA commit (every epilogue read of the stage precedes barO)
        const uint32_t counts[9] = {E, 1, 1, E, E, E, 1, 1, E};
        for (int k = 0; k < 9; ++k) mbar_init(&bar[k], counts[k]);
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
    if (P.check_tag) {  // the forward's per-piece sums are reused: are they in the workspace, and did the
                        // dQ walk before this kernel take them?
        if (threadIdx.x == 0 && (!state_tag_matches(P, (uint64_t)P.check_tag - 1) || *bwd_skip(P))) {
            *abort_flag = 1;
            report(P.status, kDevState, 0x5A7Eu);
        }
        __syncthreads();
    }
    // this backward's reverse sums now fill the slots of the forward's sums (the dQ walk, which checked
    // them, is complete)
    if (blockIdx.x == 0 && threadIdx.x == 0) *fwd_sums_used(P) = 1u;
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t R0 = tmem, R1 = tmem + 128, R2 = tmem + 256, R3 = tmem + 384;

    if (skip) {
        // the state this call relies on is not in the workspace: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer (chunks of each piece in reverse order)
        prefetch_tmap(&P.tmQ);
        prefetch_tmap(&P.tmdO);
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        {  // the first piece's carry slot
            RevPieceIter p0(P.sl, blockIdx.x);
            if (p0.valid() && slot_ok(P, p0.get().h, blockIdx.x, 0xB0F0))
                bulk_prefetch_l2(P.slots_rev + slot_of(p0.get().h, blockIdx.x) * P.slot_stride,
                                 (uint32_t)(kSlotF4 * sizeof(float4)));
        }
        int it = 0;
        bool ok = true;
        for (RevPieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            const HeadCoord hc = head_coord<FLAT>(pc.h, P.H);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                prefetch_next_carry(pi, c - pc.a, pc.e - pc.a, P.slots_rev, P.slot_stride, blockIdx.x, n_slot_floats(P), P.status);
                if (it > 0 && !wait_or_abort(empty, (it - 1) & 1, abort_flag, P.status, 0x401)) {
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
                long long nh;
                int nc;
                if (next_rev_chunk(pi, pc, c, &nh, &nc)) {  // the next chunk to be walked, into L2
                    const HeadCoord hn = head_coord<FLAT>(nh, P.H);
                    for (int nb = 0; nb < NB; ++nb) if (nb == 0 || P.nbox > 1) {
                        tile_prefetch<FLAT>(&P.tmQ, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmdO, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmK, nb * 64, nc * kC, hn);
                        tile_prefetch<FLAT>(&P.tmV, nb * 64, nc * kC, hn);
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
        const uint32_t pb = smem_u32(Pb);
        const uint32_t qb = smem_u32(stage), ob = qb + TB, kb = qb + 2 * TB, vb = qb + 3 * TB;
        int it = 0;
        bool ok = true;
        for (RevPieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            for (int c = pc.e - 1; c >= pc.a && ok; --c, ++it) {
                const uint32_t ph = it & 1;
                ok = wait_or_abort(full, ph, abort_flag, P.status, 0x403);
                if (ok && it > 0) ok = wait_or_abort(barR, ph ^ 1, abort_flag, P.status, 0x402);  // TMEM drained
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // T^T = K Q^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R0, sdesc_sw128(kb + o, 16, 1024), sdesc_sw128(qb + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barT1);
                ok = wait_or_abort(barO, ph, abort_flag, P.status, 0x404);  // dOt is in place of dO
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // Wt^T = V dOt^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R1, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(ob + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barT2);
                if (c > pc.a) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)  // P += Q^T dOt
                        mma_ss(R3, sdesc_sw128(qb + 2048 * k, kBox, 1024), sdesc_sw128(ob + 2048 * k, kBox, 1024),
                               idMM, 1u);
                }
                ok = wait_or_abort(barP1, ph, abort_flag, P.status, 0x405);  // P^T is in R0
                if (ok) ok = wait_or_abort(barPb, ph, abort_flag, P.status, 0x406);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dV = P^T dOt + K Pb
                    mma_ts(R2, R0 + 64 * (k >> 2) + 8 * (k & 3), sdesc_sw128(ob + 2048 * k, kBox, 1024), idKM, k > 0);
                    mma_ss(R2, sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(pb + 2048 * k, kBox, 1024), idKM, 1u);
                }
                mma_commit(barV);
                ok = wait_or_abort(barP2, ph, abort_flag, P.status, 0x407);  // U^T is in R0, Wt^T has been read
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dK = U^T Q + V Pb^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ts(R1, R0 + 64 * (k >> 2) + 32 + 8 * (k & 3), sdesc_sw128(qb + 2048 * k, kBox, 1024), idKM, k > 0);
                    mma_ss(R1, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(pb + o, 16, 1024), idKK, 1u);
                }
                mma_commit(barK);
                mma_commit(empty);  // dK was the last MMA to read the stage
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread <-> key row j (TMEM lane) and column half hf
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int j = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        unsigned char *ot = stage + TB;
        // g_j, dt_j and component j of y_c (half 0) or e_c (half 1) for the next chunk to be walked
        float ng = 0.f, ndt = 0.f, nye = 0.f;
        {
            RevPieceIter p0(P.sl, blockIdx.x);
            if (p0.valid()) {
                const Piece q = p0.get();
                load_chunk_stats(P, q.h, q.e - 1, j, hf, &ng, &ndt, &nye);
            }
        }
        int it = 0;
        bool ok = true;
        for (RevPieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // carried reverse sums (the later pieces of the head); the previous piece's MMAs on R3 and Pb are
            // complete (its last barV).  The slice's pieces are walked last first, so that where a slice
            // straddles two heads the piece change leads into the earlier head's last piece, whose carry is
            // zero and needs no load.
            if (pc.e == P.sl.nchunk)
                zero_carry_half(j, hf, R3 + lo, Pb, yc, ec, true);
            else if (slot_ok(P, pc.h, blockIdx.x, 0xB003))
                load_carry_half(P.slots_rev, P.slot_stride, pc.h, blockIdx.x, j, hf, R3 + lo, 0u,
                                0u, Pb, yc, ec, true, false);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barPb);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                const uint32_t ph = it & 1;
                const long long row0 = (long long)c * kC;
                const float igj = row0 + j < P.N ? 1.f / ng : 0.f, dtj = ndt, yej = nye;
                {
                    long long nh;
                    int nc;
                    if (next_rev_chunk(pi, pc, c, &nh, &nc)) load_chunk_stats(P, nh, nc, j, hf, &ng, &ndt, &nye);
                }
                ok = wait_or_abort(full, ph, abort_flag, P.status, 0x408);
                if (!ok) break;
                scale_row_half(ot, j, hf, igj);  // dO row -> dOt row in place
                if (hf == 0) sDt[j] = dtj;
                fence_proxy_async_smem();
                mbar_arrive(barO);
                if (u == 0) bulk_wait_read0();  // the previous chunk's dV and dK have left their staging tiles
                epi_sync256();  // every dt_i is in sDt
                // columns are query rows i of the chunk: keep i >= j.  Each half rewrites only the R0 columns it has
                // read: P^T of its 64 rows i into R0 + 64 hf + [0, 32), then U^T into R0 + 64 hf + [32, 64)
                ok = wait_or_abort(barT1, ph, abort_flag, P.status, 0x40A);
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t pk[32];
                    tmem_half_to_bf16(R0 + lo, hf, [&](int i, float x) { return i >= j ? 1.f + x : 0.f; }, pk);
                    tmem_st32(R0 + lo + 64 * hf, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP1);
                }
                ok = wait_or_abort(barT2, ph, abort_flag, P.status, 0x409);
                if (!ok) break;
                tc_fence_after();
                {
                    uint32_t pk[32];
                    tmem_half_to_bf16(R1 + lo, hf, [&](int i, float x) { return i >= j ? x - sDt[i] : 0.f; }, pk);
                    tmem_st32(R0 + lo + 64 * hf + 32, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP2);
                }
                // dV_j = [R2]_j + e
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x40C);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R2 + lo, hf, ec, 1.f, dvt, j);
                fence_proxy_async_smem();
                epi_sync256();
                if (u == 0) store_tile<FLAT>(&P.tmdV, dvt, (int)row0, head_coord<FLAT>(pc.h, P.H), P.nbox);
                // dK_j = [R1]_j - y
                ok = wait_or_abort(barK, ph, abort_flag, P.status, 0x40B);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R1 + lo, hf, yc, -1.f, dkt, j);
                fence_proxy_async_smem();
                epi_sync256();  // dK rows staged; every read of yc and ec for this chunk is done
                if (u == 0) store_tile<FLAT>(&P.tmdK, dkt, (int)row0, head_coord<FLAT>(pc.h, P.H), P.nbox);
                // P (with this chunk's rows, for the earlier chunks) -> Pb: its update finished before dV
                if (c > pc.a) {
                    tmem_half_to_tile(R3 + lo, Pb, j, hf);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(barR);
                if (c > pc.a) mbar_arrive(barPb);
                (hf == 0 ? yc : ec)[j] += yej;  // this chunk's rows join the later ones
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

// ----------------------------------------------------------------------------------------------------
// dK / dV walk, non-causal: dK = V Pb^T - y and dV = K Pb + e with the head's totals P, y, e
// (the sum of all its pieces' slots), so only K and V are read.  Three TMA stages of (K, V); R2 accumulates dK,
// then dV; dK leaves through the V tile and dV through the K tile.
// ----------------------------------------------------------------------------------------------------
template <bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_bwd_dkdv_nc_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64, NST = 3;
    constexpr uint32_t TB = NB * kBox;
    constexpr uint32_t STAGE = 2 * TB;  // K, V
    constexpr uint32_t E = kEpiThreads;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Pb = sm + NST * STAGE;
    float *yc = (float *)(Pb + TB);
    float *ec = yc + D;
    uint64_t *full = (uint64_t *)(ec + D);
    uint64_t *empty = full + NST;
    uint64_t *bar = empty + NST;
    uint64_t *barPb = bar, *barK = bar + 1, *barKf = bar + 2, *barV = bar + 3, *barVf = bar + 4;
    uint32_t *tslot = (uint32_t *)(bar + 5);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // MMA commit + the epilogue once its dK, dV tiles have left shared memory
        }
        const uint32_t counts[5] = {E, 1, E, 1, E};
        for (int k = 0; k < 5; ++k) mbar_init(&bar[k], counts[k]);
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
    if (P.check_tag) {  // the forward's per-piece sums are reused: are they in the workspace, and did the
                        // dQ walk before this kernel take them?
        if (threadIdx.x == 0 && (!state_tag_matches(P, (uint64_t)P.check_tag - 1) || *bwd_skip(P))) {
            *abort_flag = 1;
            report(P.status, kDevState, 0x5A7Eu);
        }
        __syncthreads();
    }
    // this backward's reverse sums now fill the slots of the forward's sums (the dQ walk, which checked
    // them, is complete)
    if (blockIdx.x == 0 && threadIdx.x == 0) *fwd_sums_used(P) = 1u;
    const bool skip = *abort_flag != 0;
    const uint32_t tmem = *tslot;
    const uint32_t R2 = tmem + 256;

    if (skip) {
        // the state this call relies on is not in the workspace: nothing to compute
    } else if (warp == 0 && lane == 0) {
        // ---- TMA producer (chunks of each piece in reverse order)
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        {  // the first piece's carry slot
            PieceIter p0(P.sl, blockIdx.x);
            if (p0.valid() && slot_ok(P, p0.get().h, blockIdx.x, 0xB0F0))
                bulk_prefetch_l2(P.slots_rev + slot_of(p0.get().h, blockIdx.x) * P.slot_stride,
                                 (uint32_t)(kSlotF4 * sizeof(float4)));
        }
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            const HeadCoord hc = head_coord<FLAT>(pc.h, P.H);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                prefetch_next_carry(pi, c - pc.a, pc.e - pc.a, P.slots_rev, P.slot_stride, blockIdx.x, n_slot_floats(P), P.status);
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x421)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tile_load<FLAT>(st + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, hc);
                    tile_load<FLAT>(st + TB + nb * kBox, &P.tmV, &full[s], nb * 64, c * kC, hc);
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
        const uint32_t pb = smem_u32(Pb);
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!wait_or_abort(barPb, pno & 1, abort_flag, P.status, 0x422)) break;
            for (int c = pc.e - 1; c >= pc.a && ok; --c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x423);
                if (ok && it > 0) ok = wait_or_abort(barVf, ph ^ 1, abort_flag, P.status, 0x424);  // R2 drained
                if (!ok) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(stages + s * STAGE), vb = kb + TB;
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // dK = V Pb^T
                    const uint32_t o = (k >> 2) * kBox + 32 * (k & 3);
                    mma_ss(R2, sdesc_sw128(vb + o, 16, 1024), sdesc_sw128(pb + o, 16, 1024), idKK, k > 0);
                }
                mma_commit(barK);
                ok = wait_or_abort(barKf, ph, abort_flag, P.status, 0x425);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // dV = K Pb
                    mma_ss(R2, sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(pb + 2048 * k, kBox, 1024), idKM, k > 0);
                mma_commit(barV);
                mma_commit(&empty[s]);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread <-> key row j (TMEM lane) and column half hf
        const int u = threadIdx.x - 64;
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int j = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // the head's totals (every piece of a head carries the same sums); the previous piece's MMAs
            // on Pb are complete (its last barV)
            if (slot_ok(P, pc.h, blockIdx.x, 0xB003))
                load_carry_half(P.slots_rev, P.slot_stride, pc.h, blockIdx.x, j, hf, 0u, 0u, 0u, Pb,
                                yc, ec, false, false);
            fence_proxy_async_smem();
            epi_sync256();
            mbar_arrive(barPb);
            for (int c = pc.e - 1; c >= pc.a; --c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                const int row0 = c * kC;
                // dK_j = [R2]_j - y, staged in the V tile (its last reader, dK = V Pb^T, is done)
                ok = wait_or_abort(barK, ph, abort_flag, P.status, 0x426);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R2 + lo, hf, yc, -1.f, st + TB, j);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barKf);
                epi_sync256();
                if (u == 0) store_tile<FLAT>(&P.tmdK, st + TB, row0, head_coord<FLAT>(pc.h, P.H), P.nbox);
                // dV_j = [R2]_j + e, staged in the K tile (its last reader, dV = K Pb, is done)
                ok = wait_or_abort(barV, ph, abort_flag, P.status, 0x427);
                if (!ok) break;
                tc_fence_after();
                tmem_half_to_out(R2 + lo, hf, ec, 1.f, st, j);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(barVf);
                epi_sync256();
                if (u == 0) {
                    store_tile<FLAT>(&P.tmdV, st, row0, head_coord<FLAT>(pc.h, P.H), P.nbox);
                    bulk_wait_read0();
                    mbar_arrive(&empty[s]);
                }
            }
            epi_sync256();  // every read of Pb, yc, ec is done before the next piece's carry
        }
    }
    if (threadIdx.x == 64) bulk_wait0();  // output stores complete before the CTA exits
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace tc

// ======================================================================================== host ===

namespace {

constexpr size_t kTB = 2 * (size_t)tc::kBox;
constexpr size_t kEpiSmemDq = 2 * 128 * 4 + 4 * 128 * 4;  // z, a, 2 row-partial arrays
constexpr size_t kSmemDq = 4 * kTB + 2 * kTB + 1024 + 2048 + kEpiSmemDq + 512;    // 1 stage of Q, dO, K, V; Sb; dQ; ones; dt
constexpr size_t kSmemDqNc = 2 * 2 * kTB + 2 * kTB + 1024 + 4096 + kEpiSmemDq + 512;  // 2 stages of Q, dO; Sb; dQ; ones; 2 dt
constexpr size_t kSmemDkdv = 4 * kTB + 3 * kTB + 3 * 128 * 4 + 512;  // stage; Pb; dV; dK; y, e, dt
constexpr size_t kSmemDkdvNc = 3 * 2 * kTB + kTB + 2 * 128 * 4 + 512;         // 3 stages of K, V
static_assert(kSmemDkdvNc <= 232448 && kSmemDkdv <= 232448 && kSmemDq <= 232448 && kSmemDqNc <= 232448, "backward kernel exceeds the shared-memory limit");

bool set_bwd_attrs() {
    static std::atomic<int> state[kMaxDevices];
    return once_per_device(state, [] {
        const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
        bool ok = true;
        for (int f = 0; f < 2 && ok; ++f)
            ok = cudaFuncSetAttribute(f ? tc::tc_bwd_dq_kernel<true, false> : tc::tc_bwd_dq_kernel<false, false>, A,
                                      (int)kSmemDq) == cudaSuccess &&
                 cudaFuncSetAttribute(f ? tc::tc_bwd_dq_kernel<true, true> : tc::tc_bwd_dq_kernel<false, true>, A,
                                      (int)kSmemDq) == cudaSuccess &&
                 cudaFuncSetAttribute(f ? tc::tc_bwd_dq_nc_kernel<true> : tc::tc_bwd_dq_nc_kernel<false>, A,
                                      (int)kSmemDqNc) == cudaSuccess &&
                 cudaFuncSetAttribute(f ? tc::tc_bwd_dkdv_kernel<true> : tc::tc_bwd_dkdv_kernel<false>, A,
                                      (int)kSmemDkdv) == cudaSuccess &&
                 cudaFuncSetAttribute(f ? tc::tc_bwd_dkdv_nc_kernel<true> : tc::tc_bwd_dkdv_nc_kernel<false>, A,
                                      (int)kSmemDkdvNc) == cudaSuccess;
        return ok;
    });
}

}  // namespace

cudaError_t tc_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s, bool reuse_fwd_state) {
    if (!set_bwd_attrs()) return cudaErrorInvalidValue;
    tc::TcParams P;
    memset(&P, 0, sizeof(P));
    if (!tc_host::fill_common(P, p, ws)) return cudaErrorInvalidDevice;
    // causal, reusing the forward's state: one reverse sweep per head where it is estimated faster, else
    // the two walks with the dQ walk taking g from the forward and delta from O (both read O's tiles
    // through a map of the same form as the others)
    const bool sweep = reuse_fwd_state && tc_sweep_chosen(p, tc_host::sm_count());
    const bool rows = reuse_fwd_state && p.causal;
    const int ops[8] = {kOpQ, kOpK, kOpV, kOpdO, kOpdQ, kOpdK, kOpdV, kOpO};
    const bool flat = tc_host::flat_heads(p, ops, rows ? 8 : 7);
    if (!tc_host::make_map(&P.tmQ, Q, p, kOpQ, flat) || !tc_host::make_map(&P.tmK, K, p, kOpK, flat) ||
        !tc_host::make_map(&P.tmV, V, p, kOpV, flat) || !tc_host::make_map(&P.tmdO, dO, p, kOpdO, flat) ||
        !tc_host::make_map(&P.tmdQ, dQ, p, kOpdQ, flat) || !tc_host::make_map(&P.tmdK, dK, p, kOpdK, flat) ||
        !tc_host::make_map(&P.tmdV, dV, p, kOpdV, flat))
        return cudaErrorInvalidValue;
    P.flat = flat ? 1 : 0;
    P.Kp = K;
    P.Vp = V;
    if (rows && !tc_host::make_map(&P.tmO, O, p, kOpO, flat)) return cudaErrorInvalidValue;
    if (sweep) return tc_backward_sweep(p, P, O, dQ, dK, dV, ws, s);
    // The reverse sums share the slot array with the forward sums: the dQ walk reads a piece's forward
    // carry when the piece starts and writes that piece's reverse sums (same slot, same CTA) when it ends.
    P.slots_rev = (float *)(ws + p.off_states2);
    P.rs_g = (float *)(ws + p.off_rowstats);
    P.rs_dt = P.rs_g + (size_t)p.BH * p.N;
    P.chunk_ye = (float *)(ws + p.off_chunkye);
    P.dQ = dQ;
    P.dK = dK;
    P.dV = dV;
    P.Kp = K;
    P.Vp = V;
    // reusing the forward's sums: they must be in the form this pass expects (raw piece sums for causal,
    // head totals for non-causal)
    P.check_tag = reuse_fwd_state ? (int)(p.causal ? tc::kTagPrefix : tc::kTagTotals) + 1 : 0;
    const unsigned nthr = 64 + tc::kEpiThreads;
    unsigned launches = 0;
    cudaError_t e = cudaSuccess;
    if (!reuse_fwd_state) {
        e = tc_host::launch_agg(P, s);
        ++launches;
        if (e == cudaSuccess && !P.whole_heads) {
            e = tc_host::launch_combine(P, P.slots, p.causal ? tc::kCombinePrefix : tc::kCombineTotal,
                                        p.causal ? tc::kTagPrefix : tc::kTagTotals, s);
            ++launches;
        }
    }
    if (e == cudaSuccess) {
        e = p.causal ? tc_host::launch_tc(rows ? (flat ? tc::tc_bwd_dq_kernel<true, true> : tc::tc_bwd_dq_kernel<false, true>)
                                               : (flat ? tc::tc_bwd_dq_kernel<true, false> : tc::tc_bwd_dq_kernel<false, false>),
                                          P.sl.G, nthr, kSmemDq, s, P)
                     : tc_host::launch_tc(flat ? tc::tc_bwd_dq_nc_kernel<true> : tc::tc_bwd_dq_nc_kernel<false>,
                                          P.sl.G, nthr, kSmemDqNc, s, P);
        ++launches;
    }
    if (e == cudaSuccess && !P.whole_heads) {  // whole heads: each piece's reverse sums are its head's totals
        e = tc_host::launch_combine(P, P.slots_rev, p.causal ? tc::kCombineSuffix : tc::kCombineTotal, 0, s);
        ++launches;
    }
    if (e == cudaSuccess) {
        e = p.causal ? tc_host::launch_tc(flat ? tc::tc_bwd_dkdv_kernel<true> : tc::tc_bwd_dkdv_kernel<false>,
                                          P.sl.G, nthr, kSmemDkdv, s, P)
                     : tc_host::launch_tc(flat ? tc::tc_bwd_dkdv_nc_kernel<true> : tc::tc_bwd_dkdv_nc_kernel<false>,
                                          P.sl.G, nthr, kSmemDkdvNc, s, P);
        ++launches;
    }
    if (e == cudaSuccess) count_launches(launches);
    return e;
}

}  // namespace la
