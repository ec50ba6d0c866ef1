// la_tc_fwd.cu -- tcgen05 / TMA kernels of the bf16 path (kernels on 128 columns; D = 32, 64 zero-extended by the
// tensor maps): per-piece state sums and the forward.
//
// Method ("Transformer Based Linear Attention with Optimized GPU Kernel Implementation", sciencestack.ai
// page, TL;DR: O(N D^2) time, O(N D) memory, normalisation scheme), per head, rows i, chunk c of kC rows:
//   O_i = (sum_{j <= i} (1 + q_i . k_j) v_j) / g_i,   g_i = sum_{j <= i} (1 + q_i . k_j)
//       = (a_c + S_c^T q_i + [P V]_i) / (n_c + q_i . z_c + r_i)
// with S_c = sum_{j < c} k_j v_j^T, z_c = sum k_j, a_c = sum v_j, n_c = c kC over earlier rows, and the
// intra-chunk weights P_ij = [j <= i](1 + q_i . k_j), r_i = sum_j P_ij.  Non-causal: S, z, a are the
// head's totals, n = N, and there is no intra-chunk term.
//
// Roles in each CTA (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues tcgen05.mma,
// warps 2-5 (128 threads, one per TMEM lane / chunk row) run the epilogues.
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

// ----------------------------------------------------------------------------------------------------
// Per-piece state sums: for every piece (head h, chunks [a, e)) of this CTA's slice,
//   S = sum k_j v_j^T (D x D),  z = sum k_j,  a = sum v_j   (fp32, rows of the piece)
// written to workspace slot (h + blockIdx.x) as [S (slot_f4 layout) | z | a], and every chunk's own
// z_c, a_c to the chunk_za array (the walks take them from there instead of forming them again).
// TMEM: two S accumulators (128 columns each) so that one piece's read-out overlaps the next piece's
// MMAs, and two per-chunk z_c, a_c blocks (16 + 16 columns) from MMAs against a tile of ones (N = 16);
// the epilogue drains z_c, a_c every chunk and adds them up for the piece in fp32 registers.
// ----------------------------------------------------------------------------------------------------
template <bool FLAT>
__global__ void __launch_bounds__(192, 1) tc_agg_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64, NST = 3;
    constexpr uint32_t STAGE = 2 * NB * kBox;  // K and V boxes
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *ones = sm + NST * STAGE;  // 16 rows x 128 B of bf16 1.0
    uint64_t *full = (uint64_t *)(ones + 2048);
    uint64_t *empty = full + NST;
    uint64_t *accfull = empty + NST;
    uint64_t *accfree = accfull + 2;
    uint64_t *zafull = accfree + 2;  // [2] the chunk's z_c, a_c are in TMEM block it & 1
    uint64_t *zafree = zafull + 2;   // [2] the epilogue has read them
    uint32_t *tslot = (uint32_t *)(zafree + 2);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accfree[b], 128);
            mbar_init(&zafull[b], 1);
            mbar_init(&zafree[b], 128);
        }
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < 512; i += blockDim.x) ((uint32_t *)ones)[i] = 0x3F803F80u;
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
    // the slots below belong to P.Kp, P.Vp: each piece's own sums (until combined), or with whole_heads the
    // heads' totals; they are new, so no backward has used them
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        write_state_tag(P, P.whole_heads ? kTagTotals : kTagRaw);
        *fwd_sums_used(P) = 0u;
        *fwd_terms_kept(P) = 0u;  // set again by the causal combine when it keeps the totals
    }
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        const int drop = blockIdx.x == 0 ? P.test_drop_load : -1;  // test hook (normally -1)
        int it = 0;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && !*abort_flag; pi.next()) {
            const Piece pc = pi.get();
            const HeadCoord hc = head_coord<FLAT>(pc.h, P.H);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x101))
                    break;
                if (it == drop) continue;  // nothing issued: the MMA issuer's wait for this stage runs out
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tile_load<FLAT>(st + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, hc);
                    tile_load<FLAT>(st + (NB + nb) * kBox, &P.tmV, &full[s], nb * 64, c * kC, hc);
                }
            }
        }
        if (*abort_flag) {  // let the copies already issued land before the CTA exits
            for (int k = it > NST ? it - NST : 0; k < it; ++k)
                if (k != drop) mbar_wait(&full[k % NST], (k / NST) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idS = idesc_bf16(128, 128, true, true);
        const uint32_t idZ = idesc_bf16(128, 16, true, false);
        const uint32_t ones_a = smem_u32(ones);
        int it = 0, p = 0;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && !*abort_flag; pi.next(), ++p) {
            const Piece pc = pi.get();
            const int buf = p & 1;
            const uint32_t acc = tmem + buf * 128;
            if (p >= 2 && !wait_or_abort(&accfree[buf], ((p >> 1) - 1) & 1, abort_flag, P.status, 0x102)) break;
            tc_fence_after();
            bool ok = true;
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST, zb = it & 1;
                if (!wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x103) ||
                    (it >= 2 && !wait_or_abort(&zafree[zb], ((it >> 1) - 1) & 1, abort_flag, P.status, 0x105))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_u32(stages + s * STAGE), vb = kb + NB * kBox;
                const uint32_t za = tmem + 256 + 32 * zb;
#pragma unroll
                for (int k = 0; k < kC / 16; ++k) {
                    const uint64_t kt = sdesc_sw128(kb + 2048 * k, kBox, 1024);  // K^T, MN-major, 16 rows
                    const uint64_t vt = sdesc_sw128(vb + 2048 * k, kBox, 1024);  // V,   MN-major, 16 rows
                    const uint64_t on = sdesc_sw128(ones_a + 32 * (k & 3), 16, 1024);
                    mma_ss(acc, kt, vt, idS, (c > pc.a || k > 0) ? 1u : 0u);  // S += K^T V
                    mma_ss(za, kt, on, idZ, k > 0 ? 1u : 0u);                // z_c = K^T 1
                    mma_ss(za + 16, vt, on, idZ, k > 0 ? 1u : 0u);           // a_c = V^T 1
                }
                mma_commit(&zafull[zb]);
                mma_commit(&empty[s]);
            }
            if (!ok) break;
            mma_commit(&accfull[buf]);
        }
    } else if (warp >= 2) {
        // ---- epilogue: per chunk z_c, a_c (TMEM -> chunk_za, running piece sums); per piece S -> slot
        const int lb = 32 * (warp & 3);
        const int d = lb + lane;
        int p = 0, it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++p) {
            const Piece pc = pi.get();
            const int buf = p & 1;
            float zs = 0.f, as = 0.f;  // the piece's z[d], a[d]
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int zb = it & 1;
                if (!wait_or_abort(&zafull[zb], (it >> 1) & 1, abort_flag, P.status, 0x106)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t z0, z1, a0, a1;
                const uint32_t za = tmem + ((uint32_t)lb << 16) + 256 + 32 * zb;
                tmem_ld2(za, z0, z1);
                tmem_ld2(za + 16, a0, a1);
                tmem_wait_ld(z0, z1);
                tmem_wait_ld(a0, a1);
                tc_fence_before();
                mbar_arrive(&zafree[zb]);
                const long long ci = ((long long)pc.h * P.sl.nchunk + c) * 256;
                if (in_range(ci + d, n_chunk_floats(P), P.status, 0xB001) &&
                    in_range(ci + 128 + d, n_chunk_floats(P), P.status, 0xB001)) {
                    P.chunk_za[ci + d] = __uint_as_float(z0);
                    P.chunk_za[ci + 128 + d] = __uint_as_float(a0);
                }
                zs += __uint_as_float(z0);
                as += __uint_as_float(a0);
            }
            if (!ok) break;
            if (!wait_or_abort(&accfull[buf], (p >> 1) & 1, abort_flag, P.status, 0x104)) break;
            tc_fence_after();
            float *slot = P.slots + slot_of(pc.h, blockIdx.x) * P.slot_stride;
            const bool sok = slot_ok(P, pc.h, blockIdx.x, 0xB002);  // the same for the whole CTA
            const uint32_t ta = tmem + ((uint32_t)lb << 16) + buf * 128;
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                uint32_t r[16];
                tmem_ld16(ta + c16 * 16, r);
                tmem_wait_ld(r);
                float4 *dst = (float4 *)slot;
#pragma unroll
                for (int q = 0; q < 4; ++q)  // columns 16 c16 + 4 q: half c16 / 4, float4 4 (c16 % 4) + q of the half
                    if (sok) dst[slot_f4(d, c16 >> 2, 4 * (c16 & 3) + q)] =
                        make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                    __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            }
            if (sok) {
                slot[(size_t)D * D + d] = zs;
                slot[(size_t)D * D + D + d] = as;
            }
            tc_fence_before();
            mbar_arrive(&accfree[buf]);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ----------------------------------------------------------------------------------------------------
// Forward output.  Per chunk (causal): T = Q K^T; O = Q Sb (Sb = bf16 state before the chunk) and
// S += K^T V (TMEM) while the epilogue forms P = [j <= i](1 + T) (bf16, in place in TMEM); O += P V; the
// epilogue then writes the next Sb from S; the running fp32 z, a advance by each chunk's z_c, a_c from the
// sums kernel.  The epilogue
// forms q_i . z and the normaliser.  Non-causal: O = Q Sb with the head's totals (no T, P or state update) into two
// alternating TMEM accumulators, so the MMA of one chunk overlaps the epilogue of the previous one, and
// q_i . z by an N = 16 MMA of Q against z (split into two bf16 parts, ~16 significant bits) beside each.
// Eight epilogue warps: two per TMEM lane quarter, each owning half of the columns; the causal row sums
// they share (r_i and q_i . z) are exchanged through two TMEM columns.
// TMEM: causal  T 0-127, O 128-255, S 256-383, exchange 416-419;
//       non-causal  O 0-127 / 128-255, q . z 288-303 / 304-319.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL, bool FLAT>
__global__ void __launch_bounds__(64 + kEpiThreads, 1) tc_fwd_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr int NST = CAUSAL ? 2 : 4;
    constexpr uint32_t QB = NB * kBox;                  // Q (or K, V) tile of one chunk
    constexpr uint32_t STAGE = CAUSAL ? 3 * QB : QB;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Sb = sm + NST * STAGE;               // bf16 state, [d][e], two 64-column boxes
    unsigned char *ztile = Sb + QB;                     // non-causal: z as an N = 16 operand (split_tile_put)
    float *zc = (float *)(ztile + (CAUSAL ? 0 : 2048));  // running z (fp32, D)
    float *ac = zc + D;                                 // running a (fp32, D)
    uint64_t *full = (uint64_t *)(ac + D);
    uint64_t *empty = full + NST;
    uint64_t *barT = empty + NST, *barP = barT + 1, *barSb = barP + 1, *barS = barSb + 1;
    uint64_t *barO = barS + 1;    // [2]
    uint64_t *barOf = barO + 2;   // [2] non-causal: accumulator drained
    uint32_t *tslot = (uint32_t *)(barOf + 2);
    AbortState *abst = (AbortState *)(tslot + 2);
    volatile int *abort_flag = &abst->flag;
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);  // MMA commit + the epilogue, once its O tile has left the Q tile
        }
        mbar_init(barT, 1);
        mbar_init(barP, kEpiThreads);
        mbar_init(barSb, kEpiThreads);
        mbar_init(barS, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&barO[b], 1);
            mbar_init(&barOf[b], kEpiThreads);
        }
        *abort_flag = 0;
        abst->limit_ns = P.wait_ns ? P.wait_ns : kWaitNs;
        fence_mbar_init();
    }
    if (!CAUSAL) {
        for (int k = threadIdx.x; k < 512; k += blockDim.x) ((uint32_t *)ztile)[k] = 0u;
        fence_proxy_async_smem();
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
    const uint32_t tmem = *tslot;
    const uint32_t tT = tmem, tS = tmem + 256;
    const uint32_t tQZ = tmem + 288;  // non-causal: q_i . z in two parts, per accumulator buffer (16 columns each)
    const uint32_t tX = tmem + (CAUSAL ? 416 : 256);

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmQ);
        if (CAUSAL) {
            prefetch_tmap(&P.tmK);
            prefetch_tmap(&P.tmV);
        }
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
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x201)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tile_load<FLAT>(st + nb * kBox, &P.tmQ, &full[s], nb * 64, c * kC, hc);
                    if (CAUSAL) {
                        tile_load<FLAT>(st + QB + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, hc);
                        tile_load<FLAT>(st + 2 * QB + nb * kBox, &P.tmV, &full[s], nb * 64, c * kC, hc);
                    }
                }
            }
        }
        if (!ok) {  // let the copies already issued land before the CTA exits
            for (int k = it > NST ? it - NST : 0; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1, 50000000ull);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        const uint32_t idKK = idesc_bf16(128, 128, false, false);
        const uint32_t idKM = idesc_bf16(128, 128, false, true);
        const uint32_t idMM = idesc_bf16(128, 128, true, true);
        const uint32_t idQZ = idesc_bf16(128, 16, false, false);
        const uint32_t sb = smem_u32(Sb);
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!CAUSAL && !wait_or_abort(barSb, pno & 1, abort_flag, P.status, 0x202)) break;
            for (int c = pc.a; c < pc.e && ok; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                const int ob = CAUSAL ? 0 : (it & 1);  // accumulator buffer
                const uint32_t tO = tmem + (CAUSAL ? 128 : 128 * ob);
                if (!CAUSAL && it >= 2) {
                    ok = wait_or_abort(&barOf[ob], ((it >> 1) - 1) & 1, abort_flag, P.status, 0x20A);
                    if (!ok) break;
                }
                ok = wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x203);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qb = smem_u32(stages + s * STAGE), kb = qb + QB, vb = qb + 2 * QB;
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)  // T = Q K^T, K steps over d
                        mma_ss(tT, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                    mma_commit(barT);
                    // once the epilogue has copied S into this chunk's Sb (and read the previous O out):
                    // O = Q Sb, then S += K^T V, both while the epilogue forms P
                    ok = wait_or_abort(barSb, ph, abort_flag, P.status, 0x205);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)  // O = Q Sb, K steps over d
                        mma_ss(tO, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(sb + 2048 * k, kBox, 1024), idKM, k > 0);
                    if (c + 1 < pc.e) {
#pragma unroll
                        for (int k = 0; k < kC / 16; ++k)  // S += K^T V
                            mma_ss(tS, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024),
                                   idMM, 1u);
                    }
                    mma_commit(barS);  // also: Q Sb, Sb's reader, is complete
                    ok = wait_or_abort(barP, ph, abort_flag, P.status, 0x204);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kC / 16; ++k)  // O += P V, K steps over j (P in TMEM, 8 columns each)
                        mma_ts(tO, tT + 8 * k, sdesc_sw128(vb + 2048 * k, kBox, 1024), idKM, 1u);
                } else {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)  // O = Q Sb, K steps over d
                        mma_ss(tO, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(sb + 2048 * k, kBox, 1024), idKM, k > 0);
                    const uint32_t zb = smem_u32(ztile);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)  // q_i . z (columns 0 and 1: two parts), K steps over d
                        mma_ss(tQZ + 16 * ob, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(zb + (k >> 2) * 1024 + 32 * (k & 3), 16, 0), idQZ, k > 0);
                }
                mma_commit(&barO[ob]);
                mma_commit(&empty[s]);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue: thread <-> chunk row i (TMEM lane) and column half hf
        const int q4 = warp & 3, hf = (warp - 2) >> 2;
        const int i = 32 * q4 + lane;
        const uint32_t lo = (uint32_t)(32 * q4) << 16;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            // carried state (causal: the earlier pieces of the head; non-causal: the whole head)
            if (CAUSAL && it > 0) {  // the previous piece's last MMAs must be done before TMEM S is reset
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x206)) break;
                tc_fence_after();
            }
            if (CAUSAL && pc.a == 0)  // the head's first piece: nothing before it
                zero_carry_half(i, hf, tS + lo, Sb, zc, ac, true);
            else if (slot_ok(P, pc.h, blockIdx.x, 0xB003))
                load_carry_half(P.slots, P.slot_stride, pc.h, blockIdx.x, i,
                                hf, tS + lo, 0u, 0u, Sb, zc, ac, CAUSAL, false);
            if (!CAUSAL && hf == 0) split_tile_put(ztile, i, zc[i]);  // the head's z for the q . z MMA
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync256();
            mbar_arrive(barSb);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                const int ob = CAUSAL ? 0 : (it & 1);
                const uint32_t tO = tmem + (CAUSAL ? 128 : 128 * ob);
                const uint32_t ph_o = CAUSAL ? ph : ((it >> 1) & 1);
                unsigned char *st = stages + s * STAGE;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                // this chunk's z_c[i] (half 0) or a_c[i] (half 1), from the sums kernel (causal)
                const long long zi = ((long long)pc.h * P.sl.nchunk + c) * 256 + hf * 128 + i;
                const float zav = CAUSAL && in_range(zi, n_chunk_floats(P), P.status, 0xB004) ? P.chunk_za[zi] : 0.f;
                float part = 0.f;
                if (CAUSAL) {
                    // P = [j <= i](1 + T) for this half's columns j; r_i partial sum in fp32
                    ok = wait_or_abort(barT, ph, abort_flag, P.status, 0x207);
                    if (!ok) break;
                    tc_fence_after();
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
                        const float p0 = j <= i ? 1.f + __uint_as_float(a0) : 0.f;
                        const float p1 = j + 1 <= i ? 1.f + __uint_as_float(a1) : 0.f;
                        pk[m] = pack_bf16(p0, p1);
                        part += p0 + p1;
                    }
                    tc_fence_before();
                    epi_sync256();  // both halves have read T before P overwrites it
                    tc_fence_after();
                    tmem_st32(tT + lo + 32 * hf, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP);
                }
                float gi;
                if (CAUSAL) {
                    part += dot_half(st, i, hf, zc);  // q_i . z over this half's d
                    // exchange columns alternate by chunk parity: the barrier below then orders every read of
                    // one chunk's pair before the other half's write of the same pair two chunks later
                    const uint32_t tXc = tX + lo + 2 * (it & 1);
                    tmem_st1(tXc + hf, __float_as_uint(part));
                    // g_i from both halves' partial sums
                    tmem_st_wait();
                    tc_fence_before();
                    epi_sync256();
                    tc_fence_after();
                    uint32_t x0, x1;
                    tmem_ld2(tXc, x0, x1);
                    tmem_wait_ld(x0, x1);
                    gi = (float)row0 + __uint_as_float(x0) + __uint_as_float(x1);
                }
                // output: O_i = (a + [P V + Q Sb]_i) / g_i, this half's 64 columns
                ok = wait_or_abort(&barO[ob], ph_o, abort_flag, P.status, 0x209);
                if (!ok) break;
                tc_fence_after();
                if (!CAUSAL) {  // g_i = N + q_i . z, formed by the MMA beside O
                    uint32_t x0, x1;
                    tmem_ld2(tQZ + 16 * ob + lo, x0, x1);
                    tmem_wait_ld(x0, x1);
                    gi = (float)P.N + __uint_as_float(x0) + __uint_as_float(x1);
                }
                const float inv = 1.f / gi;
                const bool row_ok = i < nvalid;
                // the O tile is staged in this stage's Q tile (Q is dead once O is complete; each thread
                // overwrites only the row and box it read for q . z) and leaves by TMA
                unsigned char *otile = st + hf * kBox;
#pragma unroll 1
                for (int half32 = 0; half32 < 2; ++half32) {
                    uint32_t v[32];
                    tmem_ld32(tO + lo + 64 * hf + 32 * half32, v);
                    tmem_wait_ld(v);
                    const float *aa = ac + 64 * hf + 32 * half32;
                    uint4 w[4];
                    uint32_t *wv = (uint32_t *)w;
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        wv[m] = pack_bf16((__uint_as_float(v[2 * m]) + aa[2 * m]) * inv,
                                          (__uint_as_float(v[2 * m + 1]) + aa[2 * m + 1]) * inv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) *(uint4 *)(otile + sw128_off(i, 4 * half32 + q)) = w[q];
                }
                if (row_ok && hf == 0 && (P.g || P.rs_g)) {
                    const long long gix = (long long)pc.h * P.N + row0 + i;
                    if (in_range(gix, n_row_floats(P), P.status, 0xB005)) {
                        if (P.g) P.g[gix] = gi;
                        if (P.rs_g) P.rs_g[gix] = gi;  // kept for the single-sweep backward
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                epi_sync256();  // the whole O tile is in shared memory
                if (threadIdx.x == 64) {
                    for (int nb = 0; nb < NB; ++nb)
                        if (nb == 0 || P.nbox > 1)
                            tile_store<FLAT>(&P.tmO, st + nb * kBox, nb * 64, (int)row0, head_coord<FLAT>(pc.h, P.H));
                    bulk_commit();
                    if (!CAUSAL && it > 0) {
                        // the previous chunk's O tile has been read out of shared memory: its stage may be
                        // refilled (four stages: the release can trail by a chunk, and this one's store runs on)
                        bulk_wait_read1();
                        mbar_arrive(&empty[(it - 1) % NST]);
                    }
                }
                if (!CAUSAL) mbar_arrive(&barOf[ob]);
                if (CAUSAL) {
                    // S after this chunk -> Sb for the next one (Q Sb, Sb's reader, is complete: barS)
                    ok = wait_or_abort(barS, ph, abort_flag, P.status, 0x208);
                    if (!ok) break;
                    tc_fence_after();
                    float vn = 0.f;  // z (half 0) or a (half 1) after this chunk, for row d = i
                    if (c + 1 < pc.e) {
                        tmem_half_to_tile(tS + lo, Sb, i, hf);
                        vn = (hf == 0 ? zc : ac)[i] + zav;  // z_c, a_c of this chunk from the sums kernel
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(barSb);
                    }
                    if (threadIdx.x == 64) {  // after the copy, which the next chunk's MMAs wait for
                        bulk_wait_read0();       // the O tile has been read out of shared memory
                        mbar_arrive(&empty[s]);  // the stage may be refilled
                    }
                    epi_sync256();  // everyone has read z and a of this chunk
                    if (c + 1 < pc.e) (hf == 0 ? zc : ac)[i] = vn;
                    epi_sync256();
                }
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

template __global__ void tc_fwd_kernel<true, true>(const __grid_constant__ TcParams P);
template __global__ void tc_fwd_kernel<false, true>(const __grid_constant__ TcParams P);
template __global__ void tc_fwd_kernel<true, false>(const __grid_constant__ TcParams P);
template __global__ void tc_fwd_kernel<false, false>(const __grid_constant__ TcParams P);

// ----------------------------------------------------------------------------------------------------
// Carries: in place over the piece slots of each head, in piece order, so that a walk then reads exactly
// one slot (its own) per piece: kCombinePrefix gives each piece the sum over the head's earlier pieces
// (causal, chunk order), kCombineSuffix over the later ones (causal, reverse order), kCombineTotal the
// head's total (non-causal).  grid = (ceil(kSlotF4 / 256), heads; heads beyond the grid's y extent loop);
// thread x owns float4 x of every slot of its head, and reads each slot before it writes it.  With
// P.htot set (a causal forward on a backward-sized workspace), kCombinePrefix also writes each head's
// total into slot h of P.htot, for the single-sweep backward, which walks each head from its end.  At most 32
// registers, so that eight CTAs fit on an SM and the whole grid (17 x 64 CTAs at the standard shape) runs
// in one wave: the kernel is a single round of loads and stores.
// ----------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 8) tc_combine_kernel(const __grid_constant__ TcParams P) {
    griddep_wait();  // the slots come from the previous kernel of the stream
    griddep_launch_dependents();
    if (P.combine_tag && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        write_state_tag(P, P.combine_tag);
        *fwd_sums_used(P) = 0u;
        *fwd_terms_kept(P) = P.htot != nullptr && P.combine_mode == kCombinePrefix ? 1u : 0u;
    }
    const int x = blockIdx.x * 256 + threadIdx.x;
    if (x >= kSlotF4) return;
    const long long BH = P.sl.T / P.sl.nchunk, s4 = P.slot_stride / 4;
    const int mode = P.combine_mode;
    float4 *base = (float4 *)P.combine_slots + x;
    for (long long h = blockIdx.y; h < BH; h += gridDim.y) {
        const long long x0 = h * P.sl.nchunk;
        const int b0 = cta_of(P.sl, x0), b1 = cta_of(P.sl, x0 + P.sl.nchunk - 1);
        const int n = b1 - b0 + 1;
        auto at = [&](int k) -> float4 * {  // k-th slot of the head in the order of the sums
            return base + slot_of(h, mode == kCombineSuffix ? b1 - k : b0 + k) * s4;
        };
#ifdef LA_CHECKED
        bool sok = true;  // every slot of the head inside the array (the same for all threads)
        for (int k = 0; k < n; ++k) sok = sok && slot_ok(P, h, mode == kCombineSuffix ? b1 - k : b0 + k, 0xB006);
        if (!sok) continue;
#endif
        float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g = 0; g < n; g += 4) {  // up to four loads in flight; each slot read before it is written
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (g + k < n) v[k] = *at(g + k);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (g + k < n) {
                    if (mode != kCombineTotal) *at(g + k) = run;  // exclusive: the sum before this piece
                    run.x += v[k].x;
                    run.y += v[k].y;
                    run.z += v[k].z;
                    run.w += v[k].w;
                }
        }
        if (mode == kCombineTotal)
            for (int k = 0; k < n; ++k) *at(k) = run;
        else if (P.htot && mode == kCombinePrefix &&
                 in_range(h * P.slot_stride + 4 * x + 3, n_htot_floats(P), P.status, 0xB00C))
            ((float4 *)P.htot)[h * s4 + x] = run;
    }
}

}  // namespace tc

// ======================================================================================== host ===

namespace tc_host {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    return fn;
}

int sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Operand `op` as a bf16 map with boxes of 128 rows x 64 columns of one head, 128-byte swizzle; rows
// past N and columns past D (D = 32, 64: the kernels work on 128 columns) read as zero and are not written.  flat: 3-D over {D, N, B H} (the operand's batch stride is H
// times its head stride); else 4-D over {D, N, H, B}.
bool make_map(CUtensorMap *m, const void *ptr, const Plan &p, int op, bool flat) {
    auto enc = encode_fn();
    if (!enc) return false;
    const Layout &l = p.lay[op];
    cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)p.N, (cuuint64_t)(flat ? p.BH : p.H), (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)l.sn * 2, (cuuint64_t)l.sh * 2, (cuuint64_t)l.sb * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)tc::kC, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, flat ? 3 : 4, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether every listed operand's heads can be numbered flat (batch stride = H x head stride, or B = 1).
bool flat_heads(const Plan &p, const int *ops, int n) {
    for (int k = 0; k < n; ++k) {
        const Layout &l = p.lay[ops[k]];
        if (p.B > 1 && l.sb != (long long)p.H * l.sh) return false;
    }
    return true;
}

constexpr size_t kSmemAgg = 3 * 2 * 2 * (size_t)tc::kBox + 2048 + 256;
constexpr size_t kSmemFwdCausal = 2 * 3 * 2 * (size_t)tc::kBox + 2 * (size_t)tc::kBox + 1024 + 256;
constexpr size_t kSmemFwdNonCausal = 4 * 2 * (size_t)tc::kBox + 2 * (size_t)tc::kBox + 2048 + 1024 + 256;
static_assert(kSmemFwdCausal <= 232448, "forward kernel exceeds the shared-memory limit");

bool set_smem_attrs() {
    static std::atomic<int> state[kMaxDevices];
    return once_per_device(state, [] {
        const cudaFuncAttribute A = cudaFuncAttributeMaxDynamicSharedMemorySize;
        return cudaFuncSetAttribute(tc::tc_agg_kernel<true>, A, (int)kSmemAgg) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_agg_kernel<false>, A, (int)kSmemAgg) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_fwd_kernel<true, true>, A, (int)kSmemFwdCausal) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_fwd_kernel<false, true>, A, (int)kSmemFwdNonCausal) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_fwd_kernel<true, false>, A, (int)kSmemFwdCausal) == cudaSuccess &&
               cudaFuncSetAttribute(tc::tc_fwd_kernel<false, false>, A, (int)kSmemFwdNonCausal) == cudaSuccess;
    });
}

bool fill_common(tc::TcParams &P, const Plan &p, unsigned char *ws) {
    const int nsm = sm_count();
    if (nsm <= 0) return false;
    P.sl.nchunk = (p.N + tc::kC - 1) / tc::kC;
    P.sl.T = (long long)p.BH * P.sl.nchunk;
    long long G = tc::choose_ctas(p.BH, P.sl.nchunk, nsm, p.causal != 0, p.D == 128);
    // Test hook: fewer CTAs, so that small problems also exercise multi-chunk, multi-head slices.
    if (const char *env = getenv("LA_TC_MAX_CTAS")) {
        const long long cap = atoll(env);
        if (cap >= 1 && cap < G) G = cap;
    }
    P.sl.G = (int)G;
    // non-causal, every slice one whole head: the sums kernel's piece sums are already the heads' totals
    P.whole_heads = !p.causal && G == p.BH && P.sl.T % G == 0 && P.sl.T / G == P.sl.nchunk ? 1 : 0;
    // Test hooks for the failure path: a shorter bound on barrier waits, and one load of the sums kernel
    // that is never issued, so that a wait runs out and the kernels take their abort path.
    P.wait_ns = 0;
    if (const char *env = getenv("LA_TEST_WAIT_NS")) {
        const long long ns = atoll(env);
        if (ns >= 1000000) P.wait_ns = (uint64_t)ns;
    }
    P.test_drop_load = -1;
    if (const char *env = getenv("LA_TEST_DROP_LOAD")) {
        const long long it = atoll(env);
        if (it >= 0 && it < (1LL << 30)) P.test_drop_load = (int)it;
    }
    P.N = p.N;
    P.H = p.H;
    uint64_t hsh = 0xcbf29ce484222325ull;  // FNV-1a over K's and V's strides, then D
    for (int op : {kOpK, kOpV})
        for (long long v : {p.lay[op].sb, p.lay[op].sh, p.lay[op].sn}) hsh = (hsh ^ (uint64_t)v) * 0x100000001b3ull;
    P.kv_layout = (hsh ^ (uint64_t)p.D) * 0x100000001b3ull;
    P.nbox = (p.D + 63) / 64;
    P.slot_stride = p.stride;
    P.slots = (float *)(ws + p.off_states);
    P.chunk_za = (float *)(ws + p.off_chunkza);
    P.status = (uint32_t *)ws;
    return true;
}

cudaError_t launch_tc(void (*kernel)(const tc::TcParams), dim3 grid, unsigned block, size_t smem,
                      cudaStream_t s, const tc::TcParams &P) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, P);
}

cudaError_t launch_combine(tc::TcParams P, float *slots, int mode, uint64_t tag_form, cudaStream_t s) {
    P.combine_slots = slots;
    P.combine_mode = mode;
    P.combine_tag = tag_form;
    const long long BH = P.sl.T / P.sl.nchunk;
    const dim3 grid((tc::kSlotF4 + 255) / 256, (unsigned)(BH < 65535 ? BH : 65535));
    return launch_tc(tc::tc_combine_kernel, grid, 256, 0, s, P);
}

cudaError_t launch_agg(const tc::TcParams &P, cudaStream_t s) {
    if (!set_smem_attrs()) return cudaErrorInvalidValue;
    return launch_tc(P.flat ? tc::tc_agg_kernel<true> : tc::tc_agg_kernel<false>, P.sl.G, 192, kSmemAgg, s, P);
}

}  // namespace tc_host

using namespace tc_host;

bool tc_supported(const Plan &p) { return p.dtype == 1 && (p.D == 32 || p.D == 64 || p.D == 128); }

size_t tc_slot_bytes(const Plan &p) { return ((size_t)p.BH + tc::kMaxCtas) * (size_t)p.stride * sizeof(float); }

cudaError_t tc_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                       unsigned char *ws, cudaStream_t s, bool keep_terms) {
    if (!set_smem_attrs()) return cudaErrorInvalidValue;
    tc::TcParams P;
    memset(&P, 0, sizeof(P));
    if (!fill_common(P, p, ws)) return cudaErrorInvalidDevice;
    const int ops[4] = {kOpQ, kOpK, kOpV, kOpO};
    const bool flat = flat_heads(p, ops, 4);
    if (!make_map(&P.tmQ, Q, p, kOpQ, flat) || !make_map(&P.tmK, K, p, kOpK, flat) ||
        !make_map(&P.tmV, V, p, kOpV, flat) || !make_map(&P.tmO, O, p, kOpO, flat))
        return cudaErrorInvalidValue;
    P.flat = flat ? 1 : 0;
    P.O = O;
    P.g = g;
    P.Kp = K;
    P.Vp = V;
    if (keep_terms && p.causal) {
        P.rs_g = (float *)(ws + p.off_rowstats);
        P.htot = (float *)(ws + p.off_htot);
    }
    cudaError_t e = launch_agg(P, s);
    if (e == cudaSuccess && !P.whole_heads)  // whole heads: the sums kernel has written the totals
        e = launch_combine(P, P.slots, p.causal ? tc::kCombinePrefix : tc::kCombineTotal,
                           p.causal ? tc::kTagPrefix : tc::kTagTotals, s);
    if (e == cudaSuccess)
        e = p.causal ? launch_tc(flat ? tc::tc_fwd_kernel<true, true> : tc::tc_fwd_kernel<true, false>, P.sl.G,
                                 64 + tc::kEpiThreads, kSmemFwdCausal, s, P)
                     : launch_tc(flat ? tc::tc_fwd_kernel<false, true> : tc::tc_fwd_kernel<false, false>, P.sl.G,
                                 64 + tc::kEpiThreads, kSmemFwdNonCausal, s, P);
    if (e == cudaSuccess) count_launches(P.whole_heads ? 2 : 3);
    return e;
}

}  // namespace la
