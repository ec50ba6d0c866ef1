// la_tc_fwd.cu -- tcgen05 / TMA kernels of the bf16 path (D = 128): per-piece state sums and the forward.
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
// written to workspace slot (h + blockIdx.x) as [S row-major | z | a].
// TMEM: two accumulator sets of 160 columns (S 128, z 16, a 16) so that one piece's read-out overlaps
// the next piece's MMAs.  z and a come from MMAs against a tile of ones (N = 16).
// ----------------------------------------------------------------------------------------------------
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
    uint32_t *tslot = (uint32_t *)(accfree + 2);
    volatile int *abort_flag = (volatile int *)(tslot + 1);
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
        }
        *abort_flag = 0;
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
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmK);
        prefetch_tmap(&P.tmV);
        int it = 0;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && !*abort_flag; pi.next()) {
            const Piece pc = pi.get();
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x101))
                    break;
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tma_load_3d(st + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, (int)pc.h);
                    tma_load_3d(st + (NB + nb) * kBox, &P.tmV, &full[s], nb * 64, c * kC, (int)pc.h);
                }
            }
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
            const uint32_t acc = tmem + buf * 256;
            if (p >= 2 && !wait_or_abort(&accfree[buf], ((p >> 1) - 1) & 1, abort_flag, P.status, 0x102)) break;
            tc_fence_after();
            bool ok = true;
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                if (!wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x103)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_u32(stages + s * STAGE), vb = kb + NB * kBox;
#pragma unroll
                for (int k = 0; k < kC / 16; ++k) {
                    const uint64_t kt = sdesc_sw128(kb + 2048 * k, kBox, 1024);  // K^T, MN-major, 16 rows
                    const uint64_t vt = sdesc_sw128(vb + 2048 * k, kBox, 1024);  // V,   MN-major, 16 rows
                    const uint64_t on = sdesc_sw128(ones_a + 32 * (k & 3), 16, 1024);
                    const uint32_t accum = (c > pc.a || k > 0) ? 1u : 0u;
                    mma_ss(acc, kt, vt, idS, accum);         // S += K^T V
                    mma_ss(acc + 128, kt, on, idZ, accum);   // z += K^T 1
                    mma_ss(acc + 144, vt, on, idZ, accum);   // a += V^T 1
                }
                mma_commit(&empty[s]);
            }
            if (!ok) break;
            mma_commit(&accfull[buf]);
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM -> workspace slot
        const int lb = 32 * (warp & 3);
        const int d = lb + lane;
        int p = 0;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && !*abort_flag; pi.next(), ++p) {
            const Piece pc = pi.get();
            const int buf = p & 1;
            if (!wait_or_abort(&accfull[buf], (p >> 1) & 1, abort_flag, P.status, 0x104)) break;
            tc_fence_after();
            float *slot = P.slots + slot_of(pc.h, blockIdx.x) * P.slot_stride;
            const uint32_t ta = tmem + ((uint32_t)lb << 16) + buf * 256;
#pragma unroll 1
            for (int c16 = 0; c16 < D / 16; ++c16) {
                uint32_t r[16];
                tmem_ld16(ta + c16 * 16, r);
                tmem_ld_wait();
                float4 *dst = (float4 *)(slot + (size_t)d * D + c16 * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                         __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            }
            uint32_t rz[16], ra[16];
            tmem_ld16(ta + 128, rz);
            tmem_ld16(ta + 144, ra);
            tmem_ld_wait();
            slot[(size_t)D * D + d] = __uint_as_float(rz[0]);
            slot[(size_t)D * D + D + d] = __uint_as_float(ra[0]);
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
// Forward output.  Per chunk (causal): T = Q K^T -> P = [j <= i](1 + T) (bf16, back into TMEM) ->
// O = P V + Q Sb (Sb = bf16 state before the chunk) -> S += K^T V, from which the epilogue writes the
// next Sb.  z and a (running column sums of K and V) are kept in fp32 by the epilogue warps, which also
// form q_i . z and the normaliser.  Non-causal: O = Q Sb with the head's total state, no T / P.
// ----------------------------------------------------------------------------------------------------
template <bool CAUSAL>
__global__ void __launch_bounds__(192, 1) tc_fwd_kernel(const __grid_constant__ TcParams P) {
    constexpr int D = 128, NB = D / 64;
    constexpr int NST = CAUSAL ? 2 : 4;
    constexpr uint32_t QB = NB * kBox;                  // Q (or K, V) tile of one chunk
    constexpr uint32_t STAGE = CAUSAL ? 3 * QB : QB;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    bool aligned;
    unsigned char *sm = smem_base(smem_raw, P.status, &aligned);
    unsigned char *stages = sm;
    unsigned char *Sb = sm + NST * STAGE;               // bf16 state, MN-major [d][e], two 64-column boxes
    float *zc = (float *)(Sb + QB);                     // running z (fp32, D)
    float *ac = zc + D;                                 // running a (fp32, D)
    uint64_t *full = (uint64_t *)(ac + D);
    uint64_t *empty = full + NST;
    uint64_t *barT = empty + NST, *barP = barT + 1, *barSb = barP + 1, *barO = barSb + 1, *barS = barO + 1;
    uint64_t *barOf = barS + 1;  // non-causal: the epilogue has drained the O accumulator
    uint32_t *tslot = (uint32_t *)(barOf + 1);
    volatile int *abort_flag = (volatile int *)(tslot + 1);
    if (!aligned) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 128);  // MMA commit + every epilogue thread (they read Q, K, V too)
        }
        mbar_init(barT, 1);
        mbar_init(barP, 128);
        mbar_init(barSb, 128);
        mbar_init(barO, 1);
        mbar_init(barS, 1);
        mbar_init(barOf, 128);
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
    const uint32_t tT = tmem, tO = tmem + 128, tS = tmem + 256;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        prefetch_tmap(&P.tmQ);
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
                if (it >= NST && !wait_or_abort(&empty[s], ((it / NST) - 1) & 1, abort_flag, P.status, 0x201)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], STAGE);
                unsigned char *st = stages + s * STAGE;
                for (int nb = 0; nb < NB; ++nb) {
                    tma_load_3d(st + nb * kBox, &P.tmQ, &full[s], nb * 64, c * kC, (int)pc.h);
                    if (CAUSAL) {
                        tma_load_3d(st + QB + nb * kBox, &P.tmK, &full[s], nb * 64, c * kC, (int)pc.h);
                        tma_load_3d(st + 2 * QB + nb * kBox, &P.tmV, &full[s], nb * 64, c * kC, (int)pc.h);
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
        const uint32_t sb = smem_u32(Sb);
        int it = 0, pno = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next(), ++pno) {
            const Piece pc = pi.get();
            if (!CAUSAL && !wait_or_abort(barSb, pno & 1, abort_flag, P.status, 0x202)) break;
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                if (!wait_or_abort(&full[s], (it / NST) & 1, abort_flag, P.status, 0x203)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qb = smem_u32(stages + s * STAGE), kb = qb + QB, vb = qb + 2 * QB;
                if (CAUSAL) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)  // T = Q K^T, K steps over d
                        mma_ss(tT, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                               sdesc_sw128(kb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024), idKK, k > 0);
                    mma_commit(barT);
                    if (!wait_or_abort(barP, ph, abort_flag, P.status, 0x204)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kC / 16; ++k)  // O = P V, K steps over j (P in TMEM, 8 columns each)
                        mma_ts(tO, tT + 8 * k, sdesc_sw128(vb + 2048 * k, kBox, 1024), idKM, k > 0);
                    if (!wait_or_abort(barSb, ph, abort_flag, P.status, 0x205)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                } else if (it > 0) {
                    // O is overwritten below: wait until the epilogue has read the previous chunk's O
                    // (otherwise barO could complete twice before its waiter sees the first phase)
                    if (!wait_or_abort(barOf, (it - 1) & 1, abort_flag, P.status, 0x20A)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < D / 16; ++k)  // O += Q Sb, K steps over d
                    mma_ss(tO, sdesc_sw128(qb + (k >> 2) * kBox + 32 * (k & 3), 16, 1024),
                           sdesc_sw128(sb + 2048 * k, kBox, 1024), idKM, (CAUSAL || k > 0) ? 1u : 0u);
                mma_commit(barO);
                if (CAUSAL) {
                    if (c + 1 < pc.e) {
#pragma unroll
                        for (int k = 0; k < kC / 16; ++k)  // S += K^T V, K steps over j
                            mma_ss(tS, sdesc_sw128(kb + 2048 * k, kBox, 1024), sdesc_sw128(vb + 2048 * k, kBox, 1024),
                                   idMM, 1u);
                    }
                    mma_commit(barS);
                }
                mma_commit(&empty[s]);
            }
        }
    } else if (warp >= 2) {
        // ---- epilogue warps: thread <-> chunk row i (TMEM lane) and state row d (same index)
        const int lb = 32 * (warp & 3);
        const int i = lb + lane;
        const uint32_t lane_off = (uint32_t)lb << 16;
        __nv_bfloat16 *Og = (__nv_bfloat16 *)P.O;
        int it = 0;
        bool ok = true;
        for (PieceIter pi(P.sl, blockIdx.x); pi.valid() && ok; pi.next()) {
            const Piece pc = pi.get();
            const long long h0 = pc.h * P.sl.nchunk;  // flat chunk index of the head's first chunk
            // carried state: causal = earlier pieces of the head, non-causal = all pieces of the head
            const int b_first = cta_of(P.sl, h0);
            const int b_to = CAUSAL ? (int)blockIdx.x : cta_of(P.sl, h0 + P.sl.nchunk - 1) + 1;
            if (CAUSAL && it > 0) {  // the previous piece's last S update must be done before TMEM S is reset
                if (!wait_or_abort(barS, (it - 1) & 1, abort_flag, P.status, 0x206)) break;
                tc_fence_after();
            }
            load_carry(P.slots, P.slot_stride, pc.h, CAUSAL && pc.a == 0 ? b_to : b_first, b_to, i, tS + lane_off, Sb, zc, ac, CAUSAL);
            fence_proxy_async_smem();
            tc_fence_before();
            epi_sync();
            mbar_arrive(barSb);
            for (int c = pc.a; c < pc.e; ++c, ++it) {
                const int s = it % NST;
                const uint32_t ph = it & 1;
                unsigned char *st = stages + s * STAGE;
                const long long row0 = (long long)c * kC;
                const int nvalid = (int)min((long long)kC, P.N - row0);
                float r = 0.f;
                if (CAUSAL) {
                    // P = [j <= i](1 + T), bf16, written over T's first 64 columns; r_i = sum_j P_ij (fp32)
                    if (!wait_or_abort(barT, ph, abort_flag, P.status, 0x207)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int q = 0; q < kC / 32; ++q) {
                        uint32_t t0[16], t1[16], pk[16];
                        tmem_ld16(tT + lane_off + 32 * q, t0);
                        tmem_ld16(tT + lane_off + 32 * q + 16, t1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j2 = 0; j2 < 16; ++j2) {
                            const int j = 32 * q + 2 * j2;
                            const uint32_t lo = j2 < 8 ? t0[2 * j2] : t1[2 * j2 - 16];
                            const uint32_t hi = j2 < 8 ? t0[2 * j2 + 1] : t1[2 * j2 - 15];
                            const float p0 = j <= i ? 1.f + __uint_as_float(lo) : 0.f;
                            const float p1 = j + 1 <= i ? 1.f + __uint_as_float(hi) : 0.f;
                            pk[j2] = pack_bf16(p0, p1);
                            r += p0 + p1;  // the normaliser sums the fp32 weights; only the MMA operand is bf16
                        }
                        tmem_st16(tT + lane_off + 16 * q, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(barP);
                }
                // q_i . z (z before this chunk), from the Q tile in shared memory
                float qz = 0.f;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        const uint4 v = *(const uint4 *)(st + nb * kBox + sw128_off(i, g8));
                        const float *zz = zc + nb * 64 + g8 * 8;
                        qz += bf16lo(v.x) * zz[0] + bf16hi(v.x) * zz[1] + bf16lo(v.y) * zz[2] + bf16hi(v.y) * zz[3] +
                              bf16lo(v.z) * zz[4] + bf16hi(v.z) * zz[5] + bf16lo(v.w) * zz[6] + bf16hi(v.w) * zz[7];
                    }
                }
                float anew0 = 0.f, anew1 = 0.f;
                const int t = threadIdx.x - 64;  // 0..127
                if (CAUSAL) {
                    epi_sync();  // every thread has read z before it is advanced
                    // column sums of this chunk's K (threads 0-63) or V (64-127), two columns each
                    const int col = 2 * (t & 63);
                    const unsigned char *tile = st + (t < 64 ? QB : 2 * QB) + (col / 64) * kBox;
                    const int cc = col % 64;
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
                    for (int j = 0; j < kC; ++j) {
                        const uint32_t v = *(const uint32_t *)(tile + sw128_off(j, cc / 8) + (cc % 8) * 2);
                        s0 += bf16lo(v);
                        s1 += bf16hi(v);
                    }
                    if (t < 64) {
                        zc[col] += s0;
                        zc[col + 1] += s1;
                    } else {
                        anew0 = ac[col] + s0;
                        anew1 = ac[col + 1] + s1;
                    }
                }
                mbar_arrive(&empty[s]);  // this thread is done reading the stage
                if (CAUSAL) {
                    // next chunk's Sb from the updated state (not after the piece's last chunk)
                    if (!wait_or_abort(barS, ph, abort_flag, P.status, 0x208)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (c + 1 < pc.e) {
#pragma unroll 1
                        for (int c16 = 0; c16 < D / 16; ++c16) {
                            uint32_t v[16];
                            tmem_ld16(tS + lane_off + c16 * 16, v);
                            tmem_ld_wait();
                            unsigned char *tile = Sb + (c16 / 4) * kBox;
                            const int col8 = (c16 % 4) * 2;
#pragma unroll
                            for (int g2 = 0; g2 < 2; ++g2) {
                                uint4 w;
                                w.x = pack_bf16(__uint_as_float(v[8 * g2 + 0]), __uint_as_float(v[8 * g2 + 1]));
                                w.y = pack_bf16(__uint_as_float(v[8 * g2 + 2]), __uint_as_float(v[8 * g2 + 3]));
                                w.z = pack_bf16(__uint_as_float(v[8 * g2 + 4]), __uint_as_float(v[8 * g2 + 5]));
                                w.w = pack_bf16(__uint_as_float(v[8 * g2 + 6]), __uint_as_float(v[8 * g2 + 7]));
                                *(uint4 *)(tile + sw128_off(i, col8 + g2)) = w;
                            }
                        }
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(barSb);
                    }
                }
                // output rows: O_i = (a + [P V + Q Sb]_i) / g_i
                if (!wait_or_abort(barO, ph, abort_flag, P.status, 0x209)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float n_prev = CAUSAL ? (float)row0 : (float)P.N;
                const float gi = n_prev + qz + r;
                const float inv = 1.f / gi;
                const bool row_ok = i < nvalid;
                __nv_bfloat16 *orow = Og + ((size_t)pc.h * P.N + row0 + i) * D;
#pragma unroll 1
                for (int c16 = 0; c16 < D / 16; ++c16) {
                    uint32_t v[16];
                    tmem_ld16(tO + lane_off + c16 * 16, v);
                    tmem_ld_wait();
                    uint4 w0, w1;
                    const float *aa = ac + c16 * 16;
                    w0.x = pack_bf16((__uint_as_float(v[0]) + aa[0]) * inv, (__uint_as_float(v[1]) + aa[1]) * inv);
                    w0.y = pack_bf16((__uint_as_float(v[2]) + aa[2]) * inv, (__uint_as_float(v[3]) + aa[3]) * inv);
                    w0.z = pack_bf16((__uint_as_float(v[4]) + aa[4]) * inv, (__uint_as_float(v[5]) + aa[5]) * inv);
                    w0.w = pack_bf16((__uint_as_float(v[6]) + aa[6]) * inv, (__uint_as_float(v[7]) + aa[7]) * inv);
                    w1.x = pack_bf16((__uint_as_float(v[8]) + aa[8]) * inv, (__uint_as_float(v[9]) + aa[9]) * inv);
                    w1.y = pack_bf16((__uint_as_float(v[10]) + aa[10]) * inv, (__uint_as_float(v[11]) + aa[11]) * inv);
                    w1.z = pack_bf16((__uint_as_float(v[12]) + aa[12]) * inv, (__uint_as_float(v[13]) + aa[13]) * inv);
                    w1.w = pack_bf16((__uint_as_float(v[14]) + aa[14]) * inv, (__uint_as_float(v[15]) + aa[15]) * inv);
                    if (row_ok) {
                        uint4 *dst = (uint4 *)(orow + c16 * 16);
                        dst[0] = w0;
                        dst[1] = w1;
                    }
                }
                if (row_ok && P.g) P.g[(size_t)pc.h * P.N + row0 + i] = gi;
                tc_fence_before();
                if (!CAUSAL) mbar_arrive(barOf);
                if (CAUSAL) {
                    epi_sync();  // everyone has read a before it is advanced
                    if (t >= 64) {
                        const int col = 2 * (t & 63);
                        ac[col] = anew0;
                        ac[col + 1] = anew1;
                    }
                    epi_sync();
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template __global__ void tc_fwd_kernel<true>(const __grid_constant__ TcParams P);
template __global__ void tc_fwd_kernel<false>(const __grid_constant__ TcParams P);

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
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

// [BH][N][D] bf16 tensor, boxes of 128 rows x 64 columns, 128-byte swizzle; rows past N read as zero.
bool make_map(CUtensorMap *m, const void *ptr, const Plan &p) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)p.D, (cuuint64_t)p.N, (cuuint64_t)p.BH};
    cuuint64_t strides[2] = {(cuuint64_t)p.D * 2, (cuuint64_t)p.N * p.D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)tc::kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemAgg = 3 * 2 * 2 * (size_t)tc::kBox + 2048 + 256;
constexpr size_t kSmemFwdCausal = 2 * 3 * 2 * (size_t)tc::kBox + 2 * (size_t)tc::kBox + 1024 + 256;
constexpr size_t kSmemFwdNonCausal = 4 * 2 * (size_t)tc::kBox + 2 * (size_t)tc::kBox + 1024 + 256;
static_assert(kSmemFwdCausal <= 232448, "forward kernel exceeds the shared-memory limit");

bool set_smem_attrs() {
    static int done = 0;
    if (done) return done > 0;
    bool ok = cudaFuncSetAttribute(tc::tc_agg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAgg) ==
                  cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemFwdCausal) == cudaSuccess &&
              cudaFuncSetAttribute(tc::tc_fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemFwdNonCausal) == cudaSuccess;
    done = ok ? 1 : -1;
    return ok;
}

bool fill_common(tc::TcParams &P, const Plan &p, unsigned char *ws) {
    const int nsm = sm_count();
    if (nsm <= 0) return false;
    P.sl.nchunk = (p.N + tc::kC - 1) / tc::kC;
    P.sl.T = (long long)p.BH * P.sl.nchunk;
    long long G = P.sl.T < nsm ? P.sl.T : nsm;
    if (G > tc::kMaxCtas) G = tc::kMaxCtas;
    // Test hook: fewer CTAs, so that small problems also exercise multi-chunk, multi-head slices.
    if (const char *env = getenv("LA_TC_MAX_CTAS")) {
        const long long cap = atoll(env);
        if (cap >= 1 && cap < G) G = cap;
    }
    P.sl.G = (int)G;
    P.N = p.N;
    P.slot_stride = p.stride;
    P.slots = (float *)(ws + p.off_states);
    P.status = (uint32_t *)ws;
    return true;
}

cudaError_t launch_agg(const tc::TcParams &P, cudaStream_t s) {
    if (!set_smem_attrs()) return cudaErrorInvalidValue;
    tc::tc_agg_kernel<<<P.sl.G, 192, kSmemAgg, s>>>(P);
    return cudaGetLastError();
}

}  // namespace tc_host

using namespace tc_host;

bool tc_supported(const Plan &p) { return p.dtype == 1 && p.D == 128; }

size_t tc_slot_bytes(const Plan &p) { return ((size_t)p.BH + tc::kMaxCtas) * (size_t)p.stride * sizeof(float); }

cudaError_t tc_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                       unsigned char *ws, cudaStream_t s) {
    if (!set_smem_attrs()) return cudaErrorInvalidValue;
    tc::TcParams P;
    memset(&P, 0, sizeof(P));
    if (!fill_common(P, p, ws)) return cudaErrorInvalidDevice;
    if (!make_map(&P.tmQ, Q, p) || !make_map(&P.tmK, K, p) || !make_map(&P.tmV, V, p)) return cudaErrorInvalidValue;
    P.O = O;
    P.g = g;
    tc::tc_agg_kernel<<<P.sl.G, 192, kSmemAgg, s>>>(P);
    if (p.causal)
        tc::tc_fwd_kernel<true><<<P.sl.G, 192, kSmemFwdCausal, s>>>(P);
    else
        tc::tc_fwd_kernel<false><<<P.sl.G, 192, kSmemFwdNonCausal, s>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(2);
    return e;
}

}  // namespace la
