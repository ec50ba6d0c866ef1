// la_simt.cu -- CUDA-core path of the normalised linear attention, for every supported D and for fp32
// or bf16 storage.  bf16 storage accumulates in fp32; fp32 storage accumulates (and carries its
// segment states) in fp64, because the gradients are differences of terms as large as the result
// (dQ_i = S_i dOt_i - dt_i z_i), so fp32 accumulation leaves ~1e-4 relative error on the smaller
// elements while fp64 leaves only the final rounding to fp32.  It is the path for fp32 I/O (tf32
// tensor cores are far from 1e-5) and for shapes the tensor-core kernels do not take.
//
// Method ("Transformer Based Linear Attention with Optimized GPU Kernel Implementation", sciencestack.ai
// page, TL;DR: O(N D^2) time, O(N D) memory, normalisation, analytical gradients), per head:
//   forward : S_i = sum_{j<=i} k_j v_j^T, z_i = sum k_j, a_i = sum v_j, n_i = i + 1
//             g_i = n_i + q_i . z_i,  O_i = (a_i + S_i^T q_i) / g_i            (c = 1)
//   backward: dOt_i = dO_i / g_i, dt_i = (dO_i . O_i) / g_i
//             dQ_i = S_i dOt_i - dt_i z_i
//             P_j = sum_{i>=j} q_i dOt_i^T, y_j = sum dt_i q_i, e_j = sum dOt_i
//             dK_j = P_j v_j - y_j,  dV_j = e_j + P_j^T k_j
// (non-causal: every sum runs over all rows).  Each head is cut into segments; a first kernel forms
// each segment's own D x D sum, a second turns those into exclusive prefix (or suffix) sums, and a third
// re-walks each segment row by row from its carried-in state.
#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float load_f(const float *p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// Rounds once, to nearest even, from the accumulator type to the storage type.
__device__ __forceinline__ void store_f(float *p, double x) { *p = __double2float_rn(x); }
__device__ __forceinline__ void store_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float fma_acc(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_acc(double a, double b, double c) { return fma(a, b, c); }

// Thread layout over a D x EB block of a state X[r][col]: thread t owns column col = t % EB and the
// reduction indices r = p + NP * m (p = t / EB, m < RPT).
template <int D, typename Acc>
struct Cfg {
    static constexpr int EB = D < 64 ? D : 64;  // output columns per block
    static constexpr int NP = kThreads / EB;     // parts of the reduction dimension
    static constexpr int RPT = D / NP;           // state entries per thread
    static constexpr int RB = sizeof(Acc) == 8 ? (D >= 256 ? 8 : 16) : (D >= 256 ? 16 : 32);  // staged rows
    static constexpr int NBLK = D / EB;
    static_assert(RPT >= 1 && NP * RPT == D, "bad SIMT layout");
};

enum Mode : int { kFwdO = 0, kBwdDQ = 1, kBwdDK = 2, kBwdDV = 3, kFwdDelta = 4 };
enum AggMode : int { kAggFwd = 0, kAggRev = 1 };

struct Args {
    const void *Q, *K, *V, *O, *dO;
    void *out;          // O, dQ, dK or dV
    float *g_out;       // forward: optional normaliser output
    void *rs_g;         // workspace row statistics g_i and delta_i, [BH * N] of the accumulator type
    void *rs_delta;
    void *rs_dpart;     // per-column-block partial sums of dO_i . O_i, [NBLK][BH * N]
    void *states;       // workspace segment states, [BH][nseg][stride] of the accumulator type
    Layout lq, lk, lv, lo, ldo, lout;  // operand strides (lout: the tensor `out` points to)
    long long H;
    long long N;
    long long BHN;
    long long stride;
    int nseg, seg_len, causal;
    uint32_t *status;        // workspace status word
    long long n_states;      // extents of the workspace arrays, in accumulator elements (checked in the
    long long n_rows;        // LA_CHECKED build): states, rs_g / rs_delta, rs_dpart
    long long n_dpart;
};

// Index check of the LA_CHECKED build for the workspace arrays these kernels index themselves: an index
// outside [0, n) records LA_ERR_BOUNDS (6) with the place `where` in the status word, and the caller skips
// the access (a load reads a neutral value).  The operands' element offsets come from layouts that the host
// checked against their extents.  In the normal build the check is the constant true.
__device__ __forceinline__ bool ws_ok(uint32_t *status, long long i, long long n, uint32_t where) {
#ifdef LA_CHECKED
    if (i >= 0 && i < n) return true;
    if (atomicCAS(status, 0u, 6u) == 0u) status[1] = where;
    return false;
#else
    (void)status;
    (void)i;
    (void)n;
    (void)where;
    return true;
#endif
}

// Element offset of flat head bh = b H + h of an operand with layout l.
__device__ __forceinline__ long long head_off(const Layout &l, long long bh, long long H) {
    return (bh / H) * l.sb + (bh % H) * l.sh;
}

// ------------------------------------------------------------------------------------------------
// Segment aggregate: for segment s of head bh, X = sum over its rows of u w^T plus two vector sums.
//   kAggFwd: u = k, w = v           -> S block, z = sum k, a = sum v
//   kAggRev: u = q, w = dO / g      -> P block, y = sum (delta/g) q, e = sum dO / g
// grid = (nseg * BH, NBLK); the vector sums are written by column block 0.
// ------------------------------------------------------------------------------------------------
template <typename T, typename Acc, int D, int AM>
__global__ void __launch_bounds__(kThreads) simt_aggregate(Args a) {
    using C = Cfg<D, Acc>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Acc *sU = reinterpret_cast<Acc *>(smem_raw);  // [RB][D]
    Acc *sW = sU + C::RB * D;                     // [RB][D]
    Acc *sSc = sW + C::RB * D;                    // [RB] 1/g   (rev)
    Acc *sDt = sSc + C::RB;                       // [RB] delta/g (rev)

    const int t = threadIdx.x, col = t % C::EB, p = t / C::EB;
    const int colg = blockIdx.y * C::EB + col;
    const long long bh = blockIdx.x / a.nseg;
    const int s = blockIdx.x % a.nseg;
    const long long r0 = (long long)s * a.seg_len;
    const long long r1 = min((long long)a.N, r0 + a.seg_len);
    const Layout &lu = AM == kAggFwd ? a.lk : a.lq, &lw = AM == kAggFwd ? a.lv : a.ldo;
    const T *U = (const T *)(AM == kAggFwd ? a.K : a.Q) + head_off(lu, bh, a.H);
    const T *W = (const T *)(AM == kAggFwd ? a.V : a.dO) + head_off(lw, bh, a.H);
    const Acc *rs_g = (const Acc *)a.rs_g, *rs_delta = (const Acc *)a.rs_delta;

    Acc X[C::RPT];
#pragma unroll
    for (int m = 0; m < C::RPT; ++m) X[m] = Acc(0);
    Acc vu = Acc(0), vw = Acc(0);  // vector sums for index t (t < D), block 0 only

    for (long long b0 = r0; b0 < r1; b0 += C::RB) {
        const int nb = (int)min((long long)C::RB, r1 - b0);
        if (AM == kAggRev && t < nb) {
            const long long x = bh * a.N + b0 + t;
            const bool in = ws_ok(a.status, x, a.n_rows, 0xC001);
            const Acc gi = in ? rs_g[x] : Acc(1);
            sSc[t] = Acc(1) / gi;
            sDt[t] = in ? rs_delta[x] / gi : Acc(0);
        }
        if (AM == kAggRev) __syncthreads();
        for (int idx = t; idx < C::RB * D; idx += kThreads) {
            const int r = idx / D, d = idx % D;
            Acc u = Acc(0), w = Acc(0);
            if (r < nb) {
                u = (Acc)load_f(U + (b0 + r) * lu.sn + d);
                w = (Acc)load_f(W + (b0 + r) * lw.sn + d);
                if (AM == kAggRev) w *= sSc[r];
            }
            sU[idx] = u;
            sW[idx] = w;
        }
        __syncthreads();
        for (int r = 0; r < nb; ++r) {
            const Acc wv = sW[r * D + colg];
#pragma unroll
            for (int m = 0; m < C::RPT; ++m) X[m] = fma_acc(sU[r * D + p + C::NP * m], wv, X[m]);
        }
        if (blockIdx.y == 0 && t < D) {
            for (int r = 0; r < nb; ++r) {
                if (AM == kAggFwd) {
                    vu += sU[r * D + t];
                } else {
                    vu = fma_acc(sDt[r], sU[r * D + t], vu);
                }
                vw += sW[r * D + t];
            }
        }
        __syncthreads();
    }
    const long long sbase = (bh * a.nseg + s) * a.stride;
    if (!ws_ok(a.status, sbase, a.n_states, 0xC002) ||
        !ws_ok(a.status, sbase + (long long)D * D + 2 * D - 1, a.n_states, 0xC002))
        return;
    Acc *st = (Acc *)a.states + sbase;
#pragma unroll
    for (int m = 0; m < C::RPT; ++m) st[(long long)(p + C::NP * m) * D + colg] = X[m];
    if (blockIdx.y == 0 && t < D) {
        st[(long long)D * D + t] = vu;
        st[(long long)D * D + D + t] = vw;
    }
}

// ------------------------------------------------------------------------------------------------
// Segment scan, in place over the segments of each head, for each float of the state:
//   causal, forward direction: exclusive prefix (segment s gets the sum of segments 0..s-1)
//   causal, reverse direction: exclusive suffix (segment s gets the sum of segments s+1..)
//   non-causal: every segment gets the total.
// grid = (ceil(used / 256), BH).
// ------------------------------------------------------------------------------------------------
template <typename Acc>
__global__ void __launch_bounds__(kThreads) simt_scan(Acc *states, int nseg, long long stride, long long used,
                                                      int causal, int reverse, uint32_t *status,
                                                      long long n_states) {
    const long long x = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (x >= used) return;
    const long long b0 = (long long)blockIdx.y * nseg * stride + x;
    if (!ws_ok(status, b0, n_states, 0xC003) || !ws_ok(status, b0 + (long long)(nseg - 1) * stride, n_states, 0xC003))
        return;
    Acc *base = states + b0;
    if (!causal) {
        Acc tot = Acc(0);
        for (int s = 0; s < nseg; ++s) tot += base[s * stride];
        for (int s = 0; s < nseg; ++s) base[s * stride] = tot;
        return;
    }
    Acc run = Acc(0);
    for (int k = 0; k < nseg; ++k) {
        const int s = reverse ? nseg - 1 - k : k;
        const Acc v = base[s * stride];
        base[s * stride] = run;
        run += v;
    }
}

template <typename Acc>
__device__ __forceinline__ Acc warp_dot(const Acc *x, const Acc *y, int D, int lane) {
    Acc acc = Acc(0);
    for (int d = lane; d < D; d += 32) acc = fma_acc(x[d], y[d], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// ------------------------------------------------------------------------------------------------
// Row walk of one segment from its carried-in state (workspace, after simt_scan).  Thread (col, p)
// keeps its RPT entries of the state in registers; the state is updated row by row (causal only) and
// read out through a shared-memory reduction over the NP parts.
//   kFwdO : X[d][e] = S,  u = k,      w = v,      t = q        -> O = (a + X^T q) / g
//   kBwdDQ: X[e][d] = S,  u = v,      w = k,      t = dO/g     -> dQ = X^T t - (delta/g) z
//   kBwdDK: X[e][d] = P,  u = dO/g,   w = q,      t = v        -> dK = X^T t - y      (rows reversed)
//   kBwdDV: X[d][e] = P,  u = q,      w = dO/g,   t = k        -> dV = e + X^T t      (rows reversed)
//   kFwdDelta: as kFwdO, but instead of storing O it stores, per column block, sum_e dO_ie O_ie: the
//             backward recomputes O_i in the accumulator precision rather than reading the rounded O.
// kBwdDQ sums those partials into delta_i and writes g_i and delta_i for kAggRev, kBwdDK and kBwdDV.
// grid = (nseg * BH, NBLK).
// ------------------------------------------------------------------------------------------------
template <typename T, typename Acc, int D, int MODE>
__global__ void __launch_bounds__(kThreads) simt_rows(Args a) {
    using C = Cfg<D, Acc>;
    constexpr int RB = C::RB;
    constexpr bool REV = (MODE == kBwdDK || MODE == kBwdDV);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Acc *sA = reinterpret_cast<Acc *>(smem_raw);  // u rows [RB][D]
    Acc *sB = sA + RB * D;                        // w rows
    Acc *sT = sB + RB * D;                        // t rows
    Acc *sX = sT + RB * D;                        // dQ: O rows
    Acc *sY = sX + RB * D;                        // dQ: q rows
    Acc *sRun = sY + RB * D;                      // running vector after each row: z, z, y or e
    Acc *sRun2 = sRun + RB * D;                   // forward: running a
    Acc *sRed = sRun2 + RB * D;                   // [RB][NP][EB]
    Acc *sG = sRed + RB * kThreads;
    Acc *sDt = sG + RB;

    const int t = threadIdx.x, col = t % C::EB, p = t / C::EB;
    const int lane = t & 31, warp = t >> 5;
    const int colg = blockIdx.y * C::EB + col;
    const long long N = a.N;
    const long long bh = blockIdx.x / a.nseg;
    const int s = blockIdx.x % a.nseg;
    const long long r0 = (long long)s * a.seg_len;
    const long long r1 = min(N, r0 + a.seg_len);
    const T *Qh = (const T *)a.Q + head_off(a.lq, bh, a.H), *Kh = (const T *)a.K + head_off(a.lk, bh, a.H);
    const T *Vh = (const T *)a.V + head_off(a.lv, bh, a.H), *dOh = (const T *)a.dO + head_off(a.ldo, bh, a.H);
    const long long hout = head_off(a.lout, bh, a.H);
    const long long sbase = (bh * a.nseg + s) * a.stride;
    const bool sok = ws_ok(a.status, sbase, a.n_states, 0xC004) &&
                     ws_ok(a.status, sbase + (long long)D * D + 2 * D - 1, a.n_states, 0xC004);
    const Acc *st = (const Acc *)a.states + sbase;
    Acc *rs_g = (Acc *)a.rs_g, *rs_delta = (Acc *)a.rs_delta, *rs_dpart = (Acc *)a.rs_dpart;
    constexpr bool FWD = (MODE == kFwdO || MODE == kFwdDelta);

    Acc X[C::RPT];
#pragma unroll
    for (int m = 0; m < C::RPT; ++m) {
        const int r = p + C::NP * m;
        X[m] = !sok ? Acc(0) : (FWD || MODE == kBwdDV) ? st[(long long)r * D + colg] : st[(long long)colg * D + r];
    }
    Acc run1 = Acc(0), run2 = Acc(0);
    if (t < D && sok) {
        run1 = (MODE == kBwdDV) ? st[(long long)D * D + D + t] : st[(long long)D * D + t];
        if (FWD) run2 = st[(long long)D * D + D + t];
    }

    const int nbatch = (int)((r1 - r0 + RB - 1) / RB);
    for (int bi = 0; bi < nbatch; ++bi) {
        const long long b0 = REV ? max(r0, r1 - (long long)(bi + 1) * RB) : r0 + (long long)bi * RB;
        const int nb = (int)(REV ? (r1 - (long long)bi * RB) - b0 : min((long long)RB, r1 - b0));
        if (REV) {
            if (t < nb) {
                const long long x = bh * N + b0 + t;
                const bool in = ws_ok(a.status, x, a.n_rows, 0xC005);
                const Acc gi = in ? rs_g[x] : Acc(1);
                sG[t] = gi;
                sDt[t] = in ? rs_delta[x] / gi : Acc(0);
            }
            __syncthreads();
        }
        // phase 1: stage the batch's rows in the accumulator type
        for (int idx = t; idx < RB * D; idx += kThreads) {
            const int r = idx / D, d = idx % D;
            const bool ok = r < nb;
            const long long rr = b0 + r;
            if (FWD) {
                sA[idx] = ok ? (Acc)load_f(Kh + rr * a.lk.sn + d) : Acc(0);
                sB[idx] = ok ? (Acc)load_f(Vh + rr * a.lv.sn + d) : Acc(0);
                sT[idx] = ok ? (Acc)load_f(Qh + rr * a.lq.sn + d) : Acc(0);
                if (MODE == kFwdDelta) sX[idx] = ok ? (Acc)load_f(dOh + rr * a.ldo.sn + d) : Acc(0);
            } else if (MODE == kBwdDQ) {
                sA[idx] = ok ? (Acc)load_f(Vh + rr * a.lv.sn + d) : Acc(0);
                sB[idx] = ok ? (Acc)load_f(Kh + rr * a.lk.sn + d) : Acc(0);
                sT[idx] = ok ? (Acc)load_f(dOh + rr * a.ldo.sn + d) : Acc(0);
                sY[idx] = ok ? (Acc)load_f(Qh + rr * a.lq.sn + d) : Acc(0);
            } else if (MODE == kBwdDK) {
                sA[idx] = ok ? (Acc)load_f(dOh + rr * a.ldo.sn + d) / sG[r] : Acc(0);
                sB[idx] = ok ? (Acc)load_f(Qh + rr * a.lq.sn + d) : Acc(0);
                sT[idx] = ok ? (Acc)load_f(Vh + rr * a.lv.sn + d) : Acc(0);
            } else {
                sA[idx] = ok ? (Acc)load_f(Qh + rr * a.lq.sn + d) : Acc(0);
                sB[idx] = ok ? (Acc)load_f(dOh + rr * a.ldo.sn + d) / sG[r] : Acc(0);
                sT[idx] = ok ? (Acc)load_f(Kh + rr * a.lk.sn + d) : Acc(0);
            }
        }
        __syncthreads();
        // phase 2: running vectors, in processing order
        if (t < D) {
            for (int k = 0; k < nb; ++k) {
                const int r = REV ? nb - 1 - k : k;
                if (a.causal) {
                    if (FWD) {
                        run1 += sA[r * D + t];
                        run2 += sB[r * D + t];
                    } else if (MODE == kBwdDQ) {
                        run1 += sB[r * D + t];
                    } else if (MODE == kBwdDK) {
                        run1 = fma_acc(sDt[r], sB[r * D + t], run1);
                    } else {
                        run1 += sB[r * D + t];
                    }
                }
                sRun[r * D + t] = run1;
                if (FWD) sRun2[r * D + t] = run2;
            }
        }
        __syncthreads();
        // per-row scalars of the forward-direction walks
        if (!REV) {
            for (int r = warp; r < nb; r += kThreads / 32) {
                const Acc n = a.causal ? (Acc)(b0 + r + 1) : (Acc)N;
                if (FWD) {
                    const Acc gi = n + warp_dot(sT + r * D, sRun + r * D, D, lane);
                    if (lane == 0) {
                        sG[r] = gi;
                        if (MODE == kFwdO && a.g_out && blockIdx.y == 0 &&
                            ws_ok(a.status, bh * N + b0 + r, a.n_rows, 0xC006))
                            a.g_out[bh * N + b0 + r] = (float)gi;
                    }
                } else {
                    const Acc gi = n + warp_dot(sY + r * D, sRun + r * D, D, lane);
                    Acc delta = Acc(0);
                    for (int q = 0; q < C::NBLK; ++q) {
                        const long long x = (long long)q * a.BHN + bh * N + b0 + r;
                        if (ws_ok(a.status, x, a.n_dpart, 0xC007)) delta += rs_dpart[x];
                    }
                    if (lane == 0) {
                        sG[r] = gi;
                        sDt[r] = delta / gi;
                        if (blockIdx.y == 0 && ws_ok(a.status, bh * N + b0 + r, a.n_rows, 0xC008)) {
                            rs_g[bh * N + b0 + r] = gi;
                            rs_delta[bh * N + b0 + r] = delta;
                        }
                    }
                }
            }
            __syncthreads();
            if (MODE == kBwdDQ) {
                for (int idx = t; idx < nb * D; idx += kThreads) sT[idx] = sT[idx] / sG[idx / D];
                __syncthreads();
            }
        }
        // phase 3: state update and partial read-out
        for (int k = 0; k < nb; ++k) {
            const int r = REV ? nb - 1 - k : k;
            if (a.causal) {
                const Acc wv = sB[r * D + colg];
#pragma unroll
                for (int m = 0; m < C::RPT; ++m) X[m] = fma_acc(sA[r * D + p + C::NP * m], wv, X[m]);
            }
            Acc part = Acc(0);
#pragma unroll
            for (int m = 0; m < C::RPT; ++m) part = fma_acc(sT[r * D + p + C::NP * m], X[m], part);
            sRed[(r * C::NP + p) * C::EB + col] = part;
        }
        __syncthreads();
        // phase 4: finish the rows r = p (mod NP)
        for (int r = p; r < nb; r += C::NP) {
            Acc tot = Acc(0);
#pragma unroll 4
            for (int q = 0; q < C::NP; ++q) tot += sRed[(r * C::NP + q) * C::EB + col];
            Acc v;
            if (FWD) {
                v = (sRun2[r * D + colg] + tot) / sG[r];
            } else if (MODE == kBwdDQ) {
                v = tot - sDt[r] * sRun[r * D + colg];
            } else if (MODE == kBwdDK) {
                v = tot - sRun[r * D + colg];
            } else {
                v = sRun[r * D + colg] + tot;
            }
            if (MODE == kFwdDelta) {
                sRun[r * C::EB + col] = v * sX[r * D + colg];  // sRun (z rows) is dead in phase 4
            } else {
                store_f((T *)a.out + hout + (b0 + r) * a.lout.sn + colg, v);
            }
        }
        if (MODE == kFwdDelta) {
            __syncthreads();
            if (t < nb) {
                Acc dsum = Acc(0);
                for (int c = 0; c < C::EB; ++c) dsum += sRun[t * C::EB + c];
                const long long x = (long long)blockIdx.y * a.BHN + bh * N + b0 + t;
                if (ws_ok(a.status, x, a.n_dpart, 0xC009)) rs_dpart[x] = dsum;
            }
        }
        __syncthreads();
    }
}

template <int D, typename Acc>
constexpr size_t agg_smem() {
    return (size_t)(2 * Cfg<D, Acc>::RB * D + 2 * Cfg<D, Acc>::RB) * sizeof(Acc);
}
template <int D, typename Acc>
constexpr size_t rows_smem() {
    return (size_t)(7 * Cfg<D, Acc>::RB * D + Cfg<D, Acc>::RB * kThreads + 2 * Cfg<D, Acc>::RB) * sizeof(Acc);
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

Args make_args(const Plan &p, const void *Q, const void *K, const void *V, const void *O, const void *dO,
               unsigned char *ws) {
    Args a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.dO = dO;
    a.states = ws + p.off_states;
    a.rs_g = ws + p.off_rowstats;
    a.rs_delta = ws + p.off_rowstats + (size_t)p.BH * p.N * p.acc_bytes;
    a.rs_dpart = ws + p.off_rowstats + 2 * (size_t)p.BH * p.N * p.acc_bytes;
    a.BHN = (long long)p.BH * p.N;
    a.lq = p.lay[kOpQ];
    a.lk = p.lay[kOpK];
    a.lv = p.lay[kOpV];
    a.lo = p.lay[kOpO];
    a.ldo = p.lay[kOpdO];
    a.lout = p.lay[kOpO];
    a.H = p.H;
    a.N = p.N;
    a.stride = p.stride;
    a.nseg = p.nseg;
    a.seg_len = p.seg_len;
    a.causal = p.causal;
    a.status = (uint32_t *)ws;
    a.n_states = (long long)p.BH * p.nseg * p.stride;
    a.n_rows = a.BHN;
    a.n_dpart = (long long)(p.D > 64 ? p.D / 64 : 1) * a.BHN;
    return a;
}

template <typename T, typename Acc, int D>
cudaError_t forward_impl(const Plan &p, Args a, void *O, float *g, cudaStream_t s) {
    using C = Cfg<D, Acc>;
    const dim3 grid((unsigned)(p.nseg * p.BH), C::NBLK);
    const long long used = (long long)D * D + 2 * D;
    cudaError_t e;
    if ((e = allow_smem(simt_aggregate<T, Acc, D, kAggFwd>, agg_smem<D, Acc>())) != cudaSuccess) return e;
    if ((e = allow_smem(simt_rows<T, Acc, D, kFwdO>, rows_smem<D, Acc>())) != cudaSuccess) return e;
    simt_aggregate<T, Acc, D, kAggFwd><<<grid, kThreads, agg_smem<D, Acc>(), s>>>(a);
    simt_scan<Acc><<<dim3((unsigned)((used + kThreads - 1) / kThreads), p.BH), kThreads, 0, s>>>(
        (Acc *)a.states, p.nseg, p.stride, used, p.causal, 0, a.status, a.n_states);
    a.out = O;
    a.g_out = g;
    simt_rows<T, Acc, D, kFwdO><<<grid, kThreads, rows_smem<D, Acc>(), s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(3);
    return e;
}

template <typename T, typename Acc, int D>
cudaError_t backward_impl(const Plan &p, Args a, void *dQ, void *dK, void *dV, cudaStream_t s) {
    using C = Cfg<D, Acc>;
    const dim3 grid((unsigned)(p.nseg * p.BH), C::NBLK);
    const long long used = (long long)D * D + 2 * D;
    const dim3 sgrid((unsigned)((used + kThreads - 1) / kThreads), p.BH);
    const size_t sa = agg_smem<D, Acc>(), sr = rows_smem<D, Acc>();
    cudaError_t e;
    if ((e = allow_smem(simt_aggregate<T, Acc, D, kAggFwd>, sa)) != cudaSuccess) return e;
    if ((e = allow_smem(simt_aggregate<T, Acc, D, kAggRev>, sa)) != cudaSuccess) return e;
    if ((e = allow_smem(simt_rows<T, Acc, D, kFwdDelta>, sr)) != cudaSuccess) return e;
    if ((e = allow_smem(simt_rows<T, Acc, D, kBwdDQ>, sr)) != cudaSuccess) return e;
    if ((e = allow_smem(simt_rows<T, Acc, D, kBwdDK>, sr)) != cudaSuccess) return e;
    if ((e = allow_smem(simt_rows<T, Acc, D, kBwdDV>, sr)) != cudaSuccess) return e;
    simt_aggregate<T, Acc, D, kAggFwd><<<grid, kThreads, sa, s>>>(a);
    simt_scan<Acc><<<sgrid, kThreads, 0, s>>>((Acc *)a.states, p.nseg, p.stride, used, p.causal, 0, a.status, a.n_states);
    simt_rows<T, Acc, D, kFwdDelta><<<grid, kThreads, sr, s>>>(a);
    a.out = dQ;
    a.lout = p.lay[kOpdQ];
    simt_rows<T, Acc, D, kBwdDQ><<<grid, kThreads, sr, s>>>(a);
    simt_aggregate<T, Acc, D, kAggRev><<<grid, kThreads, sa, s>>>(a);
    simt_scan<Acc><<<sgrid, kThreads, 0, s>>>((Acc *)a.states, p.nseg, p.stride, used, p.causal, 1, a.status, a.n_states);
    a.out = dK;
    a.lout = p.lay[kOpdK];
    simt_rows<T, Acc, D, kBwdDK><<<grid, kThreads, sr, s>>>(a);
    a.out = dV;
    a.lout = p.lay[kOpdV];
    simt_rows<T, Acc, D, kBwdDV><<<grid, kThreads, sr, s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(8);
    return e;
}

template <typename T, typename Acc>
cudaError_t forward_t(const Plan &p, Args a, void *O, float *g, cudaStream_t s) {
    switch (p.D) {
        case 16: return forward_impl<T, Acc, 16>(p, a, O, g, s);
        case 32: return forward_impl<T, Acc, 32>(p, a, O, g, s);
        case 64: return forward_impl<T, Acc, 64>(p, a, O, g, s);
        case 128: return forward_impl<T, Acc, 128>(p, a, O, g, s);
        case 256: return forward_impl<T, Acc, 256>(p, a, O, g, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename Acc>
cudaError_t backward_t(const Plan &p, Args a, void *dQ, void *dK, void *dV, cudaStream_t s) {
    switch (p.D) {
        case 16: return backward_impl<T, Acc, 16>(p, a, dQ, dK, dV, s);
        case 32: return backward_impl<T, Acc, 32>(p, a, dQ, dK, dV, s);
        case 64: return backward_impl<T, Acc, 64>(p, a, dQ, dK, dV, s);
        case 128: return backward_impl<T, Acc, 128>(p, a, dQ, dK, dV, s);
        case 256: return backward_impl<T, Acc, 256>(p, a, dQ, dK, dV, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t simt_forward(const Plan &p, const void *Q, const void *K, const void *V, void *O, float *g,
                         unsigned char *ws, cudaStream_t s) {
    Args a = make_args(p, Q, K, V, nullptr, nullptr, ws);
    return p.dtype == 1 ? forward_t<__nv_bfloat16, float>(p, a, O, g, s) : forward_t<float, double>(p, a, O, g, s);
}

cudaError_t simt_backward(const Plan &p, const void *Q, const void *K, const void *V, const void *O,
                          const void *dO, void *dQ, void *dK, void *dV, unsigned char *ws, cudaStream_t s) {
    Args a = make_args(p, Q, K, V, O, dO, ws);
    return p.dtype == 1 ? backward_t<__nv_bfloat16, float>(p, a, dQ, dK, dV, s)
                        : backward_t<float, double>(p, a, dQ, dK, dV, s);
}

}  // namespace la
