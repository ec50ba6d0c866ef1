// la_decode.cu -- the recurrent (inference) form of the causal head: a carried state (S, z, a, n) per
// (batch, head), advanced one token at a time (la_decode_step) or by a block of tokens
// (la_state_append).
//
// Method: the causal forward of "Transformer Based Linear Attention with Optimized GPU Kernel
// Implementation" (sciencestack.ai page, TL;DR: O(N D^2) time, O(N D) memory, a normalisation scheme),
// written as a recurrence over tokens.  With S = sum_j k_j v_j^T (S[d][e] = sum_j k_j[d] v_j[e]),
// z = sum_j k_j, a = sum_j v_j and n the number of tokens taken so far, the output of token t is
//   S += k_t v_t^T,  z += k_t,  a += v_t,  n += 1,
//   g_t = n + q_t . z,  o_t = (a + S^T q_t) / g_t,
// which is row t of the causal forward (W_tj = 1 + q_t . k_j over j <= t).
//
// A step reads and writes the D x D state once and touches O(D) of everything else, so it is bound by
// HBM (or by launch latency for few heads).  Each head's S moves as up to 64 KB slabs of contiguous rows,
// one untiled TMA bulk copy each way per CTA, which keeps three slabs in flight per SM; a head whose
// state is larger than one slab (D = 256, or fp64 state at D = 128) is spread over a thread-block
// cluster, whose CTAs combine their partial sums through distributed shared memory.  Every element of
// the state is written back by the CTA that read it, so the update is safe in place.  Accumulation type:
// fp32 for bf16 I/O, fp64 for fp32 I/O (the state carries sums over many tokens).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/la.h"
#include "la_internal.h"
#include "la_sm100.cuh"

namespace cg = cooperative_groups;

namespace la {
namespace dec {

constexpr int kThreads = 256;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename Acc, typename T> __device__ __forceinline__ Acc load_acc(const T *p) { return (Acc)to_f(*p); }

// Rounds once, to nearest even, from the accumulator type to the storage type.
template <typename T, typename Acc> __device__ __forceinline__ T store_as(Acc x);
template <> __device__ __forceinline__ float store_as<float, double>(double x) { return __double2float_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 store_as<__nv_bfloat16, float>(float x) {
    return __float2bfloat16_rn(x);
}

// How a decode step spreads one head's state over the CTAs of its cluster: each CTA takes ROWS rows of S
// (at most kSlab bytes, so that it fits in shared memory next to two more CTAs on the SM), and its
// threads take 16-byte vectors of a row: CG vectors per row, RG rows at a time, RR rows each.
constexpr int kSlab = 65536;
template <typename Acc, int D> struct DecSplit {
    static constexpr int R = (int)(((long long)D * D * sizeof(Acc) + kSlab - 1) / kSlab);  // CTAs per head
    static constexpr int ROWS = D / R;
    static constexpr int VEC = 16 / (int)sizeof(Acc);
    static constexpr int CG = D / VEC;
    static constexpr int RG = kThreads / CG < ROWS ? kThreads / CG : ROWS;
    static constexpr int RR = ROWS / RG;
    static constexpr uint32_t BYTES = (uint32_t)(ROWS * D * sizeof(Acc));
    static_assert(D % R == 0 && ROWS % RG == 0 && R <= 8, "decode split");
};

// One decode step.  grid = BH * R CTAs in clusters of R (one cluster per head).  CTA r bulk-copies rows
// [r ROWS, (r + 1) ROWS) of the head's S into shared memory (one TMA transfer), updates them there
// (S += k v^T), forms its partial column sums of S^T q, and bulk-copies the rows back; rank 0 adds the
// R partials through distributed shared memory and writes o, g, z, a and n.  If any CTA's copy does not
// land within the bounded wait, no CTA of the cluster changes the head's state and o is written as NaN.
template <typename T, typename Acc, int D>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k,
                                                               const T *__restrict__ v, T *__restrict__ o,
                                                               float *__restrict__ g_out, Acc *S, Acc *z, Acc *a,
                                                               int *n) {
    using C = DecSplit<Acc, D>;
    extern __shared__ __align__(128) unsigned char slab_raw[];
    Acc *slab = (Acc *)slab_raw;  // ROWS x D, row-major, as in global memory
    __shared__ Acc qs[D], ks[D];
    __shared__ Acc red[C::RG][D];
    __shared__ Acc part[D];
    __shared__ Acc gsh;
    __shared__ uint64_t bar;
    __shared__ int landed;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const long long head = blockIdx.x / C::R;
    const int t = threadIdx.x;
    Acc *rows = S + head * D * D + (long long)rank * C::ROWS * D;
    if (t == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
        sm100::mbar_arrive_expect_tx(&bar, C::BYTES);
        sm100::bulk_load(slab, rows, C::BYTES, &bar);
    }
    for (int x = t; x < D; x += kThreads) {
        qs[x] = load_acc<Acc>(q + head * D + x);
        ks[x] = load_acc<Acc>(k + head * D + x);
    }
    if (t == 0) landed = sm100::mbar_wait(&bar, 0, 2000000000ull) ? 1 : 0;
    __syncthreads();  // q, k in shared memory; the slab has landed (or the wait gave up)
    bool ok = landed != 0;
    if constexpr (C::R > 1) {
        // the cluster updates the head's state only if every CTA's slab landed: one CTA's rows of S must not
        // advance while another's, or z, a and n, stay behind
        cluster.sync();
#pragma unroll
        for (int r = 0; r < C::R; ++r) ok = ok && *cluster.map_shared_rank(&landed, r) != 0;
    }
    const int cgi = t % C::CG, p = t / C::CG;
    if (ok && p < C::RG) {
        Acc ve[C::VEC], acc[C::VEC];
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) {
            ve[j] = load_acc<Acc>(v + head * D + cgi * C::VEC + j);
            acc[j] = 0;
        }
#pragma unroll 4
        for (int m = 0; m < C::RR; ++m) {
            const int row = p + C::RG * m, d = rank * C::ROWS + row;
            uint4 *cell = (uint4 *)(slab + (long long)row * D + cgi * C::VEC);
            uint4 raw = *cell;
            Acc *sv = (Acc *)&raw;
            const Acc kd = ks[d], qd = qs[d];
#pragma unroll
            for (int j = 0; j < C::VEC; ++j) {
                sv[j] += kd * ve[j];
                acc[j] += sv[j] * qd;
            }
            *cell = raw;
        }
#pragma unroll
        for (int j = 0; j < C::VEC; ++j) red[p][cgi * C::VEC + j] = acc[j];
    }
    sm100::fence_proxy_async_smem();  // the slab's new values, before the bulk store reads them
    __syncthreads();
    if (ok && t == 0) {
        sm100::bulk_store(rows, slab, C::BYTES);
        sm100::bulk_commit();
    }
    if (t < D) {
        Acc sum = 0;
#pragma unroll
        for (int r = 0; r < C::RG; ++r) sum += red[r][t];
        part[t] = sum;
    }
    if (rank == 0 && t < 32) {  // g = n' + q . z' (z' = z + k)
        Acc dz = 0;
        for (int x = t; x < D; x += 32) {
            const Acc zn = z[head * D + x] + ks[x];
            if (ok) z[head * D + x] = zn;
            dz += qs[x] * zn;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dz += __shfl_xor_sync(0xffffffffu, dz, off);
        if (t == 0) {
            const int nn = n[head] + 1;
            if (ok) n[head] = nn;
            gsh = (Acc)nn + dz;
        }
    }
    cluster.sync();  // every CTA's partial sums are in its shared memory
    if (rank == 0 && t < D) {
        Acc tot = part[t];
#pragma unroll
        for (int r = 1; r < C::R; ++r) tot += *cluster.map_shared_rank(&part[t], r);
        const Acc an = a[head * D + t] + load_acc<Acc>(v + head * D + t);
        if (ok) a[head * D + t] = an;
        const Acc g = gsh;
        o[head * D + t] = ok ? store_as<T, Acc>((an + tot) / g) : store_as<T, Acc>((Acc)NAN);
        if (g_out && t == 0) g_out[head] = (float)g;
    }
    cluster.sync();  // rank 0 has read every partial before any CTA of the cluster exits
    if (t == 0) {
        if (ok) sm100::bulk_wait0();                    // the state rows are written back before the CTA exits
        else sm100::mbar_wait(&bar, 0, 2000000000ull);  // a late copy lands before the slab is released
    }
}

// Appends N tokens to the state: S += K^T V, z += sum k, a += sum v, n += N, for each head.
// grid = (BH, D / TD, D / TD) with TD = min(D, 64); block = 256 threads, each owning an RT x RT block of
// the CTA's TD x TD tile of S.  Tokens are staged through shared memory TB at a time.
template <typename T, typename Acc, int D>
__global__ void __launch_bounds__(kThreads) state_append_kernel(const T *__restrict__ K, const T *__restrict__ V,
                                                                int N, Acc *S, Acc *z, Acc *a, int *n) {
    constexpr int TD = D < 64 ? D : 64;
    constexpr int OPT = TD * TD / kThreads;  // outputs per thread: 16, 4 or 1
    constexpr int RT = OPT == 16 ? 4 : (OPT == 4 ? 2 : 1);
    constexpr int CW = TD / RT;             // threads across the tile's columns
    constexpr int TB = 32;                  // tokens per stage
    static_assert(RT * RT == OPT && CW * (TD / RT) == kThreads, "thread tiling");
    __shared__ Acc Ks[TB][TD], Vs[TB][TD];
    const long long head = blockIdx.x;
    const int d0 = blockIdx.y * TD, e0 = blockIdx.z * TD;
    const int t = threadIdx.x, tx = t % CW, ty = t / CW;
    const bool do_z = blockIdx.z == 0 && tx == 0, do_a = blockIdx.y == 0 && ty == 0;
    Acc acc[RT][RT] = {};
    Acc zs[RT] = {}, as[RT] = {};
    const T *Kh = K + head * (long long)N * D, *Vh = V + head * (long long)N * D;
    for (int j0 = 0; j0 < N; j0 += TB) {
        for (int x = t; x < TB * TD; x += kThreads) {
            const int r = x / TD, c = x % TD;
            const bool in = j0 + r < N;
            Ks[r][c] = in ? load_acc<Acc>(Kh + (long long)(j0 + r) * D + d0 + c) : (Acc)0;
            Vs[r][c] = in ? load_acc<Acc>(Vh + (long long)(j0 + r) * D + e0 + c) : (Acc)0;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < TB; ++r) {
            Acc kk[RT], vv[RT];
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                kk[i] = Ks[r][ty * RT + i];
                vv[i] = Vs[r][tx * RT + i];
            }
#pragma unroll
            for (int i = 0; i < RT; ++i) {
#pragma unroll
                for (int c = 0; c < RT; ++c) acc[i][c] += kk[i] * vv[c];
                if (do_z) zs[i] += kk[i];
                if (do_a) as[i] += vv[i];
            }
        }
        __syncthreads();
    }
    Acc *Sh = S + head * D * D;
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int c = 0; c < RT; ++c) Sh[(long long)(d0 + ty * RT + i) * D + e0 + tx * RT + c] += acc[i][c];
    if (do_z)
#pragma unroll
        for (int i = 0; i < RT; ++i) z[head * D + d0 + ty * RT + i] += zs[i];
    if (do_a)
#pragma unroll
        for (int i = 0; i < RT; ++i) a[head * D + e0 + tx * RT + i] += as[i];
    if (blockIdx.y == 0 && blockIdx.z == 0 && t == 0) n[head] += N;
}

template <typename T, typename Acc, int D>
cudaError_t launch_step(const void *q, const void *k, const void *v, void *o, float *g, void *S, void *z, void *a,
                        int *n, long long BH, cudaStream_t s) {
    using C = DecSplit<Acc, D>;
    constexpr int R = C::R;
    static std::atomic<int> attr_state[kMaxDevices];  // the slab can exceed the 48 KB default window
    if (!once_per_device(attr_state, [] {
            return cudaFuncSetAttribute(decode_step_kernel<T, Acc, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)C::BYTES) == cudaSuccess;
        }))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(BH * R));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<T, Acc, D>, (const T *)q, (const T *)k, (const T *)v, (T *)o,
                              g, (Acc *)S, (Acc *)z, (Acc *)a, n);
}

template <typename T, typename Acc, int D>
cudaError_t launch_append(const void *K, const void *V, int N, void *S, void *z, void *a, int *n, long long BH,
                          cudaStream_t s) {
    constexpr int TD = D < 64 ? D : 64;
    const dim3 grid((unsigned)BH, D / TD, D / TD);
    state_append_kernel<T, Acc, D><<<grid, kThreads, 0, s>>>((const T *)K, (const T *)V, N, (Acc *)S, (Acc *)z,
                                                             (Acc *)a, n);
    return cudaGetLastError();
}

template <typename T, typename Acc>
cudaError_t step_by_d(int D, const void *q, const void *k, const void *v, void *o, float *g, void *S, void *z,
                      void *a, int *n, long long BH, cudaStream_t s) {
    switch (D) {
        case 16: return launch_step<T, Acc, 16>(q, k, v, o, g, S, z, a, n, BH, s);
        case 32: return launch_step<T, Acc, 32>(q, k, v, o, g, S, z, a, n, BH, s);
        case 64: return launch_step<T, Acc, 64>(q, k, v, o, g, S, z, a, n, BH, s);
        case 128: return launch_step<T, Acc, 128>(q, k, v, o, g, S, z, a, n, BH, s);
        default: return launch_step<T, Acc, 256>(q, k, v, o, g, S, z, a, n, BH, s);
    }
}

template <typename T, typename Acc>
cudaError_t append_by_d(int D, const void *K, const void *V, int N, void *S, void *z, void *a, int *n,
                        long long BH, cudaStream_t s) {
    switch (D) {
        case 16: return launch_append<T, Acc, 16>(K, V, N, S, z, a, n, BH, s);
        case 32: return launch_append<T, Acc, 32>(K, V, N, S, z, a, n, BH, s);
        case 64: return launch_append<T, Acc, 64>(K, V, N, S, z, a, n, BH, s);
        case 128: return launch_append<T, Acc, 128>(K, V, N, S, z, a, n, BH, s);
        default: return launch_append<T, Acc, 256>(K, V, N, S, z, a, n, BH, s);
    }
}

bool supported_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool overlap(const void *p, size_t pb, const void *q, size_t qb) {
    const uintptr_t a0 = (uintptr_t)p, b0 = (uintptr_t)q;
    return a0 < b0 + qb && b0 < a0 + pb;
}

// Shared argument checks of the two entry points: sizes, dtype, D, pointers, alignment, and that the
// state arrays overlap neither each other nor the given inputs.
int check_state(int B, int H, int D, int dtype, const void *S, const void *z, const void *a, const int *n,
                const void *const *ins, const size_t *in_bytes, int n_in) {
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || D < 1 || (long long)B * H >= (1LL << 31)) return LA_ERR_INVALID_ARG;
    if (!supported_d(D)) return LA_ERR_UNSUPPORTED;
    if (!S || !z || !a || !n) return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z) || !aligned16(a) || !aligned16(n)) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    const size_t acc = dtype == LA_F32 ? 8 : 4;
    const void *st[4] = {S, z, a, n};
    const size_t sb[4] = {(size_t)BH * D * D * acc, (size_t)BH * D * acc, (size_t)BH * D * acc, (size_t)BH * 4};
    for (int i = 0; i < 4; ++i) {
        for (int j = i + 1; j < 4; ++j)
            if (overlap(st[i], sb[i], st[j], sb[j])) return LA_ERR_INVALID_ARG;
        for (int j = 0; j < n_in; ++j)
            if (ins[j] && overlap(st[i], sb[i], ins[j], in_bytes[j])) return LA_ERR_INVALID_ARG;
    }
    return LA_OK;
}

}  // namespace dec
}  // namespace la

extern "C" {

int la_decode_step(const void *q, const void *k, const void *v, void *o, float *normaliser, void *S, void *z,
                   void *a, int *n, int B, int H, int D, int dtype, void *stream) {
    using namespace la::dec;
    if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return LA_ERR_INVALID_ARG;
    if (normaliser && !aligned16(normaliser)) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    const size_t vb = (size_t)(BH > 0 ? BH : 0) * (size_t)(D > 0 ? D : 0) * (dtype == LA_BF16 ? 2 : 4);
    const void *ins[5] = {q, k, v, o, normaliser};
    const size_t ib[5] = {vb, vb, vb, vb, (size_t)(BH > 0 ? BH : 0) * 4};
    int rc = check_state(B, H, D, dtype, S, z, a, n, ins, ib, 5);
    if (rc) return rc;
    if (BH * 8 >= (1LL << 31)) return LA_ERR_INVALID_ARG;  // grid size (at most 8 CTAs per head)
    // the outputs must not overlap the token inputs either
    if (overlap(o, vb, q, vb) || overlap(o, vb, k, vb) || overlap(o, vb, v, vb)) return LA_ERR_INVALID_ARG;
    if (normaliser && (overlap(normaliser, ib[4], q, vb) || overlap(normaliser, ib[4], k, vb) ||
                       overlap(normaliser, ib[4], v, vb) || overlap(normaliser, ib[4], o, vb)))
        return LA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const cudaError_t e = dtype == LA_BF16
                              ? step_by_d<__nv_bfloat16, float>(D, q, k, v, o, normaliser, S, z, a, n, BH, s)
                              : step_by_d<float, double>(D, q, k, v, o, normaliser, S, z, a, n, BH, s);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    la::count_launches(1);
    return LA_OK;
}

int la_state_append(const void *K, const void *V, void *S, void *z, void *a, int *n, int B, int H, int N, int D,
                    int dtype, void *stream) {
    using namespace la::dec;
    if (N < 0) return LA_ERR_INVALID_ARG;
    if (N > 0 && (!K || !V || !aligned16(K) || !aligned16(V))) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)B * H;
    if (BH > 0 && D > 0 && (long long)N * BH * D >= (1LL << 40)) return LA_ERR_INVALID_ARG;
    const size_t tb = (size_t)(BH > 0 ? BH : 0) * (size_t)N * (size_t)(D > 0 ? D : 0) * (dtype == LA_BF16 ? 2 : 4);
    const void *ins[2] = {K, V};
    const size_t ib[2] = {tb, tb};
    int rc = check_state(B, H, D, dtype, S, z, a, n, ins, ib, 2);
    if (rc) return rc;
    if (N == 0) return LA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const cudaError_t e = dtype == LA_BF16 ? append_by_d<__nv_bfloat16, float>(D, K, V, N, S, z, a, n, BH, s)
                                           : append_by_d<float, double>(D, K, V, N, S, z, a, n, BH, s);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    la::count_launches(1);
    return LA_OK;
}

}  // extern "C"
