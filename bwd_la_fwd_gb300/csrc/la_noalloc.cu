// la_noalloc.cu -- la_forward_noalloc: the forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain the workspace la_forward needs: a plugin that a host framework hands
// only input and output pointers (the framework owns every allocation), latency-critical code that must
// not call cudaMalloc because it can block and synchronise the whole device, or a program whose device
// memory budget is fixed when it loads.  For them this entry point runs the same forward kernels with a
// workspace that lives in a fixed device array compiled into the library, so it allocates nothing.
//
// The first call on each device looks the array's device address up (cudaGetSymbolAddress) and clears the
// array's status header (cudaMemset, then a wait for it); make that first call before any stream capture
// begins.  Every call on a device shares the one array, so calls whose work overlaps on the GPU (different
// streams, or different host threads) race with each other.  Device-side conditions (a bounded wait that
// ran out) are recorded in the array's sticky status word, which la_noalloc_get_status reads and clears.
//
// The array below has static storage: every device on which this part of the library is loaded keeps
// LA_NOALLOC_SCRATCH_BYTES reserved until the process exits.  In host code its name is only a host-side
// stand-in for the symbol, not a device address, so the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels as an ordinary pointer.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/la.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up (and its header cleared) on the
// first use per device.  `create` false: report nullptr when the device has not been set up yet.
int scratch_for_current_device(void **out, bool create) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev] && create) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
        // the header (status word, state record) must start at zero; the forward writes everything else
        // it reads within the same call
        if (cudaMemset(p, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return LA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LA_OK;
}

}  // namespace

extern "C" int la_forward_noalloc(const void *Q, const void *K, const void *V, int causal, void *O, float *normaliser,
                                  int B, int H, int N, int D, int dtype, void *stream) {
    const size_t need = la_workspace_bytes(B, H, N, D, causal, dtype, 0);
    if (need == 0) {
        // invalid or unsupported shape: let la_forward report which, before anything is enqueued
        return la_forward(Q, K, V, causal, O, normaliser, B, H, N, D, dtype, nullptr, 0, stream);
    }
    if (need > (size_t)LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_WORKSPACE;  // beyond the fixed scratch size
    void *ws = nullptr;
    const int rc = scratch_for_current_device(&ws, true);
    if (rc != LA_OK) return rc;
    // la_forward checks every argument on the host before it enqueues anything
    return la_forward(Q, K, V, causal, O, normaliser, B, H, N, D, dtype, ws, LA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int la_noalloc_get_status(void *stream) {
    void *ws = nullptr;
    const int rc = scratch_for_current_device(&ws, false);
    if (rc != LA_OK) return rc;
    if (!ws) {  // no call has used this device's scratch yet
        return cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    }
    return la_get_status(ws, stream);
}
