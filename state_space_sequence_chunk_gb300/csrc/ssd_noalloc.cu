// ssd_noalloc.cu -- ssd_fwd without a caller-supplied workspace, for callers
// that cannot allocate device memory: a host framework that owns all device
// memory and hands out only fixed buffers, a latency-critical loop that must
// not call cudaMalloc/cudaFree (they can synchronise the device and take
// driver-wide locks), or a process whose memory is fully reserved by a pool.
// The scratch lives in one static device array of SSD_NOALLOC_WORKSPACE_BYTES;
// include/ssd.h states the contract.
#include <mutex>

#include "ssd_internal.cuh"

namespace {

// The scratch buffer.  In host code its name is only a stand-in for the
// device symbol, never a device address: the address is looked up with
// cudaGetSymbolAddress, once per device.
__device__ __align__(256) unsigned char g_noalloc_ws[SSD_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_ws_addr[kMaxDevices];  // device address of g_noalloc_ws, per device ordinal

// Device address of the static array on the current device (looked up on the
// first call for that device).  Returns nullptr if the lookup fails.
void* static_workspace(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ws_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_ws_addr[dev] = p;
    }
    return g_ws_addr[dev];
}

}  // namespace

extern "C" ssd_status ssd_fwd_noalloc(const ssd_dims* d, const void* x, const float* dt,
                                      const float* A, const void* B, const void* C,
                                      const float* D, const float* init_state, void* y,
                                      float* final_state, void* stream) {
    if (!d) return SSD_ERR_NULL;
    const size_t need = ssd_fwd_workspace_bytes(d);
    if (need == 0)  // invalid sizes (ssd_fwd reports which) or an empty problem
        return ssd_fwd(d, x, dt, A, B, C, D, init_state, y, final_state, nullptr, 0, stream);
    if (need > SSD_NOALLOC_WORKSPACE_BYTES) return SSD_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
    void* ws = static_workspace(dev);
    if (!ws) return SSD_ERR_CUDA;
    return ssd_fwd(d, x, dt, A, B, C, D, init_state, y, final_state, ws,
                   SSD_NOALLOC_WORKSPACE_BYTES, stream);
}
