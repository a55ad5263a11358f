// ssm_noalloc.cu -- ssm_scan_fwd_noalloc: the forward scan for callers that
// cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// allocate anything on the device themselves: a plug-in inside a host engine
// whose allocator owns all device memory, or a latency-bound loop that must
// not call cudaMalloc after start-up (it can synchronise the device and take
// unbounded time).  The ordinary ssm_scan_fwd needs a caller-allocated
// workspace; this entry point instead uses a fixed scratch array that lives in
// the library itself, so the call allocates nothing.
//
// The scratch is a file-scope __device__ array of kScratchBytes (32 MiB).
// Every GPU that loads this library holds it until the process exits.  Host
// code must not use the array's name as a device address (on the host it only
// stands in for the symbol); the device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/ssm_scan.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per
// device).  Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" SSM_API int ssm_scan_fwd_noalloc(const ssm_shape* shape, const void* u,
                                            const void* delta_raw, const float* A, const void* B,
                                            const void* C, const float* D, const void* z,
                                            const float* delta_bias, const float* h0, void* y,
                                            float* hL, ssm_stream_t stream) {
    const size_t need = ssm_scan_workspace_bytes(shape, 0);
    if (need == 0)  // invalid shape or dtype: report the precise code, touch nothing
        return ssm_scan_fwd(shape, u, delta_raw, A, B, C, D, z, delta_bias, h0, y, hL, nullptr,
                            0, stream);
    if (need > kScratchBytes) return SSM_ERR_WORKSPACE;
    void* scratch = scratch_on_current_device();
    if (!scratch) return SSM_ERR_CUDA;
    // The forward writes every scratch byte it reads later in the same call
    // (its first kernel also clears the status word), so the previous call's
    // contents never leak into this one.
    return ssm_scan_fwd(shape, u, delta_raw, A, B, C, D, z, delta_bias, h0, y, hL, scratch,
                        kScratchBytes, stream);
}
