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
// The scratch is a file-scope __device__ array of SSM_NOALLOC_SCRATCH_BYTES
// (32 MiB, defined in ssm_scan.h).  Every GPU on which the library's device
// code has been loaded holds it until the process exits.  Host code must not
// use the array's name as a device address (on the host it only stands in for
// the symbol); the device address is looked up on every call with
// cudaGetSymbolAddress, with the caller's device current.  After the first
// call on a device that is a host-side lookup; it is not cached, so a context
// created after cudaDeviceReset (where the module can load at another
// address) never receives a stale pointer.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/ssm_scan.h"

namespace {

constexpr size_t kScratchBytes = SSM_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current context.  Returns nullptr on
// failure (the CUDA error state is cleared).  Under lazy module loading the
// first lookup in a context loads the module, which reserves the array.
void* scratch_on_current_device() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
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
