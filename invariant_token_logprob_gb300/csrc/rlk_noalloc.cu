// rlk_noalloc.cu -- rlk_logprob_noalloc: the selected-token logprob for
// callers that are not allowed to allocate device memory.
//
// Who needs it: inference engines whose device memory is reserved up front by
// their own allocator (a stray cudaMalloc can fail outright or fragment the
// reserved pool), and latency-critical decode loops that must never block on
// the allocator.  Such callers cannot use rlk_logprob (it grows a cached
// workspace) and may have no buffer to hand to rlk_logprob_ws.
//
// How: the per-(row, vocabulary tile) partials that the two kernels exchange
// live in one fixed array in this file's device memory, RLK_NOALLOC_SCRATCH_BYTES
// large, reserved on every device where the library's device code is loaded
// (with lazy module loading, the devices the library has launched on) until the
// process exits.  Host code cannot use the array's name as a device address (on
// the host it only names a stand-in object), so the first call on each device
// checks the device, then looks up the array's real device address with
// cudaGetSymbolAddress while that device is current, and every call passes that
// address to the unchanged logprob path (rlk_logprob_ws).  Nothing is allocated
// or freed, by this file or by the path it calls.  The address is cached per
// device for the life of the process: after a cudaDeviceReset the module is
// loaded afresh and the array may move, so this entry point must not be used
// across a device reset.
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include <mutex>

#include "rlk.h"

// The shared scratch.  Its contents are whatever the previous call left; the
// logprob path writes every record it later reads, so nothing needs clearing.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RLK_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kScratchBytes = RLK_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 16 == 0, "scratch holds whole 16-byte partial records");

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

}  // namespace

extern "C" rlk_status rlk_logprob_noalloc(const void* hidden_bf16, const void* weight_bf16,
                                          const int32_t* targets_i32, int64_t T, int64_t H,
                                          int64_t V, float inv_temp, float* out_logp_f32,
                                          float* out_lse_f32, int32_t* out_argmax_i32,
                                          rlk_stream_t stream) {
    if (T < 0 || H < 1 || V < 1 || V > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (T == 0) return RLK_OK;
    // Refuse, before touching the device, any problem whose partials do not fit.
    if (rlk_logprob_workspace_size(T, H, V) > kScratchBytes) return RLK_ERR_WORKSPACE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RLK_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return RLK_ERR_UNSUPPORTED_DEVICE;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_ptr[dev]) {
            // One-time set-up for this (current) device.  The library holds
            // device code for compute capability 10.3 only: on any other device
            // the array does not exist, so refuse it first, with the status the
            // other entry points give.
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                    cudaSuccess) {
                cudaGetLastError();
                return RLK_ERR_UNSUPPORTED_DEVICE;
            }
            if (major != 10 || minor != 3) return RLK_ERR_UNSUPPORTED_DEVICE;
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return RLK_ERR_CUDA;
            }
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    return rlk_logprob_ws(hidden_bf16, weight_bf16, targets_i32, T, H, V, inv_temp, out_logp_f32,
                          out_lse_f32, out_argmax_i32, scratch, kScratchBytes, stream);
}
