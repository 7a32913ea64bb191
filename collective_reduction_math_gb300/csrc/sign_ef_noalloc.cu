// sign_ef_noalloc.cu -- the sign-compressed reduce-scatter for callers that
// cannot allocate device memory.
//
// mr_reduce_scatter_sign_ef needs a scratch workspace (the per-block L1
// partials of every rank) and asks its caller for it.  Some callers cannot
// provide one: code that runs where cudaMalloc is not available or not
// allowed -- a plugin handed only the tensors it works on, a runtime whose
// memory is owned by someone else's allocator, a latency-critical loop that
// cannot afford cudaMalloc's implicit device synchronisation.  For them this
// file keeps the scratch in one fixed array of device memory that is part of
// the library itself (loaded with it, held by every GPU that loads the
// library until the process exits), and hands its address to the existing
// reduce-scatter entry point.
#include <cuda_runtime.h>

#include <atomic>

#include "mr.h"
#include "mr_internal.h"

namespace {

// The scratch: room for W * blocks fp64 partials.  64 KiB covers every N for
// W <= 32 and, at W = 64, buffers of up to 2^20 elements per rank.
constexpr size_t kScratchBytes = 64 * 1024;
static __device__ __align__(256) double g_sign_scratch[kScratchBytes / sizeof(double)];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// The array's device address on the current device.  Host code sees only a
// host-side stand-in under the array's name, so the address is asked of the
// runtime, once per device, with that device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_sign_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" mr_status_t mr_reduce_scatter_sign_ef_noalloc(const void* const* grad, void* const* err, void* const* recv,
                                                         float* scales, int W, size_t N, mr_op_t op, mr_algo_t algo,
                                                         void* stream) {
    if (W >= 1 && W <= MR_MAX_RANKS && N > 0) {
        const size_t need = mr_sign_ef_workspace_bytes(W, N);
        if (need > kScratchBytes)
            return mr::report_error(MR_ERR_INVALID_ARGUMENT,
                                    "reduce_scatter_sign_ef_noalloc: W = %d, N = %zu needs %zu bytes of scratch; "
                                    "the static scratch holds %zu (use mr_reduce_scatter_sign_ef with a workspace)",
                                    W, N, need, kScratchBytes);
        void* scratch = nullptr;
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess)
            return mr::report_error(MR_ERR_CUDA, "reduce_scatter_sign_ef_noalloc: locating the static scratch failed: %s",
                                    cudaGetErrorString(e));
        return mr_reduce_scatter_sign_ef(grad, err, recv, scales, W, N, op, algo, scratch, kScratchBytes, stream);
    }
    // W out of range or nothing to do: the regular entry point reports it.
    return mr_reduce_scatter_sign_ef(grad, err, recv, scales, W, N, op, algo, nullptr, 0, stream);
}
