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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mr.h"
#include "mr_internal.h"

namespace {

// The scratch: 96 KiB.  A call never needs more than 2048 partials of
// kL1Words 32-bit words (88 KiB), whatever W and N are.
constexpr size_t kScratchBytes = 96 * 1024;
static_assert(mr::kSignMaxWorkspaceBytes <= kScratchBytes, "the static scratch must hold every call's partials");
static __device__ __align__(256) uint32_t g_sign_scratch[kScratchBytes / sizeof(uint32_t)];

// The array's device address, per device, tagged with the CUDA context it
// was looked up in.  Host code sees only a host-side stand-in under the
// array's name, so the address is asked of the runtime with the device
// current.  A device reset (cudaDeviceReset) destroys the context and the
// module with it; the next call finds a new context id and looks the address
// up again instead of using the old one.
constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};
Cached g_cache[kMaxDevices];
std::mutex g_cache_mutex;

using CtxGetCurrent = CUresult (*)(CUcontext*);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// The current context's unique id, through the driver entry points the
// runtime hands out (no link to the driver library).  False when there is no
// current context or the driver does not offer the calls.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrent get_current = nullptr;
    static CtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetId>(f);
        cudaGetLastError();
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

cudaError_t scratch_address(void** out, size_t* bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    *bytes = kScratchBytes;
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    Cached& c = g_cache[dev];
    unsigned long long id = 0;
    if (c.addr && current_context_id(&id) && id == c.ctx_id) {
        *out = c.addr;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sign_scratch);   // makes the device's context current
    if (e != cudaSuccess) return e;
    if (current_context_id(&id)) {
        c.ctx_id = id;
        c.addr = p;
    } else {
        c.addr = nullptr;    // no id to check a cached address against: look it up on every call
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

// Every argument is checked first, exactly as for mr_reduce_scatter_sign_ef
// (the same checks in the same order, so the same statuses; the messages name
// this entry point); only then is the static scratch located and handed over
// as the workspace.  It always holds the call's partials (see the
// static_assert above).
extern "C" mr_status_t mr_reduce_scatter_sign_ef_noalloc(const void* const* grad, void* const* err, void* const* recv,
                                                         float* scales, int W, size_t N, mr_op_t op, mr_algo_t algo,
                                                         void* stream) {
    return mr::run_sign_ef("reduce_scatter_sign_ef_noalloc", mr::MODE_REDUCE_SCATTER, grad, err, recv, scales, W, N,
                           op, algo, nullptr, 0, stream, scratch_address);
}
