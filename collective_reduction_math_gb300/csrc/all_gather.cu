// all_gather.cu -- the all-gather kernel: every finished shard is written to
// all W output buffers ("All-gather: everyone shows their piece", FSDP
// collectives 101).  A pure copy, no arithmetic: it reads N*b bytes and writes
// W*N*b bytes.
//
// blockIdx.y picks the shard k; blockIdx.x strides over it.  Each 16-byte
// vector of shard k is loaded once and stored, with streaming stores, at
// offset k*C of every rank's output.  Shards whose byte size or pointers are
// not 16-byte aligned are copied one element per thread.
#include <stdint.h>

#include "mr_internal.h"

namespace mr {

__global__ void __launch_bounds__(kThreads)
all_gather_kernel(const __grid_constant__ GatherParams P) {
    const int k = blockIdx.y;
    const int W = P.W;
    const char* src = static_cast<const char*>(P.in[k]);
    const uint64_t shard_bytes = P.C * (uint64_t)P.esize;
    const uint64_t dst_off = (uint64_t)k * shard_bytes;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;

    if (P.vec) {
        const uint64_t nv = shard_bytes / 16;
        for (uint64_t v = tid; v < nv; v += stride) {
            uint32_t a, b, c, d;
            asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "l"(src + v * 16));
#pragma unroll 8
            for (int j = 0; j < W; ++j) {
                char* dst = static_cast<char*>(P.out[j]) + dst_off + v * 16;
                asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                             :: "l"(dst), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
            }
        }
    } else if (P.esize == 4) {
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
        for (uint64_t i = tid; i < P.C; i += stride) {
            const uint32_t x = __ldg(s32 + i);
            for (int j = 0; j < W; ++j) static_cast<uint32_t*>(P.out[j])[k * P.C + i] = x;
        }
    } else {
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
        for (uint64_t i = tid; i < P.C; i += stride) {
            const uint16_t x = __ldg(s16 + i);
            for (int j = 0; j < W; ++j) static_cast<uint16_t*>(P.out[j])[k * P.C + i] = x;
        }
    }
}

cudaError_t launch_all_gather(const GatherParams& P, dim3 grid, cudaStream_t s) {
    all_gather_kernel<<<grid, kThreads, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace mr
