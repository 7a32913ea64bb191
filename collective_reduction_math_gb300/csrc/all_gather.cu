// all_gather.cu -- the all-gather kernel: every shard is written to all W
// output buffers ("All-gather: everyone shows their piece", FSDP collectives
// 101).  A pure copy, no arithmetic: it reads N*b bytes and writes W*N*b bytes.
//
// Shard k is cut into tiles of kThreads * kGatherUnroll 16-byte vectors; tiles
// are dealt round-robin across the shards (tile t is tile t / W of shard
// t % W) and a 1-D grid of kGatherBlocksPerSm CTAs per SM strides over them.
// Each thread loads its kGatherUnroll vectors of shard k first, so that many
// independent loads are in flight, then stores each one, with streaming
// stores, at offset k*C of every rank's output.  Shards whose byte size or
// pointers are not 16-byte aligned are copied one element per thread.
#include <stdint.h>

#include "mr_internal.h"

namespace mr {

__global__ void __launch_bounds__(kThreads)
all_gather_kernel(const __grid_constant__ GatherParams P) {
    pdl_enter();
    const int W = P.W;
    const uint64_t shard_bytes = P.C * (uint64_t)P.esize;

    if (P.vec) {
        constexpr uint64_t kTile = (uint64_t)kThreads * kGatherUnroll;
        const uint64_t nv = shard_bytes / 16;
        const uint64_t ntiles = ((nv + kTile - 1) / kTile) * (uint64_t)W;
        for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int k = (int)(t % (uint64_t)W);
            const uint64_t v0 = (t / (uint64_t)W) * kTile + threadIdx.x;
            const char* src = static_cast<const char*>(P.in[k]);
            const uint64_t dst_off = (uint64_t)k * shard_bytes;
            uint32_t x[kGatherUnroll][4];
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const uint64_t v = v0 + (uint64_t)u * kThreads;
                if (v < nv)
                    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                        : "=r"(x[u][0]), "=r"(x[u][1]), "=r"(x[u][2]), "=r"(x[u][3]) : "l"(src + v * 16));
            }
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const uint64_t v = v0 + (uint64_t)u * kThreads;
                if (v >= nv) break;
#pragma unroll 4
                for (int j = 0; j < W; ++j) {
                    char* dst = static_cast<char*>(P.out[j]) + dst_off + v * 16;
                    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                                 :: "l"(dst), "r"(x[u][0]), "r"(x[u][1]), "r"(x[u][2]), "r"(x[u][3]) : "memory");
                }
            }
        }
    } else {
        // Element by element: shard after shard, kThreads elements per tile.
        const uint64_t per = (P.C + kThreads - 1) / kThreads;
        const uint64_t ntiles = per * (uint64_t)W;
        for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int k = (int)(t / per);
            const uint64_t i = (t % per) * kThreads + threadIdx.x;
            if (i >= P.C) continue;
            const uint64_t at = (uint64_t)k * P.C + i;
            if (P.esize == 4) {
                const uint32_t x = __ldg(static_cast<const uint32_t*>(P.in[k]) + i);
                for (int j = 0; j < W; ++j) static_cast<uint32_t*>(P.out[j])[at] = x;
            } else {
                const uint16_t x = __ldg(static_cast<const uint16_t*>(P.in[k]) + i);
                for (int j = 0; j < W; ++j) static_cast<uint16_t*>(P.out[j])[at] = x;
            }
        }
    }
}

cudaError_t launch_all_gather(const GatherParams& P, dim3 grid, cudaStream_t s) {
    return launch_kernel(all_gather_kernel, grid, 0, s, 0, P);
}

}  // namespace mr
