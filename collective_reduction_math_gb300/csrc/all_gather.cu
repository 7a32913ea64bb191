// all_gather.cu -- the all-gather kernel: every shard is written to all W
// output buffers ("All-gather: everyone shows their piece", FSDP collectives
// 101).  A pure copy, no arithmetic: it reads N*b bytes and writes W*N*b bytes.
//
// Shard k is cut into tiles of kThreads threads x kGatherBytesPerThread bytes;
// tiles are dealt round-robin across the shards (tile t is tile t / W of
// shard t % W) and a 1-D grid of kGatherBlocksPerSm CTAs per SM strides over
// them.  Each thread loads its vectors of shard k first, so that several
// independent loads are in flight, then stores each one, with streaming
// stores, at offset k*C of every rank's output.  The vectors are 32 bytes
// when every pointer and the shard's byte size allow it (half the store
// instructions of 16-byte vectors: the store queue is what binds here), else
// 16 bytes; shards whose byte size or pointers are not 16-byte aligned are
// copied one element per thread.
#include <stdint.h>

#include "mr_internal.h"

namespace mr {

// 16- or 32-byte vectors of one thread, loaded through the read-only path and
// stored with streaming stores.
template <int VB> struct GVec { uint32_t w[VB / 4]; };
template <int VB> __device__ __forceinline__ GVec<VB> gload(const char* p) {
    GVec<VB> v;
    if constexpr (VB == 32) {
        asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
              "=r"(v.w[7])
            : "l"(p));
    } else {
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]) : "l"(p));
    }
    return v;
}
template <int VB> __device__ __forceinline__ void gstore(char* p, const GVec<VB>& v) {
    if constexpr (VB == 32) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
                        "r"(v.w[6]), "r"(v.w[7]) : "memory");
    } else {
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                     :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]) : "memory");
    }
}

// The vector path: each thread loads kGatherBytesPerThread bytes of shard k
// (several independent loads in flight), then stores each vector at offset
// k*C of every rank's output.
template <int VB>
__device__ __forceinline__ void gather_vectors(const GatherParams& P) {
    constexpr int UNROLL = kGatherBytesPerThread / VB;
    const int W = P.W;
    const uint64_t shard_bytes = P.C * (uint64_t)P.esize;
    constexpr uint64_t kTile = (uint64_t)kThreads * UNROLL;
    const uint64_t nv = shard_bytes / VB;
    const uint64_t ntiles = ((nv + kTile - 1) / kTile) * (uint64_t)W;
    for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int k = (int)(t % (uint64_t)W);
        const uint64_t v0 = (t / (uint64_t)W) * kTile + threadIdx.x;
        const char* src = static_cast<const char*>(P.in[k]);
        const uint64_t dst_off = (uint64_t)k * shard_bytes;
        GVec<VB> x[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < nv) x[u] = gload<VB>(src + v * VB);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v >= nv) break;
#pragma unroll 4
            for (int j = 0; j < W; ++j) gstore<VB>(static_cast<char*>(P.out[j]) + dst_off + v * VB, x[u]);
        }
    }
}

__global__ void __launch_bounds__(kThreads)
all_gather_kernel(const __grid_constant__ GatherParams P) {
    pdl_enter();
    const int W = P.W;

    if (P.vec == 2) {
        gather_vectors<32>(P);
    } else if (P.vec == 1) {
        gather_vectors<16>(P);
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

cudaError_t launch_all_gather(const GatherParams& P, dim3 grid, size_t smem, cudaStream_t s) {
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(all_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(all_gather_kernel, grid, smem, s, 0, P);
}

int all_gather_resident_per_sm() {
    static int cached = 0;
    if (cached > 0) return cached;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, all_gather_kernel, kThreads, 0) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 1;
    }
    cached = n;
    return n;
}

}  // namespace mr
