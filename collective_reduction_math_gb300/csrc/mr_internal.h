// mr_internal.h -- kernel parameter blocks and launchers shared by the C ABI
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mr.h"

namespace mr {

constexpr int kMaxRanks = MR_MAX_RANKS;
constexpr int kMaxSegments = MR_MAX_RANKS + 1;
constexpr int kThreads = 256;       // threads per CTA for every kernel
constexpr int kBlocksPerSm = 2;     // resident CTAs per SM the reduce kernels are built for

// A run of elements with one accumulation order and one output placement:
// a chunk of the ring, or a chunk cut at the tree-1 / tree-2 boundary.
struct Segment {
    uint64_t lo, hi;    // global element range [lo, hi)
    uint64_t out_lo;    // reduce-scatter: element e goes to recv[k][e - out_lo]
    int32_t k;          // the chunk (its owner rank)
    int32_t tree;       // 0: tree 1, 1: tree 2 (tree algorithm only)
};

enum { MODE_ALLREDUCE = 0, MODE_REDUCE_SCATTER = 1 };

struct ReduceParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    Segment seg[kMaxSegments];
    int W;
    int nseg;
    int mode;
    int vec;        // 1: every pointer (and every reduce-scatter chunk start) is
                    // aligned to the vector width, so the vector path may run
    float scale;    // fl32(1/W): the float avg pre-scale
};

struct GatherParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    uint64_t C;     // elements per shard
    int W;
    int esize;      // bytes per element (2 or 4)
    int vec;        // 1: 16-byte vector path (pointers aligned, C*esize % 16 == 0)
};

// Vector width in bytes used by the reduce kernels for a given W.
inline int reduce_vector_bytes(int W) { return W <= 16 ? 16 : 4; }

cudaError_t launch_reduce_fp32(const ReduceParams& P, int op, int algo, dim3 grid, cudaStream_t s);
cudaError_t launch_reduce_bf16(const ReduceParams& P, int op, int algo, dim3 grid, cudaStream_t s);
cudaError_t launch_reduce_int32(const ReduceParams& P, int op, int algo, dim3 grid, cudaStream_t s);
cudaError_t launch_all_gather(const GatherParams& P, dim3 grid, cudaStream_t s);

}  // namespace mr
