// reduce_bf16_hier_hop.cu -- the fused all-reduce / reduce-scatter kernels for
// bf16 buffers in the hier order with per-hop bf16 rounding (one translation unit per element
// type and order keeps the build parallel).
#include "reduce_kernel.cuh"

namespace mr {

cudaError_t launch_reduce_bf16_hier_hop(const ReduceParams& P, int op, dim3 grid, cudaStream_t s) {
    return launch_reduce<MR_BF16, MR_HIER, true>(P, op, grid, s);
}

}  // namespace mr
