// reduce_bf16_ring_hop.cu -- the fused all-reduce / reduce-scatter kernels for
// bf16 buffers in the ring order with per-hop bf16 rounding (one translation unit per element
// type and order keeps the build parallel).
#include "reduce_kernel.cuh"

namespace mr {

cudaError_t launch_reduce_bf16_ring_hop(const ReduceParams& P, int op, dim3 grid, cudaStream_t s) {
    return launch_reduce<MR_BF16, MR_RING, true>(P, op, grid, s);
}

}  // namespace mr
