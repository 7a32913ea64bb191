// reduce_bf16_tree.cu -- the fused all-reduce / reduce-scatter kernels for
// bf16 buffers in the tree order (one translation unit per element
// type and order keeps the build parallel).
#include "reduce_kernel.cuh"

namespace mr {

cudaError_t launch_reduce_bf16_tree(const ReduceParams& P, int op, dim3 grid, cudaStream_t s) {
    return launch_reduce<MR_BF16, MR_TREE, false>(P, op, grid, s);
}

}  // namespace mr
