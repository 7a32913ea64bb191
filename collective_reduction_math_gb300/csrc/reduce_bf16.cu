// reduce_bf16.cu -- the fused all-reduce / reduce-scatter kernels for bf16
// buffers (one translation unit per element type keeps the build parallel).
#include "reduce_kernel.cuh"

namespace mr {

cudaError_t launch_reduce_bf16(const ReduceParams& P, int op, int algo, dim3 grid, cudaStream_t s) {
    return launch_reduce<MR_BF16>(P, op, algo, grid, s);
}

}  // namespace mr
