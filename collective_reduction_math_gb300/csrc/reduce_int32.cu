// reduce_int32.cu -- the fused all-reduce / reduce-scatter kernels for int32
// buffers (one translation unit per element type keeps the build parallel).
#include "reduce_kernel.cuh"

namespace mr {

cudaError_t launch_reduce_int32(const ReduceParams& P, int op, int algo, dim3 grid, cudaStream_t s) {
    return launch_reduce<MR_INT32>(P, op, algo, grid, s);
}

}  // namespace mr
