// sign_ef_kernel.cu -- 1-bit sign compression with error feedback, then the
// reduction ("Communication Optimization: Gradient Compression, NCCL ...":
// 1-bit SGD sends sign(g) with the scale ||g||_1 / d; with error feedback the
// compressed vector is taken of g plus the residual owed from the previous
// step, and the new residual is what was not sent).
//
// Per rank r and element e:  p = g + e_prev;  q = (p >= 0 ? +s_r : -s_r);
// e_new = p - q;  and the q are reduced across ranks like the all-reduce
// reduces its contributions (same chunks, same ring or tree order; avg
// pre-scales each q by fl32(1/W)).  s_r = ||p_r||_1 / N needs the whole
// buffer before any element can be decoded, so there are two launches:
//   sign_l1_kernel      per-block partial L1 norms of p into a workspace:
//                       each thread a compensated (Neumaier) fp32 sum over
//                       its elements, then an fp64 tree over the block;
//   sign_ef_kernel      every CTA first sums each rank's partials in fp64 in
//                       one fixed order (a warp per rank) and rounds
//                       s_r = sum / N once to fp32 (CTA 0 also writes the
//                       scales out); then decode, error update and
//                       reduction in one pass.
// HBM bytes: the first kernel reads g and e (2 W N 4); the second reads them
// again, writes e (W N 4) and the output (W N 4 for all-reduce, N 4 for
// reduce-scatter).
#include <cuda_runtime.h>

#include "reduce_kernel.cuh"

namespace mr {

// Neumaier's compensated sum, every step one IEEE fp32 operation.
struct CompSum {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float a) {
        const float t = __fadd_rn(s, a);
        if (fabsf(s) >= fabsf(a)) c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), a));
        else c = __fadd_rn(c, __fadd_rn(__fsub_rn(a, t), s));
        s = t;
    }
};

__device__ __forceinline__ double block_sum_f64(double v, double* warp_part) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __dadd_rn(v, __shfl_down_sync(0xffffffffu, v, o));
    if (lane == 0) warp_part[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < kThreads / 32 ? warp_part[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = __dadd_rn(t, __shfl_down_sync(0xffffffffu, t, o));
    }
    return t;    // valid in thread 0
}

__global__ void __launch_bounds__(kThreads)
sign_l1_kernel(const __grid_constant__ SignParams P) {
    pdl_enter();
    __shared__ double warp_part[kThreads / 32];
    const int r = blockIdx.y, b = blockIdx.x;
    const float* g = static_cast<const float*>(P.grad[r]);
    const float* e = static_cast<const float*>(P.err[r]);
    const uint64_t stride = (uint64_t)P.nb * kThreads;
    CompSum acc;
    uint64_t done = 0;
    if (P.l1_vec) {
        const uint64_t nv = P.N / 4;
        for (uint64_t v = (uint64_t)b * kThreads + threadIdx.x; v < nv; v += stride) {
            const Vec<16> gv = load_vec<16>(reinterpret_cast<const char*>(g) + v * 16);
            const Vec<16> ev = load_vec<16>(reinterpret_cast<const char*>(e) + v * 16);
#pragma unroll
            for (int l = 0; l < 4; ++l)
                acc.add(fabsf(__fadd_rn(__uint_as_float(gv.w[l]), __uint_as_float(ev.w[l]))));
        }
        done = nv * 4;
    }
    for (uint64_t i = done + (uint64_t)b * kThreads + threadIdx.x; i < P.N; i += stride)
        acc.add(fabsf(__fadd_rn(__ldg(g + i), __ldg(e + i))));
    const double t = block_sum_f64(__dadd_rn((double)acc.s, (double)acc.c), warp_part);
    if (threadIdx.x == 0) P.partials[(uint64_t)r * P.nb + b] = t;
}

template <int OP, int ALGO, int WCAP, int VB>
__global__ void __launch_bounds__(kThreads, 2)
sign_ef_kernel(const __grid_constant__ SignParams P) {
    using A = Arith<MR_FP32, OP>;
    constexpr int LANES = VB / 4;
    __shared__ float scale[WCAP];
    pdl_enter();    // also orders this kernel after the partials of sign_l1_kernel

    const int W = P.W;
    const bool rs = (P.mode == MODE_REDUCE_SCATTER);
    // The scales: one warp per rank; lane j adds partials j, j+32, ... in
    // order, then a fixed butterfly over the lanes, read from lane 0 (the
    // same order on every CTA and every run).  All of a lane's loads are
    // independent, so this costs one round trip rather than nb.
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int r = warp; r < W; r += kThreads / 32) {
            double S = 0.0;
            for (int b = lane; b < P.nb; b += 32) S = __dadd_rn(S, P.partials[(uint64_t)r * P.nb + b]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) S = __dadd_rn(S, __shfl_xor_sync(0xffffffffu, S, o));
            if (lane == 0) {
                const float sc = __double2float_rn(__ddiv_rn(S, (double)P.N));
                scale[r] = sc;
                if (blockIdx.x == 0 && P.scales) P.scales[r] = sc;
            }
        }
    }
    __syncthreads();

    // Decode one element of rank rho, update its error, return its (pre-scaled) share.
    auto decode = [&](int rho, float g, float e, float* e_new) -> float {
        const float p = __fadd_rn(g, e);
        const float q = p >= 0.0f ? scale[rho] : -scale[rho];
        *e_new = __fsub_rn(p, q);
        return OP == MR_AVG ? __fmul_rn(q, P.avg) : q;
    };
    auto element = [&](const Segment& sg, uint64_t e) {
        float y[WCAP];
#pragma unroll
        for (int i = 0; i < WCAP; ++i) {
            if (i < W) {
                const int rho = order_rank<ALGO>(W, sg, i);
                float* ep = static_cast<float*>(P.err[rho]) + e;
                float en;
                y[i] = decode(rho, __ldg(static_cast<const float*>(P.grad[rho]) + e), *ep, &en);
                *ep = en;
            }
        }
        const uint32_t res = A::post(fold<A, ALGO, WCAP>(y, W), W);
        if (rs) {
            static_cast<uint32_t*>(P.out[sg.k])[e - sg.out_lo] = res;
        } else {
#pragma unroll
            for (int j = 0; j < WCAP; ++j)
                if (j < W) static_cast<uint32_t*>(P.out[j])[e] = res;
        }
    };

    if (P.vec) {
        // Vector tiles dealt round-robin across the segments, as in the
        // all-reduce kernel.  Per order position, the rank's scale s and the
        // share a decoded value contributes (s, or s * fl32(1/W) for avg; the
        // sign is applied after, which IEEE multiplication allows exactly)
        // are kept in registers while the CTA stays on one segment.
        float sc[WCAP], sh[WCAP];
        int cur = -1;
        const uint64_t ntiles = P.tiles_max * (uint64_t)P.nseg;
        for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int seg = (int)(t % (uint64_t)P.nseg);
            const uint64_t local = t / (uint64_t)P.nseg;
            if (local >= P.tile_start[seg + 1] - P.tile_start[seg]) continue;
            const Segment& sg = P.seg[seg];
            if (seg != cur) {
                cur = seg;
#pragma unroll
                for (int i = 0; i < WCAP; ++i) {
                    if (i < W) {
                        sc[i] = scale[order_rank<ALGO>(W, sg, i)];
                        sh[i] = OP == MR_AVG ? __fmul_rn(sc[i], P.avg) : sc[i];
                    }
                }
            }
            const uint64_t va = (sg.lo + LANES - 1) / LANES, vb = sg.hi / LANES;
            const uint64_t v = va + local * kThreads + threadIdx.x;
            if (v >= vb) continue;
            const uint64_t off = v * VB;
            Vec<VB> gv[WCAP], ev[WCAP];
#pragma unroll
            for (int i = 0; i < WCAP; ++i) {
                if (i < W) {
                    const int rho = order_rank<ALGO>(W, sg, i);
                    gv[i] = load_vec<VB>(static_cast<const char*>(P.grad[rho]) + off);
                    ev[i] = load_vec<VB>(static_cast<const char*>(P.err[rho]) + off);
                }
            }
            Vec<VB> res;
#pragma unroll
            for (int l = 0; l < LANES; ++l) {
                float y[WCAP];
#pragma unroll
                for (int i = 0; i < WCAP; ++i) {
                    if (i < W) {
                        // the decode above, with the scales from registers
                        const float p = __fadd_rn(__uint_as_float(gv[i].w[l]), __uint_as_float(ev[i].w[l]));
                        const bool pos = p >= 0.0f;
                        ev[i].w[l] = __float_as_uint(__fsub_rn(p, pos ? sc[i] : -sc[i]));
                        y[i] = pos ? sh[i] : -sh[i];
                    }
                }
                res.w[l] = A::post(fold<A, ALGO, WCAP>(y, W), W);
            }
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                if (i < W) store_vec<VB>(static_cast<char*>(P.err[order_rank<ALGO>(W, sg, i)]) + off, ev[i]);
            if (rs) {
                store_vec<VB>(static_cast<char*>(P.out[sg.k]) + off - sg.out_lo * 4, res);
            } else {
#pragma unroll
                for (int j = 0; j < WCAP; ++j)
                    if (j < W) store_vec<VB>(static_cast<char*>(P.out[j]) + off, res);
            }
        }
        // Heads and tails of the segments, outside whole vectors.
        for (int i = blockIdx.x; i < P.nseg; i += gridDim.x) {
            const Segment& sg = P.seg[i];
            const uint64_t va = (sg.lo + LANES - 1) / LANES, vb = sg.hi / LANES;
            const uint64_t h1 = va < vb ? va * LANES : sg.hi;
            const uint64_t t0 = va < vb ? vb * LANES : sg.hi;
            const uint64_t nh = h1 - sg.lo, n = nh + (sg.hi - t0);
            for (uint64_t x = threadIdx.x; x < n; x += kThreads) element(sg, x < nh ? sg.lo + x : t0 + (x - nh));
        }
    } else {
        const uint64_t ntiles = P.tile_start[P.nseg];
        int seg = 0;
        for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            while (t >= P.tile_start[seg + 1]) ++seg;
            const Segment& sg = P.seg[seg];
            const uint64_t e = sg.lo + (t - P.tile_start[seg]) * kThreads + threadIdx.x;
            if (e < sg.hi) element(sg, e);
        }
    }
}

cudaError_t launch_sign_l1(const SignParams& P, cudaStream_t s) {
    return launch_kernel(sign_l1_kernel, dim3((unsigned)P.nb, (unsigned)P.W, 1), 0, s, 0, P);
}

template <int OP, int ALGO>
static cudaError_t launch_ef_algo(const SignParams& P, dim3 grid, cudaStream_t s) {
    if (P.W <= 8) return launch_kernel(sign_ef_kernel<OP, ALGO, 8, 16>, grid, 0, s, 0, P);
    if (P.W <= 16) return launch_kernel(sign_ef_kernel<OP, ALGO, 16, 8>, grid, 0, s, 0, P);
    return launch_kernel(sign_ef_kernel<OP, ALGO, 64, 4>, grid, 0, s, 0, P);
}

cudaError_t launch_sign_ef(const SignParams& P, int op, int algo, dim3 grid, cudaStream_t s) {
    if (op == MR_SUM)
        return algo == MR_RING ? launch_ef_algo<MR_SUM, MR_RING>(P, grid, s) : launch_ef_algo<MR_SUM, MR_TREE>(P, grid, s);
    return algo == MR_RING ? launch_ef_algo<MR_AVG, MR_RING>(P, grid, s) : launch_ef_algo<MR_AVG, MR_TREE>(P, grid, s);
}

}  // namespace mr
