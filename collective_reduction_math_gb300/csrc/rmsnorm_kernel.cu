// rmsnorm_kernel.cu -- all-reduce with the residual add and RMSNorm fused
// after the sum: "in decoding, the merge and the RMSNorm that follow are fused
// into the preceding all-reduce, so the collective absorbs a kernel" (post on
// NCCL all-reduce, "How this survives ten thousand GPUs").
//
// The buffer is rows x hidden.  A thread-block cluster of C CTAs owns a row at
// a time (a persistent grid of clusters strides over the rows); CTA c of the
// cluster takes the c-th slice of the row's columns.  With few rows (decode)
// C > 1 spreads one row over several SMs; with many rows C = 1.
//   pass 1  for every element: reduce the W contributions exactly as the
//           all-reduce kernel does (same chunks, same ring or tree order,
//           fp32), add the residual (one fp32 add), keep the fp32 h in
//           shared memory, and accumulate h*h into a per-thread fp32
//           partial (increasing element order);
//   reduce  the partials with a fixed tree: warp shuffles give the warp
//           partials, which each warp pushes into every cluster peer's shared
//           memory (DSMEM stores) before the cluster barrier; then every
//           thread adds, from its own CTA's copies, each CTA's warp partials
//           in a fixed tree and the C slice totals in cluster-rank order, so
//           every CTA -- and every run -- gets the same value;
//           inv = 1 / sqrt(ss / hidden + eps), each step one IEEE operation;
//   pass 2  out = (h * inv) * weight, rounded once, stored to all W outputs;
//           residual_out gets h rounded once, from the same fp32 h.  Pass 1
//           stores nothing to global memory, so the cluster barrier between
//           the passes has no stores to wait for, and each thread's first
//           weight vector is loaded once, before the first row.
// Whatever depends on the parameters alone (the first row's segment and the
// addresses of each thread's first vector) is worked out before the kernel
// waits on the one before it.  With one CTA per row and several rows per CTA,
// a second variant keeps two row buffers and runs pass 2 of a row in one loop
// with pass 1 of the CTA's next row, so that row's loads are in flight while
// this row's stores issue (same arithmetic, same order).
// Bytes per row: W reads and W writes of the row, plus the residual read,
// residual_out write and weight read (the weight stays in L2 across rows).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "reduce_kernel.cuh"

namespace cg = cooperative_groups;

namespace mr {

// Three resident CTAs per SM up to W = 8 (measured on GB300 at 4096 x 8192
// bf16, W = 8: 6.08 against 5.48 TB/s with the register budget left free);
// wider variants keep more registers for their W values.
template <int DT, int ALGO, int WCAP, int VB, bool PIPE>
__global__ void __launch_bounds__(kThreads, PIPE ? 2 : WCAP <= 8 ? 3 : WCAP <= 16 ? 2 : 1)
allreduce_rmsnorm_kernel(const __grid_constant__ NormParams P) {
    using A = Arith<DT, MR_SUM>;
    using raw_t = typename A::raw_t;
    constexpr int EB = Elem<DT>::kBytes;
    constexpr int LANES = VB / EB;
    static_assert(LANES % 4 == 0 || VB < 16, "vector lanes are moved to shared memory as float4");
    static_assert(kThreads == 256, "the row sum adds 8 warp partials per CTA");

    extern __shared__ float4 row_smem[];
    float* hs = reinterpret_cast<float*>(row_smem);      // this CTA's slice of the row's fp32 h
    // Every warp's partial of the row's sum of squares, by row parity and
    // cluster rank: each CTA pushes its own into every cluster peer.
    __shared__ float wpart[2][kMaxNormCluster][kThreads / 32];

    const int W = P.W;
    const uint64_t H = P.hidden;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = P.csize;                  // a power of two: divide by shifting
    const int lc = 31 - __clz(C);
    const int crank = (int)cluster.block_rank();
    const uint64_t first_row = blockIdx.x >> lc, row_stride = gridDim.x >> lc;
    // This CTA's columns: vectors [v_lo, v_hi) (vector path) or elements
    // [c_lo, c_hi) (element path).
    const uint64_t nv_all = H / LANES;
    const uint64_t v_lo = (nv_all * crank) >> lc, v_hi = (nv_all * (crank + 1)) >> lc;
    const uint64_t c_lo = (H * crank) >> lc, c_hi = (H * (crank + 1)) >> lc;

    auto input = [&](const Segment& sg, int i) -> const char* {
        return static_cast<const char*>(P.in[order_rank<ALGO>(W, sg, i)]);
    };
    auto segment_at = [&](uint64_t e, int from) {
        int s = from;
        while (e >= P.seg[s].hi) ++s;
        return s;
    };
    // The segment holding element e, from an fp32 estimate of its chunk
    // (floor(e * W / N), exact to within a chunk or two) and a short walk:
    // a walk from segment 0 chains one parameter-bank load per segment
    // passed, in front of the row's first load.
    const uint64_t n_all = P.rows * H;
    const float chunks_per_elem = (float)W / (float)n_all;
    auto segment_near = [&](uint64_t e) {
        int s = (int)((float)e * chunks_per_elem);
        s = s < 0 ? 0 : s >= P.nseg ? P.nseg - 1 : s;
        while (s > 0 && e < P.seg[s].lo) --s;
        while (e >= P.seg[s].hi) ++s;
        return s;
    };
    // One element of pass 1: returns h and writes residual_out.
    auto element_h = [&](uint64_t e, int sgi) -> float {
        const Segment& sg = P.seg[sgi];
        float y[WCAP];
#pragma unroll
        for (int i = 0; i < WCAP; ++i)
            if (i < W) y[i] = A::read(__ldg(reinterpret_cast<const raw_t*>(input(sg, i)) + e), 0.0f);
        float h = fold<A, ALGO, WCAP>(y, W);
        if (P.residual) h = __fadd_rn(h, A::read(__ldg(static_cast<const raw_t*>(P.residual) + e), 0.0f));
        return h;
    };
    // The h of one whole vector from its W loaded contributions (pass 1).
    auto vector_h = [&](uint64_t e0, const Vec<VB> (&raw)[WCAP], float (&hv)[LANES]) {
        Vec<VB> rv;
        if (P.residual) rv = load_vec<VB>(static_cast<const char*>(P.residual) + e0 * EB);
#pragma unroll
        for (int l = 0; l < LANES; ++l) {
            float y[WCAP];
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                if (i < W) y[i] = A::read(get_lane<raw_t, VB>(raw[i], l), 0.0f);
            float h = fold<A, ALGO, WCAP>(y, W);
            if (P.residual) h = __fadd_rn(h, A::read(get_lane<raw_t, VB>(rv, l), 0.0f));
            hv[l] = h;
        }
    };
    // Adds a vector's h*h to the thread's partial and keeps h in the slice
    // (row buffer b; a thread reads back only the slots it wrote).
    auto keep = [&](int b, uint64_t sv, const float (&hv)[LANES], float& ss) {
#pragma unroll
        for (int l = 0; l < LANES; ++l) ss = __fadd_rn(ss, __fmul_rn(hv[l], hv[l]));
        if constexpr (LANES % 4 == 0) {
            float4* rb = row_smem + (uint64_t)b * P.buf_f4;
#pragma unroll
            for (int q = 0; q < LANES / 4; ++q)
                rb[sv * (LANES / 4) + q] = make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
        } else {
#pragma unroll
            for (int l = 0; l < LANES; ++l) hs[sv * LANES + l] = hv[l];
        }
    };
    // Pass 1 of one whole vector v of the row at `base` (segment hint sgi).
    auto pass1_vector = [&](uint64_t base, uint64_t v, int& sgi, int b, float& ss) {
        const uint64_t e0 = base + v * LANES;
        sgi = segment_at(e0, sgi);
        float hv[LANES];
        if (e0 + LANES <= P.seg[sgi].hi) {
            const Segment& sg = P.seg[sgi];
            Vec<VB> raw[WCAP];
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                if (i < W) raw[i] = load_vec<VB>(input(sg, i) + e0 * EB);
            vector_h(e0, raw, hv);
        } else {
            // the vector straddles a chunk (or tree) boundary
#pragma unroll
            for (int l = 0; l < LANES; ++l) hv[l] = element_h(e0 + l, segment_at(e0 + l, sgi));
        }
        keep(b, v - v_lo, hv, ss);
    };

    // Before waiting on the previous kernel, everything that depends on the
    // parameters alone: the first row's segment and, up to 16 ranks, the W
    // addresses of this thread's first vector.  Its loads then issue the
    // moment the wait returns, instead of after a chain of parameter reads
    // (measured with per-phase timestamps at decode size: pass 1 ended 2.7 us
    // after the wait, most of it before the first load).
    constexpr bool kPre = WCAP <= 16;
    const char* pre[kPre ? WCAP : 1];
    bool pre_ok = false;
    int sgi_first = 0, sgi_pre = 0;
    if (first_row < P.rows) {
        const uint64_t base = first_row * H;
        sgi_first = segment_near(base + (P.vec ? v_lo * LANES : c_lo));
        if constexpr (kPre) {
            const uint64_t v = v_lo + threadIdx.x;
            if (P.vec && v < v_hi) {
                const uint64_t e0 = base + v * LANES;
                sgi_pre = segment_at(e0, sgi_first);
                if (e0 + LANES <= P.seg[sgi_pre].hi) {
                    pre_ok = true;
#pragma unroll
                    for (int i = 0; i < WCAP; ++i)
                        if (i < W) pre[i] = input(P.seg[sgi_pre], i) + e0 * EB;
                }
            }
        }
    }
    pdl_enter();

    // The first row's first vector, from those addresses (its h*h opens the
    // thread's partial for that row).
    float ss_first = 0.0f;
    if (kPre && pre_ok) {
        const uint64_t e0 = first_row * H + (v_lo + threadIdx.x) * LANES;
        Vec<VB> raw[WCAP];
#pragma unroll
        for (int i = 0; i < WCAP; ++i)
            if (i < W) raw[i] = load_vec<VB>(pre[i]);
        float hv[LANES];
        vector_h(e0, raw, hv);
        keep(0, threadIdx.x, hv, ss_first);
    }

    // This thread's first pass-2 weight vector: the same for every row.
    Vec<VB> w_first;
    if (P.vec && v_lo + threadIdx.x < v_hi)
        w_first = load_vec<VB>(static_cast<const char*>(P.weight) + (v_lo + threadIdx.x) * VB);

    // ---- the row's sum of squares, in a fixed tree -------------------------
    // Warp shuffles give each warp's partial, which the warp pushes into every
    // cluster peer's slot for (this CTA, this warp): a shared-memory store
    // each, remote but for the CTA itself; the cluster barrier's release makes
    // them visible.  After the barrier every thread adds, from its own CTA's
    // copies, each CTA's 8 warp partials in one fixed tree,
    // ((w0 + w4) + (w2 + w6)) + ((w1 + w5) + (w3 + w7)), then the C slice
    // totals in cluster-rank order: every CTA -- and every run -- gets the
    // same sum, with no remote read and no second barrier.  The slots
    // alternate by row parity, so a fast CTA's next row cannot overwrite a slot
    // a peer is still reading: it would first need that peer at the next row's
    // barrier.  Returns inv = 1 / sqrt(ss / hidden + eps).
    auto row_inv = [&](float ss, int parity) -> float {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_down_sync(0xffffffffu, ss, o));
        ss = __shfl_sync(0xffffffffu, ss, 0);
        if (lane < C) {
            if (C == 1) wpart[parity][0][warp] = ss;
            else *cluster.map_shared_rank(&wpart[parity][crank][warp], lane) = ss;
        }
        if (C > 1) cluster.sync();
        else __syncthreads();
        float row_ss = 0.0f;
        for (int r = 0; r < C; ++r) {
            const float* q = wpart[parity][r];
            const float t = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[4]), __fadd_rn(q[2], q[6])),
                                      __fadd_rn(__fadd_rn(q[1], q[5]), __fadd_rn(q[3], q[7])));
            row_ss = __fadd_rn(row_ss, t);
        }
        return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(row_ss, (float)H), P.eps)));
    };

    // ---- pass 2 of one vector v of the row at `base`, h from row buffer b ----
    auto pass2_vector = [&](uint64_t base, uint64_t v, int b, float inv) {
        const uint64_t sv = v - v_lo;
        float hv[LANES];
        if constexpr (LANES % 4 == 0) {
            const float4* rb = row_smem + (uint64_t)b * P.buf_f4;
#pragma unroll
            for (int q = 0; q < LANES / 4; ++q) {
                const float4 f = rb[sv * (LANES / 4) + q];
                hv[4 * q] = f.x;
                hv[4 * q + 1] = f.y;
                hv[4 * q + 2] = f.z;
                hv[4 * q + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int l = 0; l < LANES; ++l) hv[l] = hs[sv * LANES + l];
        }
        const Vec<VB> wv = (v == v_lo + threadIdx.x) ? w_first
                                                      : load_vec<VB>(static_cast<const char*>(P.weight) + v * VB);
        Vec<VB> o;
#pragma unroll
        for (int l = 0; l < LANES; ++l)
            set_lane<raw_t, VB>(o, l, A::post(__fmul_rn(__fmul_rn(hv[l], inv),
                                                        A::read(get_lane<raw_t, VB>(wv, l), 0.0f)), W));
        const uint64_t off = (base + v * LANES) * EB;
        if (P.residual_out) {
            Vec<VB> ro;
#pragma unroll
            for (int l = 0; l < LANES; ++l) set_lane<raw_t, VB>(ro, l, A::post(hv[l], W));
            store_vec<VB>(static_cast<char*>(P.residual_out) + off, ro);
        }
#pragma unroll
        for (int j = 0; j < WCAP; ++j)
            if (j < W) store_vec<VB>(static_cast<char*>(P.out[j]) + off, o);
    };

    if constexpr (PIPE) {
        // One CTA per row, two row buffers: pass 2 of a row runs in one loop
        // with pass 1 of this CTA's next row, so that row's loads are in flight
        // while this row's stores issue.  Each row's arithmetic and its
        // partials' order are those of the loop below.  Built for 2 CTAs per
        // SM: at the 80 registers of 3 per SM the loop spills and runs slower
        // than the plain row loop.
        uint64_t row = first_row;
        float ss = 0.0f;
        if (row < P.rows) {
            const uint64_t base = row * H;
            const bool peeled = kPre && pre_ok;
            int sgi = peeled ? sgi_pre : sgi_first;
            ss = peeled ? ss_first : 0.0f;
            for (uint64_t v = v_lo + threadIdx.x + (peeled ? kThreads : 0); v < v_hi; v += kThreads)
                pass1_vector(base, v, sgi, 0, ss);
        }
        for (int parity = 0, b = 0; row < P.rows; row += row_stride, parity ^= 1, b ^= 1) {
            const float inv = row_inv(ss, parity);
            const uint64_t next = row + row_stride;
            const uint64_t base = row * H, nbase = next * H;
            int sgi = next < P.rows ? segment_near(nbase + v_lo * LANES) : 0;
            float ss_next = 0.0f;
            for (uint64_t v = v_lo + threadIdx.x; v < v_hi; v += kThreads) {
                if (next < P.rows) pass1_vector(nbase, v, sgi, b ^ 1, ss_next);
                pass2_vector(base, v, b, inv);
            }
            ss = ss_next;
        }
        return;
    } else {

    int parity = 0;
    for (uint64_t row = first_row; row < P.rows; row += row_stride, parity ^= 1) {
        const uint64_t base = row * H;
        const bool peeled = kPre && pre_ok && row == first_row;     // its first vector is done
        int sgi = row != first_row ? segment_near(base + (P.vec ? v_lo * LANES : c_lo))
                : peeled ? sgi_pre : sgi_first;
        float ss = peeled ? ss_first : 0.0f;

        // ---- pass 1 -------------------------------------------------------
        if (P.vec) {
            for (uint64_t v = v_lo + threadIdx.x + (peeled ? kThreads : 0); v < v_hi; v += kThreads)
                pass1_vector(base, v, sgi, 0, ss);
        } else {
            for (uint64_t i = c_lo + threadIdx.x; i < c_hi; i += kThreads) {
                const uint64_t e = base + i;
                sgi = segment_at(e, sgi);
                const float h = element_h(e, sgi);
                hs[i - c_lo] = h;
                ss = __fadd_rn(ss, __fmul_rn(h, h));
            }
        }

        const float inv = row_inv(ss, parity);

        // ---- pass 2 -------------------------------------------------------
        if (P.vec) {
            for (uint64_t v = v_lo + threadIdx.x; v < v_hi; v += kThreads) pass2_vector(base, v, 0, inv);
        } else {
            for (uint64_t i = c_lo + threadIdx.x; i < c_hi; i += kThreads) {
                const float w = A::read(__ldg(static_cast<const raw_t*>(P.weight) + i), 0.0f);
                if (P.residual_out) static_cast<raw_t*>(P.residual_out)[base + i] = A::post(hs[i - c_lo], W);
                const raw_t o = A::post(__fmul_rn(__fmul_rn(hs[i - c_lo], inv), w), W);
#pragma unroll
                for (int j = 0; j < WCAP; ++j)
                    if (j < W) static_cast<raw_t*>(P.out[j])[base + i] = o;
            }
        }
        __syncthreads();    // the row buffer and the partials are reused by the next row
    }
    }
    // No barrier at exit: peers write into this CTA's shared memory only
    // before a row's cluster barrier, which this CTA has passed, and never
    // read it.
}

template <int DT, int ALGO, int WCAP, int VB, bool PIPE>
static cudaError_t launch_one(const NormParams& P, dim3 grid, size_t smem, cudaStream_t s) {
    auto k = allreduce_rmsnorm_kernel<DT, ALGO, WCAP, VB, PIPE>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(k, grid, smem, s, (unsigned)P.csize, P);
}

template <int DT, int ALGO>
static cudaError_t launch_algo(const NormParams& P, dim3 grid, size_t smem, cudaStream_t s) {
    if (P.pipe) {
        if (P.W <= 8) return launch_one<DT, ALGO, 8, 16, true>(P, grid, smem, s);
        return launch_one<DT, ALGO, 16, 16, true>(P, grid, smem, s);
    }
    if (P.W <= 8) return launch_one<DT, ALGO, 8, 16, false>(P, grid, smem, s);
    if (P.W <= 16) return launch_one<DT, ALGO, 16, 16, false>(P, grid, smem, s);
    return launch_one<DT, ALGO, 64, 4, false>(P, grid, smem, s);
}

cudaError_t launch_allreduce_rmsnorm(const NormParams& P, int dtype, int algo, dim3 grid, size_t smem,
                                     cudaStream_t s) {
    if (dtype == MR_FP32)
        return algo == MR_RING ? launch_algo<MR_FP32, MR_RING>(P, grid, smem, s)
                               : launch_algo<MR_FP32, MR_TREE>(P, grid, smem, s);
    if (dtype == MR_BF16)
        return algo == MR_RING ? launch_algo<MR_BF16, MR_RING>(P, grid, smem, s)
                               : launch_algo<MR_BF16, MR_TREE>(P, grid, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace mr
