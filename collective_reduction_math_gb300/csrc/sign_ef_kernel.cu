// sign_ef_kernel.cu -- 1-bit sign compression with error feedback, then the
// reduction ("Communication Optimization: Gradient Compression, NCCL ...":
// 1-bit SGD sends sign(g) with the scale ||g||_1 / d; with error feedback the
// compressed vector is taken of g plus the residual owed from the previous
// step, and the new residual is what was not sent).
//
// Per rank r and element e:  p = g + e_prev;  q = (p >= 0 ? +s_r : -s_r);
// e_new = p - q;  and the q are reduced across ranks like the all-reduce
// reduces its contributions (same chunks, same ring or tree order; avg
// pre-scales each q by fl32(1/W)).  s_r is the exact mean magnitude
// sum(|p_r|) / N rounded once to fp32 (ties to even).  It needs the whole
// buffer before any element can be decoded, so there are two launches:
//   sign_l1_kernel      per-block exact partial sums of |p| into a workspace:
//                       integers in units of 2^-149, so that no addition
//                       rounds and any order gives the same bits;
//   sign_ef_kernel      every CTA first adds each rank's partials (integer
//                       adds) and rounds the quotient by N to fp32 (CTA 0
//                       also writes the scales out); then decode, error
//                       update and reduction in one pass.
// HBM bytes: the first kernel reads g and e (2 W N 4); the second reads them
// again, writes e (W N 4) and the output (W N 4 for all-reduce, N 4 for
// reduce-scatter).
#include <cuda_runtime.h>

#include "reduce_kernel.cuh"

namespace mr {

// Adds |p| into a thread's exact sum.  The sum is a column of kL1Limbs
// 64-bit shared-memory slots (stride kThreads), slot c worth 2^(32c) units
// of 2^-149.  |p| = m * 2^(pos - 149) with m < 2^24, so m << (pos mod 32)
// (below 2^55) goes into slot pos / 32; a slot holds a 32-bit digit after
// normalisation and absorbs 256 such additions before it could overflow.
struct ExactL1 {
    unsigned long long* col;
    uint32_t flags = 0;     // bit 0: an infinite |p|; bit 1: a NaN
    int n = 0;              // additions since the last normalisation

    __device__ __forceinline__ void add(float p) {
        const uint32_t u = __float_as_uint(p) & 0x7FFFFFFFu;
        const uint32_t eb = u >> 23;
        if (eb == 255u) {
            flags |= (u & 0x7FFFFFu) ? 2u : 1u;
            return;
        }
        const uint32_t m = (u & 0x7FFFFFu) | (eb ? 0x800000u : 0u);
        const uint32_t pos = eb ? eb - 1u : 0u;
        col[(pos >> 5) * kThreads] += (unsigned long long)m << (pos & 31u);
    }
    // Carries up the column, leaving a 32-bit digit in every slot.
    __device__ __forceinline__ void normalize() {
        unsigned long long carry = 0;
#pragma unroll
        for (int c = 0; c < kL1Limbs; ++c) {
            const unsigned long long x = col[c * kThreads] + carry;
            col[c * kThreads] = x & 0xFFFFFFFFull;
            carry = x >> 32;
        }
        n = 0;
    }
    __device__ __forceinline__ void counted(int k) {
        n += k;
        if (n >= 256 - 4) normalize();
    }
};

__global__ void __launch_bounds__(kThreads)
sign_l1_kernel(const __grid_constant__ SignParams P) {
    __shared__ unsigned long long acc[kL1Limbs * kThreads];
    __shared__ unsigned long long blk[kL1Limbs];
    const int r = blockIdx.y, b = blockIdx.x, tid = threadIdx.x;
#pragma unroll
    for (int c = 0; c < kL1Limbs; ++c) acc[c * kThreads + tid] = 0;
    pdl_enter();
    const float* g = static_cast<const float*>(P.grad[r]);
    const float* e = static_cast<const float*>(P.err[r]);
    const uint64_t stride = (uint64_t)P.nb * kThreads;
    ExactL1 sum{acc + tid};
    uint64_t done = 0;
    if (P.l1_vec) {
        const uint64_t nv = P.N / 4;
        for (uint64_t v = (uint64_t)b * kThreads + tid; v < nv; v += stride) {
            const Vec<16> gv = load_vec<16>(reinterpret_cast<const char*>(g) + v * 16);
            const Vec<16> ev = load_vec<16>(reinterpret_cast<const char*>(e) + v * 16);
#pragma unroll
            for (int l = 0; l < 4; ++l) sum.add(__fadd_rn(__uint_as_float(gv.w[l]), __uint_as_float(ev.w[l])));
            sum.counted(4);
        }
        done = nv * 4;
    }
    for (uint64_t i = done + (uint64_t)b * kThreads + tid; i < P.N; i += stride) {
        sum.add(__fadd_rn(__ldg(g + i), __ldg(e + i)));
        sum.counted(1);
    }
    sum.normalize();
    __syncthreads();
    // The block's sum: warp w adds slot rows w, w + 8, ... over the threads
    // (integer adds, below 2^40 per row).
    const int warp = tid >> 5, lane = tid & 31;
    for (int c = warp; c < kL1Limbs; c += kThreads / 32) {
        unsigned long long s = 0;
        for (int j = lane; j < kThreads; j += 32) s += acc[c * kThreads + j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) blk[c] = s;
    }
    const int any_inf = __syncthreads_or((int)(sum.flags & 1u));
    const int any_nan = __syncthreads_or((int)(sum.flags & 2u));
    if (tid == 0) {
        uint32_t* out = P.partials + (uint64_t)r * kL1Words * (uint64_t)P.nb + b;
        unsigned long long carry = 0;
#pragma unroll
        for (int c = 0; c < kL1Limbs; ++c) {
            const unsigned long long x = blk[c] + carry;
            out[(uint64_t)c * P.nb] = (uint32_t)x;
            carry = x >> 32;
        }
        out[(uint64_t)kL1Limbs * P.nb] = (any_inf ? 1u : 0u) | (any_nan ? 2u : 0u);
    }
}

// The nearest fp32 to S / N (ties to even), S = sum_c s[c] * 2^(32c) units of
// 2^-149 (each s[c] below 2^42), N < 2^37.  The quotient is taken from the
// top 64 bits T of S: S = T * 2^k + L (L < 2^k), T = q N + r, so
// S / N = (q + f) * 2^k with 0 <= f < 1 and f > 0 exactly when r or L is
// nonzero.  For k > 0, T >= 2^63 and q >= 2^26: the rounding is decided by
// q's own bits, f only breaks an exact tie.  For k = 0 and q < 2^24 the
// result lies where fp32 is spaced 2^-149 apart (subnormals and the lowest
// normal binade), and q + r / N is rounded to an integer.
__device__ __forceinline__ float exact_mean_f32(const unsigned long long (&s)[kL1Limbs], uint32_t flags, uint64_t N) {
    if (flags & 2u) return __uint_as_float(0x7FC00000u);
    if (flags & 1u) return __uint_as_float(0x7F800000u);
    uint32_t L[kL1Limbs];
    unsigned long long carry = 0;
#pragma unroll
    for (int c = 0; c < kL1Limbs; ++c) {
        const unsigned long long x = s[c] + carry;
        L[c] = (uint32_t)x;
        carry = x >> 32;
    }
    int h = kL1Limbs - 1;
    while (h >= 0 && L[h] == 0u) --h;
    if (h < 0) return 0.0f;
    unsigned long long T;
    int k = 0;
    bool low = false;
    if (h <= 1) {
        T = ((unsigned long long)(h == 1 ? L[1] : 0u) << 32) | L[0];
    } else {
        const int d = 32 - __clz(L[h]);                     // 1..32 bits of S above limb h-1
        const unsigned long long lo64 = ((unsigned long long)L[h - 1] << 32) | L[h - 2];
        T = (lo64 >> d) | ((unsigned long long)L[h] << (64 - d));
        k = 32 * (h - 2) + d;
        low = (d == 32 ? L[h - 2] : (L[h - 2] & ((1u << d) - 1u))) != 0u;
        for (int c = 0; c < h - 2; ++c) low = low || L[c] != 0u;
    }
    const unsigned long long q = T / N, r = T % N;
    if (q < (1ull << 24)) {                                 // only with k == 0
        unsigned long long m = q;
        if (r > N - r || (r == N - r && (m & 1ull))) ++m;
        return __uint_as_float((uint32_t)m);                // m * 2^-149 (m <= 2^24)
    }
    const int sh = 64 - __clzll((long long)q) - 24;         // >= 1 bits of q below the 24 kept
    unsigned long long m = q >> sh;
    const unsigned long long rem = q & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (r != 0ull || low || (m & 1ull)))) ++m;
    int E = sh + k + 1;                                     // biased exponent of m * 2^(sh + k - 149)
    if (m == (1ull << 24)) {
        m >>= 1;
        ++E;
    }
    if (E >= 255) return __uint_as_float(0x7F800000u);
    return __uint_as_float(((uint32_t)E << 23) | ((uint32_t)m & 0x7FFFFFu));
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
    // The scales: one warp per rank; lane j adds the partials of blocks j,
    // j + 32, ... (integer adds, so the order does not matter), the lanes'
    // sums are combined across the warp, and lane 0 rounds the mean.
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int r = warp; r < W; r += kThreads / 32) {
            const uint32_t* base = P.partials + (uint64_t)r * kL1Words * (uint64_t)P.nb;
            unsigned long long s[kL1Limbs];
#pragma unroll
            for (int c = 0; c < kL1Limbs; ++c) s[c] = 0;
            uint32_t flags = 0;
            for (int b = lane; b < P.nb; b += 32) {
#pragma unroll
                for (int c = 0; c < kL1Limbs; ++c) s[c] += __ldg(base + (uint64_t)c * P.nb + b);
                flags |= __ldg(base + (uint64_t)kL1Limbs * P.nb + b);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int c = 0; c < kL1Limbs; ++c) s[c] += __shfl_xor_sync(0xffffffffu, s[c], o);
            }
            flags = __reduce_or_sync(0xffffffffu, flags);
            if (lane == 0) {
                const float sc = exact_mean_f32(s, flags, P.N);
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
