// reduce_kernel.cuh -- the fused reduction kernel: all-reduce (reduce-scatter
// and all-gather in one pass) and reduce-scatter over W rank buffers in one
// GPU's HBM.
//
// Per element (post on NCCL all-reduce, "What all-reduce promises" and "The
// ring, exactly as the kernel runs it"): read the W contributions, widen bf16
// to fp32, pre-scale float avg by 1/W, combine them in the planned order in
// registers, apply the postOp (bf16 rounding, integer avg divide), and store
// the result to all W outputs (all-reduce) or to the owner's shard
// (reduce-scatter).  Nothing is staged in memory between the reads and the
// writes: the partial sum lives only in registers, the way the page's fused
// receive-reduce-send primitives keep it in flight.
//
// Memory-bound: 2*W*N*b HBM bytes for all-reduce, (W+1)*N*b for
// reduce-scatter, at most W-1 combines per element.  No tensor cores.
//
// Layout of the work: the buffer is cut into segments (one chunk, or a chunk
// cut at the tree-1/tree-2 boundary), each with one accumulation order, and
// each segment into tiles of kThreads*U aligned vectors.  A 1-D grid of
// CTAs (a few per SM) strides over the tiles, dealt round-robin across the
// segments, so a tile's order is uniform across its CTA.  The unaligned head and tail of a segment
// (fewer than one vector each), and whole segments whose pointers are not
// vector-aligned, run the same arithmetic one element per thread.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "mr_internal.h"
#include "order.cuh"

namespace mr {

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------

template <int DT> struct Elem;
template <> struct Elem<MR_FP32> { using raw_t = uint32_t; using acc_t = float;    static constexpr int kBytes = 4; };
template <> struct Elem<MR_BF16> { using raw_t = uint16_t; using acc_t = float;    static constexpr int kBytes = 2; };
template <> struct Elem<MR_INT32> { using raw_t = uint32_t; using acc_t = uint32_t; static constexpr int kBytes = 4; };

// Total-order key of an fp32 value: a signed integer that orders -0 below +0
// and otherwise follows the numeric order (NaN excluded).  The map flips the
// magnitude bits of negative values and is its own inverse.
__device__ __forceinline__ int32_t f32_order_key(float x) {
    int32_t b = __float_as_int(x);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float f32_from_order_key(int32_t k) {
    return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF));
}

template <int DT, int OP> struct Arith {
    using E = Elem<DT>;
    using raw_t = typename E::raw_t;
    using acc_t = typename E::acc_t;
    // Float min and max run in the order-key domain: each contribution is
    // mapped to its key once as it is read, the fold is an integer min / max
    // (one instruction per combine), and post maps the result back.  The map
    // is a bijection that preserves the order, so this is exact.
    static constexpr bool kKeyed = DT != MR_INT32 && (OP == MR_MIN || OP == MR_MAX);

    // Read one contribution: widen, and pre-scale a float avg by fl32(1/W).
    static __device__ __forceinline__ acc_t read(raw_t x, float s) {
        if constexpr (DT == MR_INT32) {
            return x;
        } else {
            float f = (DT == MR_FP32) ? __uint_as_float(x) : __uint_as_float((uint32_t)x << 16);
            if constexpr (OP == MR_AVG) f = __fmul_rn(f, s);
            if constexpr (kKeyed) return __int_as_float(f32_order_key(f));
            return f;
        }
    }

    static __device__ __forceinline__ acc_t combine(acc_t a, acc_t b) {
        if constexpr (DT == MR_INT32) {
            if constexpr (OP == MR_SUM || OP == MR_AVG) return a + b;   // wraps mod 2^32
            if constexpr (OP == MR_PROD) return a * b;
            if constexpr (OP == MR_MIN) return (uint32_t)::min((int32_t)a, (int32_t)b);
            if constexpr (OP == MR_MAX) return (uint32_t)::max((int32_t)a, (int32_t)b);
        } else {
            if constexpr (OP == MR_SUM || OP == MR_AVG) return __fadd_rn(a, b);
            if constexpr (OP == MR_PROD) return __fmul_rn(a, b);
            if constexpr (OP == MR_MIN) return __int_as_float(::min(__float_as_int(a), __float_as_int(b)));
            if constexpr (OP == MR_MAX) return __int_as_float(::max(__float_as_int(a), __float_as_int(b)));
        }
    }

    // The op's identity element e: combine(a, e) and combine(e, a) give a,
    // bit for bit, for every integer a, and for every float a but a NaN,
    // whose payload a GPU add or multiply may make canonical (min and max,
    // folded on keys, keep even that): 0 or 1 for integer sums and products,
    // the extreme value or key for min and max, -0.0 for float sums (x + -0.0
    // = x under round-to-nearest, and -0.0 + -0.0 = -0.0), 1.0 for float
    // products.  The identity-padded tree, which relies on it, runs for int32
    // only.
    static __device__ __forceinline__ acc_t identity() {
        if constexpr (DT == MR_INT32) {
            if constexpr (OP == MR_SUM || OP == MR_AVG) return 0u;
            if constexpr (OP == MR_PROD) return 1u;
            if constexpr (OP == MR_MIN) return 0x7FFFFFFFu;
            if constexpr (OP == MR_MAX) return 0x80000000u;
        } else {
            if constexpr (OP == MR_SUM || OP == MR_AVG) return -0.0f;
            if constexpr (OP == MR_PROD) return 1.0f;
            if constexpr (OP == MR_MIN) return __int_as_float(0x7FFFFFFF);
            if constexpr (OP == MR_MAX) return __int_as_float((int)0x80000000u);
        }
    }

    // Per-hop rounding: a bf16 running total rounded to bf16 (as it would
    // cross a wire); the identity for fp32 and int32, and for min and max,
    // whose running value is always one of the bf16 contributions.
    static __device__ __forceinline__ acc_t hop(acc_t a) {
        if constexpr (DT == MR_BF16 && !kKeyed) return __uint_as_float((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) << 16);
        else return a;
    }

    // The postOp where the sum completes.
    static __device__ __forceinline__ raw_t post(acc_t a, int W) {
        if constexpr (kKeyed) a = f32_from_order_key(__float_as_int(a));
        if constexpr (DT == MR_FP32) return __float_as_uint(a);
        if constexpr (DT == MR_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(a));
        if constexpr (DT == MR_INT32) {
            if constexpr (OP == MR_AVG) return (uint32_t)((int32_t)a / W);
            return a;
        }
    }
};

// Per-hop bf16 sums on packed pairs.  With per-hop rounding a bf16 sum or avg
// adds two bf16 values in fp32 and rounds the result to bf16 at every hop.
// fp32 carries 24 significant bits, at least 2*8+1 for bf16's 8, so that
// double rounding equals the single correctly rounded bf16 sum (and below
// fp32's normal range the fp32 sum of two bf16 values is exact); one packed
// bf16x2 add therefore does two lanes' hop at once, with the same result.
struct Bf16PairSum {
    using acc_t = uint32_t;
    static __device__ __forceinline__ acc_t combine(acc_t a, acc_t b) {
        __nv_bfloat162 x, y;
        memcpy(&x, &a, 4);
        memcpy(&y, &b, 4);
        const __nv_bfloat162 r = __hadd2(x, y);
        acc_t o;
        memcpy(&o, &r, 4);
        return o;
    }
    static __device__ __forceinline__ acc_t identity() { return 0x80008000u; }   // -0.0 in both lanes
    static __device__ __forceinline__ acc_t hop(acc_t a) { return a; }
};

// bf16 min and max on packed pairs.  The 16-bit order key of a bf16 value
// (x with its 15 magnitude bits flipped when the sign bit is set) orders
// exactly as the 32-bit key of its fp32 widening, whose low half is then 0 or
// 0xFFFF with the sign; so the two lanes of a word fold as signed 16-bit
// keys, one vmin2 / vmax2 per pair, with the lane-wise fold's result.  The
// map is its own inverse.
template <int OP> struct Bf16PairKey {
    using acc_t = uint32_t;
    static __device__ __forceinline__ uint32_t key(uint32_t w) {
        return w ^ (((w >> 15) & 0x00010001u) * 0x7FFFu);
    }
    static __device__ __forceinline__ acc_t combine(acc_t a, acc_t b) {
        if constexpr (OP == MR_MIN) return __vmins2(a, b);
        else return __vmaxs2(a, b);
    }
    // The extreme signed 16-bit key in both lanes.
    static __device__ __forceinline__ acc_t identity() { return OP == MR_MIN ? 0x7FFF7FFFu : 0x80008000u; }
    static __device__ __forceinline__ acc_t hop(acc_t a) { return a; }
    // The two bf16 results: the keys mapped back, each lane then rounded to
    // bf16 from its fp32 widening in one packed conversion, as the lane-wise
    // fold's postOp does (the identity but for NaN, which the conversion
    // makes canonical).
    static __device__ __forceinline__ uint32_t post(acc_t k) {
        const uint32_t w = key(k);
        const __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        uint32_t o;
        memcpy(&o, &p, 4);
        return o;
    }
};

// ---------------------------------------------------------------------------
// The folds.  y[p] holds the contribution at order position p; only the
// first W positions are valid.  All register indices are compile-time.
// ---------------------------------------------------------------------------

// `hop`: round the running total after every combine (bf16 per-hop order).
template <class A>
__device__ __forceinline__ typename A::acc_t comb(typename A::acc_t a, typename A::acc_t b, bool hop) {
    typename A::acc_t r = A::combine(a, b);
    return hop ? A::hop(r) : r;
}

// Ring: a left fold in chunk order.
template <class A, int WCAP>
__device__ __forceinline__ typename A::acc_t fold_ring(const typename A::acc_t (&y)[WCAP], int W, bool hop) {
    typename A::acc_t a = y[0];
#pragma unroll
    for (int i = 1; i < WCAP; ++i)
        if (i < W) a = comb<A>(a, y[i], hop);
    return a;
}

// Tree: subtotals level by level (lowest set bit 2, 4, ...), so every child is
// complete before its parent uses it; each node takes its own value, then its
// lower child's subtotal, then its upper child's; the root takes its one child.
template <class A, int WCAP>
__device__ __forceinline__ typename A::acc_t fold_tree(typename A::acc_t (&y)[WCAP], int W, bool hop) {
#pragma unroll
    for (int b = 2; b < WCAP; b <<= 1) {
#pragma unroll
        for (int p = b; p < WCAP; p += 2 * b) {
            if (p < W) {
                typename A::acc_t a = comb<A>(y[p], y[p - b / 2], hop);
                bool taken = false;
#pragma unroll
                for (int h = b / 2; h >= 1; h >>= 1) {
                    if (!taken && p + h < W) {
                        a = comb<A>(a, y[p + h], hop);
                        taken = true;
                    }
                }
                y[p] = a;
            }
        }
    }
    typename A::acc_t a = y[0];
    bool taken = false;
#pragma unroll
    for (int h = WCAP / 2; h >= 1; h >>= 1) {
        if (!taken && h < W) {
            a = comb<A>(a, y[h], hop);
            taken = true;
        }
    }
    return a;
}

// The in-batch part of the batched tree fold.  Positions come
// in batches of 8, [8m, 8m+8); positions 8m+1 .. 8m+7 lie in whole subtrees
// of the batch (the subtree of a node at level b spans (p-b, p+b)), so the
// levels 2 and 4 of a batch fold on their own (y[0] is the batch head, at
// level 8 or above).  Returns the subtotal of the node that the head's
// upper-child search finds inside the batch: the largest h in {4, 2, 1}
// with h < Wb (valid when Wb >= 2).
template <class A>
__device__ __forceinline__ typename A::acc_t tree_batch_top(typename A::acc_t (&y)[8], int Wb, bool hop) {
#pragma unroll
    for (int b = 2; b < 8; b <<= 1) {
#pragma unroll
        for (int p = b; p < 8; p += 2 * b) {
            if (p < Wb) {
                typename A::acc_t a = comb<A>(y[p], y[p - b / 2], hop);
                bool taken = false;
#pragma unroll
                for (int h = b / 2; h >= 1; h >>= 1) {
                    if (!taken && p + h < Wb) {
                        a = comb<A>(a, y[p + h], hop);
                        taken = true;
                    }
                }
                y[p] = a;
            }
        }
    }
    return Wb > 4 ? y[4] : Wb > 2 ? y[2] : y[1];
}

// The batched folds, generic over what a "unit" is (one lane's value, or a
// packed pair of bf16 lanes) and where a batch comes from: load(m, Wb, raw)
// loads positions [8m, 8m + Wb) into raw[0, Wb), unit(raw[q], u) is unit u of
// one position's contribution, comb(a, b) combines two units.  The vector
// tiles and the element-wise heads and tails run the same code.

// A left fold over many positions (ring; hierarchical when HIER, gmask
// marking where each group starts): the positions come in batches of 8 and
// the fold's state -- the running group part and the total of the groups so
// far -- carries from batch to batch.  Same order, same operations as the
// position-by-position fold.
template <bool HIER, int UNITS, class T, class R, class Load, class Unit, class Comb>
__device__ __forceinline__ void batched_left_fold(int W, uint64_t gmask, Load load, Unit unit, Comb comb,
                                                  T (&part)[UNITS]) {
    T total[UNITS];
    bool have_total = false;
    for (int b0 = 0; b0 < W; b0 += 8) {
        R raw[8];
        load(b0 >> 3, min(8, W - b0), raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = b0 + i;
            if (p >= W) break;
            if (p == 0) {
#pragma unroll
                for (int u = 0; u < UNITS; ++u) part[u] = unit(raw[i], u);
            } else if (HIER && ((gmask >> p) & 1u)) {
                if (have_total) {
#pragma unroll
                    for (int u = 0; u < UNITS; ++u) total[u] = comb(total[u], part[u]);
                } else {
#pragma unroll
                    for (int u = 0; u < UNITS; ++u) total[u] = part[u];
                }
                have_total = true;
#pragma unroll
                for (int u = 0; u < UNITS; ++u) part[u] = unit(raw[i], u);
            } else {
#pragma unroll
                for (int u = 0; u < UNITS; ++u) part[u] = comb(part[u], unit(raw[i], u));
            }
        }
    }
    if (have_total) {
#pragma unroll
        for (int u = 0; u < UNITS; ++u) part[u] = comb(total[u], part[u]);
    }
}

// The tree order over many positions: each batch of 8 positions is loaded and
// folded up to its in-batch top node (top, i.e. tree_batch_top), keeping per
// batch only the head's own value and that subtotal (top_at(m, u): where
// batch m's top of unit u waits).  The heads 8m then form the same bit-trick
// tree over m (level = lowest set bit of m): a head takes its own value, then
// its lower child (the previous batch's top for m odd, else head m - B/2),
// then its upper child (head m + h for the largest h in {B/2, ..., 1} below
// the number of heads, else its own batch's top).  The root takes its one
// child.  These are fold_tree's combines in fold_tree's order.
template <int NB, int UNITS, class T, class R, class Load, class Unit, class Comb, class Top, class TopAt>
__device__ __forceinline__ void batched_tree(int W, Load load, Unit unit, Comb comb, Top top, TopAt top_at,
                                             T (&root)[UNITS]) {
    const int M = (W + 7) >> 3;
    T head[NB][UNITS];
#pragma unroll
    for (int m = 0; m < NB; ++m) {
        if (m < M) {
            const int Wb = min(8, W - 8 * m);
            R raw[8];
            load(m, Wb, raw);
#pragma unroll
            for (int u = 0; u < UNITS; ++u) {
                T y[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < Wb) y[q] = unit(raw[q], u);
                head[m][u] = y[0];
                top_at(m, u) = top(y, Wb);
            }
        }
    }
#pragma unroll
    for (int B = 1; B < NB; B <<= 1) {
#pragma unroll
        for (int m = B; m < NB; m += 2 * B) {
            if (m < M) {
#pragma unroll
                for (int u = 0; u < UNITS; ++u) {
                    T a = comb(head[m][u], B == 1 ? top_at(m - 1, u) : head[m - B / 2][u]);
                    bool taken = false;
#pragma unroll
                    for (int h = B / 2; h >= 1; h >>= 1) {
                        if (!taken && m + h < M) {
                            a = comb(a, head[m + h][u]);
                            taken = true;
                        }
                    }
                    if (!taken && 8 * m + 1 < W) a = comb(a, top_at(m, u));
                    head[m][u] = a;
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
        T a = head[0][u];
        bool taken = false;
#pragma unroll
        for (int h = NB / 2; h >= 1; h >>= 1) {
            if (!taken && h < M) {
                a = comb(a, head[h][u]);
                taken = true;
            }
        }
        root[u] = a;
    }
}

// The same tree over padded positions (the int32 trees over 16 slots take
// it): the positions past W are padded with the op's exact identity e and the
// fold runs the whole tree over NB batches of 8, with no condition on W but
// which positions to load: each head's upper child is head m + B/2 (B > 1)
// or its own batch's node 4, each in-batch node's upper child p + b/2.  A
// subtree of the padded tree whose positions all lie past W is e; one whose
// upper child's subtree is e takes, in place of the real tree's next smaller
// upper child, the padded child's lower subtree, which is that child.  So
// every node folds the real tree's operands in the real tree's order, with
// extra combines with e that change no bit: these are fold_tree's results.
template <int NB, int UNITS, class T, class R, class Load, class Unit, class Comb, class Ident, class TopAt>
__device__ __forceinline__ void batched_tree_padded(int W, Load load, Unit unit, Comb comb, Ident ident, TopAt top_at,
                                                    T (&root)[UNITS]) {
    const int M = (W + 7) >> 3;
    T head[NB][UNITS];
#pragma unroll
    for (int m = 0; m < NB; ++m) {
        if (m < M) {
            const int Wb = min(8, W - 8 * m);
            R raw[8];
            load(m, Wb, raw);
#pragma unroll
            for (int u = 0; u < UNITS; ++u) {
                T y[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) y[q] = q < Wb ? unit(raw[q], u) : ident();
                // levels 2 and 4 inside the batch
                y[2] = comb(comb(y[2], y[1]), y[3]);
                y[6] = comb(comb(y[6], y[5]), y[7]);
                y[4] = comb(comb(y[4], y[2]), y[6]);
                head[m][u] = y[0];
                top_at(m, u) = y[4];
            }
        } else {
#pragma unroll
            for (int u = 0; u < UNITS; ++u) {
                head[m][u] = ident();
                top_at(m, u) = ident();
            }
        }
    }
#pragma unroll
    for (int B = 1; B < NB; B <<= 1) {
#pragma unroll
        for (int m = B; m < NB; m += 2 * B) {
#pragma unroll
            for (int u = 0; u < UNITS; ++u) {
                T a = comb(head[m][u], B == 1 ? top_at(m - 1, u) : head[m - B / 2][u]);
                head[m][u] = comb(a, B == 1 ? top_at(m, u) : head[m + B / 2][u]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < UNITS; ++u) root[u] = NB > 1 ? comb(head[0][u], head[NB / 2][u]) : comb(head[0][u], top_at(0, u));
}

// Hierarchical: positions come group by group (gmask marks the first position
// of each group); each group's positions are folded left to right, then the
// group totals left to right.
template <class A, int WCAP>
__device__ __forceinline__ typename A::acc_t fold_hier(const typename A::acc_t (&y)[WCAP], int W, uint64_t gmask,
                                                       bool hop) {
    typename A::acc_t part = y[0], total = y[0];
    bool have_total = false;
#pragma unroll
    for (int i = 1; i < WCAP; ++i) {
        if (i < W) {
            if ((gmask >> i) & 1u) {
                total = have_total ? comb<A>(total, part, hop) : part;
                have_total = true;
                part = y[i];
            } else {
                part = comb<A>(part, y[i], hop);
            }
        }
    }
    return have_total ? comb<A>(total, part, hop) : part;
}

template <class A, int ALGO, int WCAP>
__device__ __forceinline__ typename A::acc_t fold(typename A::acc_t (&y)[WCAP], int W, bool hop = false,
                                                  uint64_t gmask = 0) {
    if constexpr (ALGO == MR_RING) return fold_ring<A, WCAP>(y, W, hop);
    else if constexpr (ALGO == MR_TREE) return fold_tree<A, WCAP>(y, W, hop);
    else return fold_hier<A, WCAP>(y, W, gmask, hop);
}

// ---------------------------------------------------------------------------
// Global memory access
// ---------------------------------------------------------------------------

template <int VB> struct Vec { uint32_t w[VB / 4]; };

// Inputs are read once and never re-read: read-only path, no L1 allocation.
template <int VB> __device__ __forceinline__ Vec<VB> load_vec(const char* p) {
    Vec<VB> v;
    if constexpr (VB == 16) {
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]) : "l"(p));
    } else if constexpr (VB == 8) {
        asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.w[0]), "=r"(v.w[1]) : "l"(p));
    } else {
        asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    }
    return v;
}

// Outputs are written once: streaming (evict-first) stores.
template <int VB> __device__ __forceinline__ void store_vec(char* p, const Vec<VB>& v) {
    if constexpr (VB == 16) {
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                     :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]) : "memory");
    } else if constexpr (VB == 8) {
        asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(v.w[0]), "r"(v.w[1]) : "memory");
    } else {
        asm volatile("st.global.cs.u32 [%0], %1;" :: "l"(p), "r"(v.w[0]) : "memory");
    }
}

template <class raw_t, int VB> __device__ __forceinline__ raw_t get_lane(const Vec<VB>& v, int l) {
    if constexpr (sizeof(raw_t) == 4) return v.w[l];
    else return (raw_t)(v.w[l >> 1] >> (16 * (l & 1)));
}

template <class raw_t, int VB> __device__ __forceinline__ void set_lane(Vec<VB>& v, int l, raw_t x) {
    if constexpr (sizeof(raw_t) == 4) {
        v.w[l] = x;
    } else {
        if (l & 1) v.w[l >> 1] |= (uint32_t)x << 16;
        else v.w[l >> 1] = (uint32_t)x;
    }
}

// The vector path's fold: all LANES elements of one vector at once.  The
// hierarchical order, and the ring on bf16 (8-lane) and int32 vectors and on
// fp32 vectors beyond 8 ranks, run positions outer and lanes inner, so each
// position's (warp-uniform) decisions -- inside W, start of a group, per-hop
// rounding -- are taken once per vector rather than once per lane; the tree,
// and the ring on fp32 vectors up to 8 ranks, run lane by lane.  Each choice
// was measured on GB300 (fp32 ring at W = 8 faster lane by lane; lanes inner:
// int32 ring max at W = 16 6.0 against 4.8 TB/s, fp32 ring at W = 10-12 6.1
// against 4.9).  contrib(x) widens, pre-scales and (per-hop) rounds one raw
// contribution.
template <class A, int ALGO, int WCAP, int VB, int LANES, class Contrib>
__device__ __forceinline__ void fold_lanes(const Vec<VB> (&raw)[WCAP], int W, uint64_t gmask, bool hop,
                                           Contrib contrib, typename A::acc_t (&out)[LANES]) {
    using acc_t = typename A::acc_t;
    using raw_t = typename A::raw_t;
    if constexpr (ALGO == MR_TREE || (ALGO == MR_RING && LANES <= 4 && std::is_same<acc_t, float>::value && WCAP <= 8)) {
#pragma unroll
        for (int l = 0; l < LANES; ++l) {
            acc_t y[WCAP];
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                if (i < W) y[i] = contrib(get_lane<raw_t, VB>(raw[i], l));
            if constexpr (ALGO == MR_TREE) out[l] = fold_tree<A, WCAP>(y, W, hop);
            else out[l] = fold_ring<A, WCAP>(y, W, hop);
        }
    } else if constexpr (ALGO == MR_RING) {
#pragma unroll
        for (int l = 0; l < LANES; ++l) out[l] = contrib(get_lane<raw_t, VB>(raw[0], l));
#pragma unroll
        for (int i = 1; i < WCAP; ++i) {
            if (i < W) {
#pragma unroll
                for (int l = 0; l < LANES; ++l) out[l] = comb<A>(out[l], contrib(get_lane<raw_t, VB>(raw[i], l)), hop);
            }
        }
    } else {
        acc_t total[LANES];
        bool have_total = false;
#pragma unroll
        for (int l = 0; l < LANES; ++l) out[l] = contrib(get_lane<raw_t, VB>(raw[0], l));   // the running group part
#pragma unroll
        for (int i = 1; i < WCAP; ++i) {
            if (i < W) {
                if ((gmask >> i) & 1u) {
                    if (have_total) {
#pragma unroll
                        for (int l = 0; l < LANES; ++l) total[l] = comb<A>(total[l], out[l], hop);
                    } else {
#pragma unroll
                        for (int l = 0; l < LANES; ++l) total[l] = out[l];
                    }
                    have_total = true;
#pragma unroll
                    for (int l = 0; l < LANES; ++l) out[l] = contrib(get_lane<raw_t, VB>(raw[i], l));
                } else {
#pragma unroll
                    for (int l = 0; l < LANES; ++l) out[l] = comb<A>(out[l], contrib(get_lane<raw_t, VB>(raw[i], l)), hop);
                }
            }
        }
        if (have_total) {
#pragma unroll
            for (int l = 0; l < LANES; ++l) out[l] = comb<A>(total[l], out[l], hop);
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Rank at order position i of segment sg.
template <int ALGO>
__device__ __forceinline__ int order_rank(int W, const Segment& sg, int i, int group = 1) {
    if constexpr (ALGO == MR_RING) return ring_rank(W, sg.k, i);
    else if constexpr (ALGO == MR_TREE) return tree_rank(W, sg.tree, i);
    else return hier_rank(W, group, sg.hc, sg.hd, i);
}

template <int DT, int OP, int ALGO, int WCAP, int VB, int U, bool HOP, bool BATCH, bool PAD = false>
__global__ void __launch_bounds__(kThreads, reduce_blocks_per_sm(WCAP, U, BATCH, reduce_wide_heads(WCAP, ALGO)))
reduce_kernel(const __grid_constant__ ReduceParams P) {
    using A = Arith<DT, OP>;
    using raw_t = typename A::raw_t;
    using acc_t = typename A::acc_t;
    constexpr int EB = Elem<DT>::kBytes;
    constexpr int LANES = VB / EB;


    const int W = P.W;
    const float s = P.scale;
    const bool rs = (P.mode == MODE_REDUCE_SCATTER);
    constexpr bool hop = DT == MR_BF16 && HOP;
    // Two bf16 lanes per packed word: per-hop sum and avg (Bf16PairSum), and
    // min and max on 16-bit order keys (Bf16PairKey) except in the plain
    // 16-slot fold, where the keyed pairs spilled and ran 4-14 % slower.
    constexpr bool kPairKeys = DT == MR_BF16 && (OP == MR_MIN || OP == MR_MAX) && (BATCH || WCAP <= 8);
    constexpr bool kPairs = kPairKeys || (DT == MR_BF16 && HOP && (OP == MR_SUM || OP == MR_AVG));   // reduce_pairs()
    using PairA = typename std::conditional<kPairKeys, Bf16PairKey<OP>, Bf16PairSum>::type;
    const uint64_t gmask = P.gmask;
    // a contribution as read: widened, pre-scaled, and for per-hop bf16 rounded
    auto contrib = [&](raw_t x) -> acc_t {
        const acc_t y = A::read(x, s);
        return (OP == MR_AVG && hop) ? A::hop(y) : y;
    };

    // Pairs: one 32-bit word holds two bf16 contributions as read (avg:
    // pre-scaled in fp32, both lanes rounded to bf16 in one packed conversion,
    // lo lane in x; min and max: their 16-bit order keys).
    auto pair = [&](uint32_t w) -> uint32_t {
        if constexpr (kPairKeys) {
            return Bf16PairKey<OP>::key(w);
        } else if constexpr (OP == MR_AVG) {
            const float lo = __fmul_rn(__uint_as_float(w << 16), s);
            const float hi = __fmul_rn(__uint_as_float(w & 0xFFFF0000u), s);
            const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
            uint32_t o;
            memcpy(&o, &p, 4);
            return o;
        } else {
            return w;
        }
    };
    // The batched folds run on "units": a lane's fp32 (or int32) value, or
    // with pairs a packed word of two bf16 lanes.
    using unit_t = typename std::conditional<kPairs, uint32_t, acc_t>::type;
    constexpr int UNITS = kPairs ? VB / 4 : LANES;
    auto unit = [&](const Vec<VB>& v, int u) -> unit_t {
        if constexpr (kPairs) return pair(v.w[u]);
        else return contrib(get_lane<raw_t, VB>(v, u));
    };
    auto ucomb = [&](unit_t a, unit_t b) -> unit_t {
        if constexpr (kPairs) return PairA::combine(a, b);
        else return comb<A>(a, b, hop);
    };
    auto utop = [&](unit_t (&y)[8], int Wb) -> unit_t {
        if constexpr (kPairs) return tree_batch_top<PairA>(y, Wb, false);
        else return tree_batch_top<A>(y, Wb, hop);
    };
    auto uident = []() -> unit_t {
        if constexpr (kPairs) return PairA::identity();
        else return A::identity();
    };
    // A pair's result: the packed sum itself, or the keys' bf16 values.
    auto pair_post = [&](uint32_t r) -> uint32_t {
        if constexpr (kPairKeys) return Bf16PairKey<OP>::post(r);
        else return r;
    };
    auto upost = [&](const unit_t (&r)[UNITS], Vec<VB>& res) {
        if constexpr (kPairs) {
#pragma unroll
            for (int u = 0; u < UNITS; ++u) res.w[u] = pair_post(r[u]);
        } else {
#pragma unroll
            for (int l = 0; l < LANES; ++l) set_lane<raw_t, VB>(res, l, A::post(r[l], W));
        }
    };

    // Input pointers in the current segment's accumulation order: in
    // registers for the plain fold, in a shared-memory table for the batched
    // one (BATCH: the ranks are loaded and folded in batches of 8, so only 8
    // vectors are live at a time).
    constexpr bool kTable = BATCH;
    constexpr bool kTreeBatched = BATCH && ALGO == MR_TREE;
    // PAD: the identity-padded tree (no condition on W inside a batch), which
    // the host takes for the int32 trees over 16 slots when W is not a
    // multiple of 8: at 9-11 ranks the conditional fold's branches on the
    // ragged last batch (3x the ring's, ncu) held them at 5.67-5.84 TB/s;
    // padded they run at 5.89-6.35 (sum 6.21-6.35).  With whole batches
    // (W = 16) the conditional fold measured 1-2.6 % faster, and the float
    // trees 4-10 % slower padded at 9-13 ranks.
    constexpr bool kPaddedTree = kTreeBatched && PAD;
    // The 32- and 64-slot trees keep their batches' top subtotals in dynamic
    // shared memory (see reduce_top_shared).
    constexpr bool kTopShared = kTreeBatched && WCAP >= 32;   // reduce_top_shared()
    extern __shared__ float dyn_smem[];
    unit_t* const top_smem = reinterpret_cast<unit_t*>(dyn_smem);
    static_assert(!BATCH || WCAP % 8 == 0, "batches of 8 positions");
    // The 64-slot trees (2 CTAs per SM) keep one table per warp: a warp that
    // moves to another segment rewrites its own copy between two warp
    // barriers while the CTA's other warps run on.  The other batched folds
    // (3 CTAs per SM) share one table per CTA: there the CTA-wide barrier
    // measured faster (warps that stay on one tile together, 3-6 % at 10-28
    // ranks), at 2 CTAs per SM slower (the 64-slot trees 3-12 %).
    constexpr bool kWarpTable = kTable && WCAP == 64 && ALGO == MR_TREE;
    constexpr int kTables = kWarpTable ? kThreads / 32 : 1;
    __shared__ const char* table[kTables][kTable ? WCAP : 1];
    const char* src[kTable ? 1 : WCAP];
    int cur = -1;
    auto enter = [&](int seg) {
        if (seg == cur) return;
        cur = seg;
        if constexpr (kWarpTable) {
            const int wp = threadIdx.x >> 5;
            __syncwarp();
            for (int i = threadIdx.x & 31; i < W; i += 32)
                table[wp][i] = static_cast<const char*>(P.in[order_rank<ALGO>(W, P.seg[seg], i, P.group)]);
            __syncwarp();
        } else if constexpr (kTable) {
            __syncthreads();
            if (threadIdx.x < W)
                table[0][threadIdx.x] = static_cast<const char*>(P.in[order_rank<ALGO>(W, P.seg[seg], threadIdx.x, P.group)]);
            __syncthreads();
        } else {
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                src[i] = (i < W) ? static_cast<const char*>(P.in[order_rank<ALGO>(W, P.seg[seg], i, P.group)]) : nullptr;
        }
    };
    auto input = [&](int i) -> const char* {
        if constexpr (kWarpTable) return table[threadIdx.x >> 5][i];
        else if constexpr (kTable) return table[0][i];
        else return src[i];
    };

    // One element, reduced from scratch (heads, tails, unaligned buffers);
    // the batched kernels fold it in batches as their vector tiles do.
    auto element = [&](const Segment& sg, uint64_t e) {
        raw_t r;
        if constexpr (BATCH) {
            auto load = [&](int m, int Wb, raw_t (&raw)[8]) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < Wb) raw[q] = __ldg(reinterpret_cast<const raw_t*>(input(8 * m + q)) + e);
            };
            auto one = [&](raw_t x, int) -> acc_t { return contrib(x); };
            auto cb = [&](acc_t a, acc_t b) -> acc_t { return comb<A>(a, b, hop); };
            acc_t res[1];
            if constexpr (ALGO == MR_TREE) {
                acc_t tops[WCAP / 8];
                batched_tree<WCAP / 8, 1, acc_t, raw_t>(
                    W, load, one, cb, [&](acc_t (&y)[8], int Wb) -> acc_t { return tree_batch_top<A>(y, Wb, hop); },
                    [&](int m, int) -> acc_t& { return tops[m]; }, res);
            } else {
                batched_left_fold<ALGO == MR_HIER, 1, acc_t, raw_t>(W, gmask, load, one, cb, res);
            }
            r = A::post(res[0], W);
        } else {
            acc_t y[WCAP];
#pragma unroll
            for (int i = 0; i < WCAP; ++i)
                if (i < W) y[i] = contrib(__ldg(reinterpret_cast<const raw_t*>(input(i)) + e));
            r = A::post(fold<A, ALGO, WCAP>(y, W, hop, gmask), W);
        }
        if (rs) {
            static_cast<raw_t*>(P.out[sg.k])[e - sg.out_lo] = r;
        } else {
#pragma unroll 8
            for (int j = 0; j < W; ++j) static_cast<raw_t*>(P.out[j])[e] = r;
        }
    };

    // Before waiting on the previous kernel, whatever depends on the
    // parameters alone: this CTA's first vector tile and its segment's input
    // pointers (a 64-bit divide and a chain of parameter reads).  A small
    // call is one tile per CTA, so its loads then issue as soon as the wait
    // returns.
    uint64_t t_first = blockIdx.x;
    if (P.vec) {
        const uint64_t ntiles = P.tiles_max * (uint64_t)P.nseg;
        for (; t_first < ntiles; t_first += gridDim.x) {
            const int s0 = (int)(t_first % (uint64_t)P.nseg);
            if (t_first / (uint64_t)P.nseg < P.tile_start[s0 + 1] - P.tile_start[s0]) {
                enter(s0);
                break;
            }
        }
    }
    pdl_enter();    // the previous kernel on the stream has finished with our buffers

    int seg = 0;
    if (P.vec) {
        // Vector tiles are dealt round-robin across segments: tile t is tile
        // t / nseg of segment t % nseg, and CTAs stride over t.  The grid's
        // live tiles are thus spread over every chunk of every rank buffer;
        // measured on GB300 this keeps HBM busier than sweeping the segments
        // one after another.
        const uint64_t ntiles = P.tiles_max * (uint64_t)P.nseg;
        constexpr uint64_t kTile = (uint64_t)kThreads * U;    // vectors per tile
        for (uint64_t t = t_first; t < ntiles; t += gridDim.x) {
            seg = (int)(t % (uint64_t)P.nseg);
            const uint64_t local = t / (uint64_t)P.nseg;
            if (local >= P.tile_start[seg + 1] - P.tile_start[seg]) continue;
            enter(seg);
            const Segment& sg = P.seg[seg];
            const uint64_t va = (sg.lo + LANES - 1) / LANES, vb = sg.hi / LANES;
            const uint64_t v0 = va + local * kTile + threadIdx.x;
            if constexpr (BATCH) {
                // Many ranks: the positions are loaded and folded in batches
                // of 8 (8 independent 16-byte loads in flight, as at W = 8).
                static_assert(U == 1, "the batched folds take one vector per thread per tile");
                if (v0 < vb) {
                    const uint64_t off = v0 * VB;
                    auto load = [&](int m, int Wb, Vec<VB> (&raw)[8]) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q < Wb) raw[q] = load_vec<VB>(input(8 * m + q) + off);
                    };
                    unit_t res_u[UNITS];
                    if constexpr (kTreeBatched) {
                        // The batches' in-batch top subtotals are read once,
                        // when the heads are folded; with kTopShared they wait
                        // in this thread's own shared-memory slots
                        // ([batch][unit][thread]) rather than in registers.
                        constexpr int NB = WCAP / 8;
                        unit_t top_reg[kTopShared ? 1 : NB][kTopShared ? 1 : UNITS];
                        auto top_at = [&](int m, int u) -> unit_t& {
                            if constexpr (kTopShared) return top_smem[((uint64_t)m * UNITS + u) * kThreads + threadIdx.x];
                            else return top_reg[m][u];
                        };
                        if constexpr (kPaddedTree)
                            batched_tree_padded<NB, UNITS, unit_t, Vec<VB>>(W, load, unit, ucomb, uident, top_at, res_u);
                        else
                            batched_tree<NB, UNITS, unit_t, Vec<VB>>(W, load, unit, ucomb, utop, top_at, res_u);
                    } else {
                        batched_left_fold<ALGO == MR_HIER, UNITS, unit_t, Vec<VB>>(W, gmask, load, unit, ucomb, res_u);
                    }
                    Vec<VB> res;
                    upost(res_u, res);
                    if (rs) {
                        store_vec<VB>(static_cast<char*>(P.out[sg.k]) + off - sg.out_lo * EB, res);
                    } else {
#pragma unroll 8
                        for (int j = 0; j < W; ++j) store_vec<VB>(static_cast<char*>(P.out[j]) + off, res);
                    }
                }
                continue;
            }
            if constexpr (!BATCH) {
                // U*W independent 16-byte loads in flight before the first fold.
                Vec<VB> raw[U][WCAP];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = v0 + (uint64_t)u * kThreads;
                    if (v < vb) {
#pragma unroll
                        for (int i = 0; i < WCAP; ++i)
                            if (i < W) raw[u][i] = load_vec<VB>(input(i) + v * VB);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = v0 + (uint64_t)u * kThreads;
                    if (v >= vb) break;
                    const uint64_t off = v * VB;
                    Vec<VB> res;
                    if constexpr (kPairs) {
#pragma unroll
                        for (int k = 0; k < VB / 4; ++k) {
                            uint32_t y[WCAP];
#pragma unroll
                            for (int i = 0; i < WCAP; ++i)
                                if (i < W) y[i] = pair(raw[u][i].w[k]);
                            res.w[k] = pair_post(fold<PairA, ALGO, WCAP>(y, W, false, gmask));
                        }
                    } else {
                        acc_t r[LANES];
                        fold_lanes<A, ALGO, WCAP, VB, LANES>(raw[u], W, gmask, hop, contrib, r);
#pragma unroll
                        for (int l = 0; l < LANES; ++l) set_lane<raw_t, VB>(res, l, A::post(r[l], W));
                    }
                    if (rs) {
                        store_vec<VB>(static_cast<char*>(P.out[sg.k]) + off - sg.out_lo * EB, res);
                    } else {
#pragma unroll
                        for (int j = 0; j < WCAP; ++j)
                            if (j < W) store_vec<VB>(static_cast<char*>(P.out[j]) + off, res);
                    }
                }
            }
        }
        // The elements outside whole vectors (fewer than 2*LANES per segment):
        // segment i's are done by CTA i mod gridDim.x.
        for (int i = blockIdx.x; i < P.nseg; i += gridDim.x) {
            enter(i);
            const Segment& sg = P.seg[i];
            const uint64_t va = (sg.lo + LANES - 1) / LANES, vb = sg.hi / LANES;
            const uint64_t h1 = va < vb ? va * LANES : sg.hi;   // head [lo, h1)
            const uint64_t t0 = va < vb ? vb * LANES : sg.hi;   // tail [t0, hi)
            const uint64_t nh = h1 - sg.lo, n = nh + (sg.hi - t0);
            for (uint64_t x = threadIdx.x; x < n; x += kThreads)
                element(sg, x < nh ? sg.lo + x : t0 + (x - nh));
        }
    } else {
        // Buffers not aligned to the vector width: tiles of kThreads elements,
        // segment after segment.
        const uint64_t ntiles = P.tile_start[P.nseg];
        for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
            while (t >= P.tile_start[seg + 1]) ++seg;
            enter(seg);
            const Segment& sg = P.seg[seg];
            const uint64_t e = sg.lo + (t - P.tile_start[seg]) * kThreads + threadIdx.x;
            if (e < sg.hi) element(sg, e);
        }
    }
}

// Launch with at least P.spread_smem bytes of dynamic shared memory per CTA
// (see plan_tiles: it caps how many CTAs share an SM).
template <class K>
cudaError_t launch_spread(K k, dim3 grid, size_t smem, cudaStream_t stream, const ReduceParams& P) {
    if (P.spread_smem > smem) smem = P.spread_smem;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(k, grid, smem, stream, 0, P);
}

// Instantiate and launch the kernel for one element type and one order.
template <int DT, int ALGO, bool HOP>
cudaError_t launch_reduce(const ReduceParams& P, int op, dim3 grid, cudaStream_t stream) {
    auto go = [&](auto op_c) -> cudaError_t {
        constexpr int OP = decltype(op_c)::value;
        const bool rs = P.mode == MODE_REDUCE_SCATTER;
        // The batched kernels above 16 ranks; the trees' top subtotals take
        // dynamic shared memory.
        auto launch_wide = [&](auto wc) -> cudaError_t {
            constexpr int WC = decltype(wc)::value;
            constexpr int VB = kReduceVectorBytes;
            auto k = reduce_kernel<DT, OP, ALGO, WC, VB, reduce_unroll_for(WC, false), HOP, true>;
            size_t smem = 0;
            if constexpr (reduce_top_shared(WC, ALGO))
                smem = reduce_top_shared_bytes(WC, reduce_pairs(DT, OP, HOP) ? VB / 4 : VB / Elem<DT>::kBytes);
            return launch_spread(k, grid, smem, stream, P);
        };
        switch (reduce_wcap(P.W, ALGO)) {
            case 2: return launch_spread(reduce_kernel<DT, OP, ALGO, 2, 16, reduce_unroll_for(2, false), HOP, false>, grid, 0, stream, P);
            case 4: return launch_spread(reduce_kernel<DT, OP, ALGO, 4, 16, reduce_unroll_for(4, false), HOP, false>, grid, 0, stream, P);
            case 8:
                if (rs) return launch_spread(reduce_kernel<DT, OP, ALGO, 8, 16, reduce_unroll_for(8, true), HOP, false>, grid, 0, stream, P);
                return launch_spread(reduce_kernel<DT, OP, ALGO, 8, 16, reduce_unroll_for(8, false), HOP, false>, grid, 0, stream, P);
            case 16:
                if constexpr (DT == MR_INT32 && ALGO == MR_TREE) {
                    if (P.W % 8 != 0)
                        return launch_spread(reduce_kernel<DT, OP, ALGO, 16, 16, 1, HOP, true, true>, grid, 0, stream, P);
                }
                if (reduce_batched(P.W, ALGO, DT, HOP))
                    return launch_spread(reduce_kernel<DT, OP, ALGO, 16, 16, 1, HOP, true>, grid, 0, stream, P);
                return launch_spread(reduce_kernel<DT, OP, ALGO, 16, 16, reduce_unroll_for(16, false), HOP, false>, grid, 0, stream, P);
            case 32:
                if constexpr (ALGO == MR_TREE) return launch_wide(std::integral_constant<int, 32>{});
                return cudaErrorInvalidValue;
            default:
                return launch_wide(std::integral_constant<int, 64>{});
        }
    };
    switch (op) {
        case MR_SUM: return go(std::integral_constant<int, MR_SUM>{});
        case MR_PROD: return go(std::integral_constant<int, MR_PROD>{});
        case MR_MIN: return go(std::integral_constant<int, MR_MIN>{});
        case MR_MAX: return go(std::integral_constant<int, MR_MAX>{});
        case MR_AVG: return go(std::integral_constant<int, MR_AVG>{});
    }
    return cudaErrorInvalidValue;
}

}  // namespace mr
