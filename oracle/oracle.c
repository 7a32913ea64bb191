/*
 * oracle.c -- the CPU oracle.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Compiled with -ffp-contract=off so that no multiply-add is ever fused: every
 * fp32 operation below is one IEEE binary32 operation, rounded to nearest even.
 * Single-threaded, element by element, in the order the method defines.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Element access                                                            */
/* ------------------------------------------------------------------------- */

typedef union {
    float f;     /* fp32 and bf16 accumulate in fp32 */
    uint32_t u;  /* int32 accumulates in 32-bit two's complement, wrapping */
} acc_t;

static size_t elem_size(int dtype) { return dtype == OR_BF16 ? 2u : 4u; }

/*
 * bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 pattern.
 * int32 is kept as its bit pattern so that sum and product wrap modulo 2^32.
 */
static acc_t widen(int dtype, const void* buf, size_t e) {
    acc_t a;
    if (dtype == OR_BF16) {
        uint16_t h;
        memcpy(&h, (const char*)buf + 2u * e, 2);
        a.u = (uint32_t)h << 16;
    } else {
        memcpy(&a.u, (const char*)buf + 4u * e, 4);
    }
    return a;
}

/* ------------------------------------------------------------------------- */
/* bf16 rounding                                                             */
/* ------------------------------------------------------------------------- */

/*
 * Nearest bf16, ties to even.  Adding 0x7FFF plus the lowest kept bit to the
 * fp32 pattern carries into the kept half exactly when the dropped half is
 * above one half, or exactly one half with an odd kept half.  Values past the
 * largest finite bf16 carry into the exponent and become +-infinity.  A NaN
 * keeps its sign and is made quiet.
 */
uint16_t or_f32_to_bf16_rne(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void or_f32_to_bf16_rne_array(const uint32_t* in, uint16_t* out, size_t n) {
    for (size_t i = 0; i < n; i++) {
        float f;
        memcpy(&f, &in[i], 4);
        out[i] = or_f32_to_bf16_rne(f);
    }
}

/* ------------------------------------------------------------------------- */
/* The reduction ops ("What all-reduce promises": sum, prod, min, max, avg)  */
/* ------------------------------------------------------------------------- */

/* min and max order -0 below +0, so that both are independent of the order
 * in which the ranks are visited. */
static float min_f32(float a, float b) {
    if (b < a) return b;
    if (a < b) return a;
    if (a == 0.0f && b == 0.0f) return signbit(b) ? b : a;
    return a;
}

static float max_f32(float a, float b) {
    if (a < b) return b;
    if (b < a) return a;
    if (a == 0.0f && b == 0.0f) return signbit(b) ? a : b;
    return a;
}

/* a (+) b for the op; avg combines like sum. */
static acc_t combine(int dtype, int op, acc_t a, acc_t b) {
    if (dtype == OR_INT32) {
        switch (op) {
        case OR_SUM:
        case OR_AVG: a.u = a.u + b.u; break;
        case OR_PROD: a.u = a.u * b.u; break;
        case OR_MIN: if ((int32_t)b.u < (int32_t)a.u) a = b; break;
        case OR_MAX: if ((int32_t)a.u < (int32_t)b.u) a = b; break;
        }
    } else {
        switch (op) {
        case OR_SUM:
        case OR_AVG: a.f = a.f + b.f; break;
        case OR_PROD: a.f = a.f * b.f; break;
        case OR_MIN: a.f = min_f32(a.f, b.f); break;
        case OR_MAX: a.f = max_f32(a.f, b.f); break;
        }
    }
    return a;
}

/*
 * The pre-scale of a float avg: each contribution is multiplied by 1/W as it
 * is read, with 1/W rounded once to fp32.  Integers are not scaled.
 */
static float avg_scale(int W) { return (float)(1.0 / (double)W); }

static acc_t read_contribution(int dtype, int op, float s, const void* buf, size_t e) {
    acc_t y = widen(dtype, buf, e);
    if (op == OR_AVG && dtype != OR_INT32) y.f = y.f * s;
    return y;
}

/* The postOp at the step where a chunk's sum completes: one truncating divide
 * of the finished integer sum for avg, one bf16 rounding for bf16, nothing for
 * fp32.  Writes element e of buf. */
static void store_result(int dtype, int op, int W, acc_t acc, void* buf, size_t e) {
    if (dtype == OR_FP32) {
        memcpy((char*)buf + 4u * e, &acc.u, 4);
    } else if (dtype == OR_BF16) {
        uint16_t h = or_f32_to_bf16_rne(acc.f);
        memcpy((char*)buf + 2u * e, &h, 2);
    } else {
        int32_t v = (int32_t)acc.u;
        if (op == OR_AVG) v = v / W;
        memcpy((char*)buf + 4u * e, &v, 4);
    }
}

/* ------------------------------------------------------------------------- */
/* Chunking (Eq. 2 of the M2N paper: l = floor(i*S/D))                       */
/* ------------------------------------------------------------------------- */

size_t or_chunk_lo(int W, size_t N, int k) {
    /* floor(k*N/W) without forming k*N: N = q*W + r. */
    size_t q = N / (size_t)W, r = N % (size_t)W;
    return (size_t)k * q + ((size_t)k * r) / (size_t)W;
}

/* ------------------------------------------------------------------------- */
/* Ring order ("The ring, exactly as the kernel runs it")                    */
/* ------------------------------------------------------------------------- */

/*
 * With ranks in a ring 0 -> 1 -> ... -> W-1 -> 0, rank k+1 sends its own part
 * of chunk k first; each of the next W-1 hops adds the receiving rank's part;
 * the total is complete on rank k, which owns chunk k.
 */
void or_ring_order(int W, int k, int* order) {
    for (int i = 0; i < W; i++) order[i] = (k + 1 + i) % W;
}

/* ------------------------------------------------------------------------- */
/* Double binary tree ("The double binary tree")                             */
/* ------------------------------------------------------------------------- */

/*
 * Tree 1: the lowest set bit b of rank r fixes its depth (rank 0, the root,
 * takes b = the smallest power of two >= W).  Parent: clear b and set the next
 * bit up; if that falls outside the ranks, just clear b.  Children: r - b/2
 * (for b > 1), and r + h for the largest h in b/2, b/4, ..., 1 that stays
 * inside the ranks.
 */
static void tree1(int W, int* parent, int* child) {
    int B = 1;
    while (B < W) B <<= 1;
    for (int r = 0; r < W; r++) {
        int b = (r == 0) ? B : (r & -r);
        if (r == 0) {
            parent[r] = -1;
        } else {
            int p = (r & ~b) | (b << 1);
            if (p >= W) p = r & ~b;
            parent[r] = p;
        }
        int n = 0;
        child[2 * r] = child[2 * r + 1] = -1;
        if (r > 0 && b > 1) child[2 * r + n++] = r - b / 2;
        for (int h = b / 2; h >= 1; h /= 2) {
            if (r + h < W) {
                child[2 * r + n++] = r + h;
                break;
            }
        }
    }
}

/*
 * Tree 2 swaps the roles of leaves and interior ranks: for even W it is the
 * mirror image of tree 1 (rank W-1-r takes the place of r); for odd W it is
 * tree 1 shifted by one rank (rank (r+1) mod W takes the place of r).
 */
static int tree2_rank(int W, int r) { return (W % 2 == 0) ? (W - 1 - r) : ((r + 1) % W); }

int or_tree_build(int W, int which, int* parent, int* child) {
    int p1[OR_MAX_RANKS], c1[2 * OR_MAX_RANKS];
    if (W < 1 || W > OR_MAX_RANKS) return -1;
    tree1(W, p1, c1);
    if (which == 1) {
        memcpy(parent, p1, sizeof(int) * (size_t)W);
        memcpy(child, c1, sizeof(int) * 2u * (size_t)W);
        return 0;
    }
    for (int r = 0; r < W; r++) {
        int m = tree2_rank(W, r);
        parent[m] = p1[r] < 0 ? -1 : tree2_rank(W, p1[r]);
        for (int i = 0; i < 2; i++)
            child[2 * m + i] = c1[2 * r + i] < 0 ? -1 : tree2_rank(W, c1[2 * r + i]);
    }
    return tree2_rank(W, 0);
}



/* ------------------------------------------------------------------------- */
/* The reduction of one element position                                     */
/* ------------------------------------------------------------------------- */

typedef struct {
    int dtype, op, algo, W;
    int group;   /* ranks per group (hierarchical order) */
    int hop;     /* 1: round the running total to bf16 after every hop (bf16 only) */
    size_t N;
    float s;
    int root[2];
    int child[2][2 * OR_MAX_RANKS];
} plan_t;

/* Per-hop rounding: with hop set, a bf16 running total is rounded to bf16
 * after every combine, as when each partial crosses a wire as bf16. */
static acc_t hop_round(const plan_t* P, acc_t a) {
    if (P->hop && P->dtype == OR_BF16) a.u = (uint32_t)or_f32_to_bf16_rne(a.f) << 16;
    return a;
}

static acc_t combine_hop(const plan_t* P, acc_t a, acc_t b) { return hop_round(P, combine(P->dtype, P->op, a, b)); }

/* Reduce up the tree, each parent adding its children's subtotals to its own
 * contribution: subtotal(v) = y_v (+) subtotal(first child) (+) subtotal(second). */
static acc_t tree_subtotal(const plan_t* P, int v, const int* child, const acc_t* y) {
    acc_t acc = y[v];
    for (int i = 0; i < 2; i++) {
        int c = child[2 * v + i];
        if (c >= 0) acc = combine_hop(P, acc, tree_subtotal(P, c, child, y));
    }
    return acc;
}

static int make_plan_ex(plan_t* P, int dtype, int op, int algo, int group, int hop, int W, size_t N) {
    int parent[OR_MAX_RANKS];
    if (W < 1 || W > OR_MAX_RANKS) return -1;
    if (dtype < OR_FP32 || dtype > OR_INT32) return -1;
    if (op < OR_SUM || op > OR_AVG) return -1;
    if (algo != OR_RING && algo != OR_TREE && algo != OR_HIER) return -1;
    if (algo == OR_HIER && (group < 1 || W % group != 0)) return -1;
    P->dtype = dtype;
    P->op = op;
    P->algo = algo;
    P->group = algo == OR_HIER ? group : W;
    P->hop = hop ? 1 : 0;
    P->W = W;
    P->N = N;
    P->s = avg_scale(W);
    P->root[0] = or_tree_build(W, 1, parent, P->child[0]);
    P->root[1] = or_tree_build(W, 2, parent, P->child[1]);
    return 0;
}

static int make_plan(plan_t* P, int dtype, int op, int algo, int W, size_t N) {
    return make_plan_ex(P, dtype, op, algo, W, 0, W, N);
}

/* y[r] = rank r's (pre-scaled) contribution at element e, which lies in chunk k. */
static acc_t reduce_position(const plan_t* P, int k, size_t e, const acc_t* y) {
    if (P->algo == OR_RING) {
        int order[OR_MAX_RANKS];
        or_ring_order(P->W, k, order);
        acc_t acc = y[order[0]];
        for (int i = 1; i < P->W; i++) acc = combine_hop(P, acc, y[order[i]]);
        return acc;
    }
    if (P->algo == OR_HIER) {
        /* Hierarchical all-reduce ("Communication Optimization ...", the
         * five-step topology-aware all-reduce): ranks form G = W/g groups of g
         * (rank a*g + i is local rank i of group a).  A ring reduce-scatter
         * inside each group leaves chunk c (of g) summed over the group on
         * local rank c -- its ring order is i = c+1, ..., c; a ring all-reduce
         * across the groups then cuts chunk c into G pieces and sums piece d
         * over the groups in order a = d+1, ..., d; the all-gather inside the
         * groups copies. */
        int g = P->group, G = P->W / g, c = 0, d = 0;
        int og[OR_MAX_RANKS], oG[OR_MAX_RANKS];
        while (or_chunk_lo(g, P->N, c + 1) <= e) c++;
        size_t clo = or_chunk_lo(g, P->N, c), clen = or_chunk_lo(g, P->N, c + 1) - clo;
        while (clo + or_chunk_lo(G, clen, d + 1) <= e) d++;
        or_ring_order(g, c, og);
        or_ring_order(G, d, oG);
        acc_t total;
        for (int ia = 0; ia < G; ia++) {
            int a = oG[ia];
            acc_t part = y[a * g + og[0]];
            for (int ii = 1; ii < g; ii++) part = combine_hop(P, part, y[a * g + og[ii]]);
            total = ia ? combine_hop(P, total, part) : part;
        }
        return total;
    }
    /* The first floor(N/2) elements climb tree 1, the rest tree 2. */
    int t = (e < P->N / 2) ? 0 : 1;
    return tree_subtotal(P, P->root[t], P->child[t], y);
}

static acc_t reduce_from_buffers(const plan_t* P, int k, size_t e, const void* const* in) {
    acc_t y[OR_MAX_RANKS];
    for (int r = 0; r < P->W; r++) y[r] = hop_round(P, read_contribution(P->dtype, P->op, P->s, in[r], e));
    return reduce_position(P, k, e, y);
}

/* ------------------------------------------------------------------------- */
/* The collectives                                                           */
/* ------------------------------------------------------------------------- */

int or_allreduce_ex(int dtype, int op, int algo, int group, int hop, int W, size_t N,
                    const void* const* in, void* const* out) {
    plan_t P;
    if (make_plan_ex(&P, dtype, op, algo, group, hop, W, N) != 0) return -1;
    for (int k = 0; k < W; k++) {
        size_t lo = or_chunk_lo(W, N, k), hi = or_chunk_lo(W, N, k + 1);
        for (size_t e = lo; e < hi; e++) {
            acc_t acc = reduce_from_buffers(&P, k, e, in);
            for (int j = 0; j < W; j++) store_result(dtype, op, W, acc, out[j], e);
        }
    }
    return 0;
}

int or_reduce_scatter_ex(int dtype, int op, int algo, int group, int hop, int W, size_t N,
                         const void* const* in, void* const* out) {
    plan_t P;
    if (make_plan_ex(&P, dtype, op, algo, group, hop, W, N) != 0) return -1;
    if (N % (size_t)W != 0) return -1;
    for (int k = 0; k < W; k++) {
        size_t lo = or_chunk_lo(W, N, k), hi = or_chunk_lo(W, N, k + 1);
        for (size_t e = lo; e < hi; e++) {
            acc_t acc = reduce_from_buffers(&P, k, e, in);
            store_result(dtype, op, W, acc, out[k], e - lo);
        }
    }
    return 0;
}

int or_allreduce(int dtype, int op, int algo, int W, size_t N, const void* const* in, void* const* out) {
    if (algo == OR_HIER) return -1;
    return or_allreduce_ex(dtype, op, algo, W, 0, W, N, in, out);
}

int or_reduce_scatter(int dtype, int op, int algo, int W, size_t N, const void* const* in, void* const* out) {
    if (algo == OR_HIER) return -1;
    return or_reduce_scatter_ex(dtype, op, algo, W, 0, W, N, in, out);
}

int or_all_gather(int dtype, int W, size_t N, const void* const* in, void* const* out) {
    if (W < 1 || W > OR_MAX_RANKS) return -1;
    if (dtype < OR_FP32 || dtype > OR_INT32) return -1;
    if (N % (size_t)W != 0) return -1;
    size_t b = elem_size(dtype);
    for (int k = 0; k < W; k++) {
        size_t lo = or_chunk_lo(W, N, k), hi = or_chunk_lo(W, N, k + 1);
        for (size_t i = 0; i < hi - lo; i++)
            for (int j = 0; j < W; j++)
                memcpy((char*)out[j] + b * (lo + i), (const char*)in[k] + b * i, b);
    }
    return 0;
}

int or_reduce_one(int dtype, int op, int algo, int W, size_t N, size_t e,
                  const void* y_raw, void* res) {
    plan_t P;
    acc_t y[OR_MAX_RANKS];
    if (make_plan(&P, dtype, op, algo, W, N) != 0) return -1;
    if (e >= N) return -1;
    int k = 0;
    while (or_chunk_lo(W, N, k + 1) <= e) k++;
    for (int r = 0; r < W; r++) y[r] = read_contribution(dtype, op, P.s, y_raw, (size_t)r);
    acc_t acc = reduce_position(&P, k, e, y);
    store_result(dtype, op, W, acc, res, 0);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* All-reduce with a residual add and RMSNorm after the sum                  */
/* ("How this survives ten thousand GPUs", post on NCCL all-reduce: in       */
/* decoding, the merge and the RMSNorm that follow the all-reduce are fused  */
/* into it)                                                                  */
/* ------------------------------------------------------------------------- */

/* The buffer is `rows` rows of `hidden` elements.  For each element the W
 * contributions are summed exactly as or_allreduce sums them (same chunks,
 * same order, fp32), then the residual is added in fp32:
 *     h = s + residual.
 * residual_out (if non-NULL) receives h rounded to the element type.  Each
 * row is then normalised by its root mean square and scaled by the weight:
 *     out = h / sqrt(mean(h^2) + eps) * weight,
 * evaluated in fp64 from the fp32 h (the exact reference the fp32 kernel is
 * held to within a derived tolerance) and rounded once to the element type;
 * every out[j] receives it.  fp32 and bf16 only. */
int or_allreduce_rmsnorm(int dtype, int algo, int W, size_t rows, size_t hidden,
                         const void* const* in, const void* residual, const void* weight, double eps,
                         void* const* out, void* residual_out) {
    plan_t P;
    size_t N = rows * hidden;
    if (dtype == OR_INT32) return -1;
    if (make_plan(&P, dtype, OR_SUM, algo, W, N) != 0) return -1;
    if (hidden == 0 || !weight) return -1;
    float* h = (float*)malloc(sizeof(float) * (hidden ? hidden : 1));
    if (!h) return -1;
    for (size_t row = 0; row < rows; row++) {
        double ss = 0.0;
        for (size_t i = 0; i < hidden; i++) {
            size_t e = row * hidden + i;
            int k = 0;
            while (or_chunk_lo(W, N, k + 1) <= e) k++;
            acc_t s = reduce_from_buffers(&P, k, e, in);
            float hv = s.f;
            if (residual) hv = hv + widen(dtype, residual, e).f;
            h[i] = hv;
            if (residual_out) {
                acc_t a;
                a.f = hv;
                store_result(dtype, OR_SUM, W, a, residual_out, e);
            }
            ss += (double)hv * (double)hv;
        }
        double inv = 1.0 / sqrt(ss / (double)hidden + eps);
        for (size_t i = 0; i < hidden; i++) {
            size_t e = row * hidden + i;
            acc_t a;
            a.f = (float)((double)h[i] * inv * (double)widen(dtype, weight, i).f);
            for (int j = 0; j < W; j++) store_result(dtype, OR_SUM, W, a, out[j], e);
        }
    }
    free(h);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* 1-bit sign compression with error feedback, then the reduction            */
/* (Communication Optimization: Gradient Compression, NCCL ... -- the 1-bit  */
/* SGD paragraph and the error-feedback paragraph of the top-K section)      */
/* ------------------------------------------------------------------------- */

/* p_r = g_r + e_r (one fp32 add per element), and the rank's scale
 *     s_r = ||p_r||_1 / N,
 * read as a real number: the exact sum of the |p| divided exactly by N, then
 * rounded once to the nearest fp32, ties to even.  (A NaN among the p makes
 * the scale NaN; otherwise an infinite |p| makes it +infinity.)
 *
 * Every finite fp32 is an integer multiple of 2^-149, the smallest subnormal,
 * and below 2^277 of those units, so the sum is kept exactly as an integer
 * count of 2^-149 units in L1_WORDS 32-bit words (384 bits: room for 2^107
 * terms).  The quotient by N is taken bit by bit, from the top, like long
 * division on paper. */
#define L1_WORDS 12
#define L1_BITS (32 * L1_WORDS)

typedef struct {
    uint32_t w[L1_WORDS];   /* little-endian words of the count of 2^-149 units */
    int any_nan, any_inf;
} l1_sum_t;

static int big_bit(const uint32_t* w, int bit) { return (int)((w[bit / 32] >> (bit % 32)) & 1u); }

/* sum += |a| */
static void l1_add(l1_sum_t* s, float a) {
    uint32_t u;
    memcpy(&u, &a, 4);
    u &= 0x7FFFFFFFu;
    uint32_t biased = u >> 23, frac = u & 0x7FFFFFu;
    if (biased == 255u) {
        if (frac) s->any_nan = 1;
        else s->any_inf = 1;
        return;
    }
    /* |a| = m * 2^(pos - 149): a normal number carries the implicit bit and
     * exponent biased - 150; a subnormal has exponent -149. */
    uint64_t m = biased ? (uint64_t)(frac | 0x800000u) : (uint64_t)frac;
    int pos = biased ? (int)biased - 1 : 0;
    uint64_t v = m << (pos % 32);       /* below 2^55: spans two words */
    uint64_t carry = 0;
    for (int j = pos / 32; j < L1_WORDS; j++) {
        uint64_t add = 0;
        if (j == pos / 32) add = v & 0xFFFFFFFFu;
        else if (j == pos / 32 + 1) add = v >> 32;
        uint64_t t = (uint64_t)s->w[j] + add + carry;
        s->w[j] = (uint32_t)t;
        carry = t >> 32;
    }
}

/* The nearest fp32 to S / N, ties to even, for S = the sum in 2^-149 units. */
static float l1_mean(const l1_sum_t* s, uint64_t N) {
    if (s->any_nan) return NAN;
    if (s->any_inf) return INFINITY;
    /* Q = floor(S / N), R = S mod N */
    uint32_t q[L1_WORDS];
    memset(q, 0, sizeof(q));
    uint64_t r = 0;
    for (int bit = L1_BITS - 1; bit >= 0; bit--) {
        int top = (int)(r >> 63);
        r = (r << 1) | (uint64_t)big_bit(s->w, bit);
        if (top || r >= N) {            /* (top: the true value passed 2^64, so it exceeds N) */
            r -= N;
            q[bit / 32] |= 1u << (bit % 32);
        }
    }
    int len = 0;                        /* bit length of Q */
    for (int bit = L1_BITS - 1; bit >= 0; bit--)
        if (big_bit(q, bit)) {
            len = bit + 1;
            break;
        }
    if (len <= 24) {
        /* S / N < 2^-125: the fp32 values there (subnormals and the lowest
         * normal binade) are the integer multiples of 2^-149, so round
         * Q + R/N to an integer: up past one half, a tie to the even one. */
        uint64_t m = (uint64_t)q[0];
        if (r > N - r || (r == N - r && (m & 1u))) m++;
        return (float)ldexp((double)m, -149);
    }
    /* keep the top 24 bits of Q; the rest of Q and R/N decide the rounding */
    int shift = len - 24;
    uint64_t m = 0;
    for (int bit = len - 1; bit >= shift; bit--) m = (m << 1) | (uint64_t)big_bit(q, bit);
    int half = big_bit(q, shift - 1);
    int below = r != 0;
    for (int bit = shift - 2; bit >= 0 && !below; bit--) below = big_bit(q, bit);
    if (half && (below || (m & 1u))) m++;
    return (float)ldexp((double)m, shift - 149);   /* exact, or +inf past the largest fp32 */
}

int or_sign_ef_scales(int W, size_t N, const float* const* grad, const float* const* err, float* scales) {
    if (W < 1 || W > OR_MAX_RANKS || N == 0) return -1;
    for (int r = 0; r < W; r++) {
        l1_sum_t sum;
        memset(&sum, 0, sizeof(sum));
        for (size_t e = 0; e < N; e++) {
            float p = grad[r][e] + err[r][e];
            l1_add(&sum, p);
        }
        scales[r] = l1_mean(&sum, (uint64_t)N);
    }
    return 0;
}

/* Given the scales: every rank's element decodes to q = +s_r if p >= 0 and
 * -s_r otherwise (sign(p) times the scale), the carried error becomes
 * e_r = p - q (fp32), and the decoded values are reduced exactly as the
 * all-reduce reduces its contributions (same chunks, same ring or tree order;
 * avg pre-scales each q by fl32(1/W)).  mode 0 writes the result to every
 * out[j] (N elements), mode 1 writes chunk k to out[k] (N/W elements). */
int or_sign_ef_collective(int mode, int op, int algo, int W, size_t N, const float* const* grad,
                          float* const* err, const float* scales, void* const* out) {
    plan_t P;
    if (op != OR_SUM && op != OR_AVG) return -1;
    if (make_plan(&P, OR_FP32, op, algo, W, N) != 0) return -1;
    if (mode == 1 && N % (size_t)W != 0) return -1;
    for (int k = 0; k < W; k++) {
        size_t lo = or_chunk_lo(W, N, k), hi = or_chunk_lo(W, N, k + 1);
        for (size_t e = lo; e < hi; e++) {
            acc_t y[OR_MAX_RANKS];
            for (int r = 0; r < W; r++) {
                float p = grad[r][e] + err[r][e];
                float q = (p >= 0.0f) ? scales[r] : -scales[r];
                err[r][e] = p - q;
                y[r].f = (op == OR_AVG) ? q * P.s : q;
            }
            acc_t acc = reduce_position(&P, k, e, y);
            if (mode == 0) {
                for (int j = 0; j < W; j++) store_result(OR_FP32, op, W, acc, out[j], e);
            } else {
                store_result(OR_FP32, op, W, acc, out[k], e - lo);
            }
        }
    }
    return 0;
}
