/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the element-wise
 * arithmetic of all-reduce, reduce-scatter and all-gather over W simulated
 * rank buffers.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may link or call this code.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * includes this header.
 *
 * Every routine is written from the method's own definitions:
 *   - "What all-reduce promises" and "The ring, exactly as the kernel runs it"
 *     (rakshithvasudev.github.io, post on NCCL all-reduce): the contract,
 *     the five reduction ops, avg as a 1/n pre-scale for floats and one
 *     divide of the finished sum for integers, and the ring schedule in which
 *     a chunk's running total gains one neighbour per hop;
 *   - "The double binary tree" (same post): the bit-trick tree, the mirrored
 *     or shifted second tree, each tree carrying half of the buffer;
 *   - "All-gather: everyone shows their piece" and "Why backward needs a
 *     different collective" (FSDP collectives 101): all-gather as
 *     concatenation, reduce-scatter as "each rank keeps its own slice";
 *   - Eq. (2), "Local shard bounds" (NCCL M2N paper): chunk bounds
 *     l = floor(i * S / D).
 *
 * Data is passed as host arrays.  Element types: 0 = fp32, 1 = bf16 (raw
 * 16-bit patterns, fp32 accumulation, one round-to-nearest-even at the end),
 * 2 = int32 (two's complement, wrapping).  Ops: 0 sum, 1 prod, 2 min, 3 max,
 * 4 avg.  Algorithms: 0 ring, 1 tree.
 *
 * Parity unpinned: NaN and infinity payloads through min/max and through the
 * bf16 rounding (kept out of all test data).
 */
#ifndef MR_ORACLE_H
#define MR_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_FP32 = 0, OR_BF16 = 1, OR_INT32 = 2 };
enum { OR_SUM = 0, OR_PROD = 1, OR_MIN = 2, OR_MAX = 3, OR_AVG = 4 };
enum { OR_RING = 0, OR_TREE = 1, OR_HIER = 2 };

#define OR_MAX_RANKS 64

/* Round an fp32 value to the nearest bf16, ties to even. */
uint16_t or_f32_to_bf16_rne(float x);
/* Apply or_f32_to_bf16_rne to n fp32 bit patterns (for exhaustive tests). */
void or_f32_to_bf16_rne_array(const uint32_t* in, uint16_t* out, size_t n);

/* Lower bound of chunk k of an N-element buffer split W ways: floor(k*N/W). */
size_t or_chunk_lo(int W, size_t N, int k);

/* Ring accumulation order of chunk k: order[0..W-1] = k+1, k+2, ..., k (mod W). */
void or_ring_order(int W, int k, int* order);

/*
 * Tree `which` (1 or 2) over W ranks.  parent[r] = -1 for the root; child[2r],
 * child[2r+1] are r's children in ascending order (-1 if absent).
 * Returns the root.
 */
int or_tree_build(int W, int which, int* parent, int* child);

/* The three collectives.  Return 0 on success, -1 on a bad argument.
 *   allreduce:      in[r], out[r]: N elements each; every out[r] gets the result.
 *   reduce_scatter: in[r]: N elements; out[k]: N/W elements (chunk k). N % W == 0.
 *   all_gather:     in[k]: N/W elements (shard k); out[j]: N elements.  N % W == 0.
 * Output pointers may repeat (the same buffer W times) when a test only keeps
 * one copy of an all-reduce result. */
int or_allreduce(int dtype, int op, int algo, int W, size_t N,
                 const void* const* in, void* const* out);
int or_reduce_scatter(int dtype, int op, int algo, int W, size_t N,
                      const void* const* in, void* const* out);
int or_all_gather(int dtype, int W, size_t N,
                  const void* const* in, void* const* out);

/* The same with a choice of order: algo OR_RING, OR_TREE or OR_HIER (groups
 * of `group` ranks, W % group == 0: ring reduce-scatter inside the groups,
 * ring all-reduce across them); hop = 1 rounds a bf16 running total to bf16
 * after every combine (no effect for fp32 and int32). */
int or_allreduce_ex(int dtype, int op, int algo, int group, int hop, int W, size_t N,
                    const void* const* in, void* const* out);
int or_reduce_scatter_ex(int dtype, int op, int algo, int group, int hop, int W, size_t N,
                         const void* const* in, void* const* out);

/* Reduce a single element position: y[0..W-1] are rank r's raw values at
 * global element e of an N-element buffer (used to check sampled outputs of
 * very large runs one by one).  Writes the raw result to *res. */
int or_reduce_one(int dtype, int op, int algo, int W, size_t N, size_t e,
                  const void* y, void* res);

/* All-reduce (sum) of `rows` x `hidden` elements, then h = sum + residual
 * (residual may be NULL) and out[j] = RMSNorm(h) * weight for every j;
 * residual_out (may be NULL) receives h.  fp32 / bf16 only.  The norm is
 * evaluated in fp64 from the fp32 h. */
int or_allreduce_rmsnorm(int dtype, int algo, int W, size_t rows, size_t hidden,
                         const void* const* in, const void* residual, const void* weight, double eps,
                         void* const* out, void* residual_out);

/* 1-bit sign compression with error feedback (fp32 only).
 * or_sign_ef_scales: s_r = ||g_r + e_r||_1 / N for every rank: the exact
 *   sum of the magnitudes, divided exactly by N, rounded once to the nearest
 *   fp32 (ties to even); NaN if any p is NaN, else +inf if any |p| is.
 * or_sign_ef_collective: with the given scales, decode q = sign(p) * s_r,
 * update err[r] = p - q in place, and reduce the q (sum or avg) into out:
 * mode 0 all-reduce (out[j]: N elements), mode 1 reduce-scatter (out[k]:
 * N/W elements). */
int or_sign_ef_scales(int W, size_t N, const float* const* grad, const float* const* err, float* scales);
int or_sign_ef_collective(int mode, int op, int algo, int W, size_t N, const float* const* grad,
                          float* const* err, const float* scales, void* const* out);

#ifdef __cplusplus
}
#endif

#endif
