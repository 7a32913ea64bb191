/*
 * mr.h -- collective reduction math on one GPU.
 *
 * The element-wise arithmetic of all-reduce, reduce-scatter and all-gather over
 * W rank buffers that all live in the HBM of one GPU ("simulated ranks").  No
 * byte crosses to another GPU: rank r is simply the r-th pointer of an array.
 *
 * Sources (page title, section):
 *   [AR]   post on NCCL all-reduce (rakshithvasudev.github.io), "What all-reduce
 *          promises": one same-shaped tensor per rank, combined element-wise
 *          with sum, prod, min, max or avg; every rank ends with the identical
 *          result.  avg pre-scales each float contribution by 1/n as it is read
 *          and divides an integer sum once at the end.
 *   [RING] same post, "The ring, exactly as the kernel runs it": the buffer is
 *          cut into n chunks; chunk k's running total starts on one rank and
 *          gains one neighbour's contribution per hop over n-1 hops; all-reduce
 *          is reduce-scatter followed by all-gather, fused.
 *   [TREE] same post, "The double binary tree": the bit-trick binary tree, the
 *          mirrored (even n) or shifted (odd n) second tree, each tree carrying
 *          half of the buffer.
 *   [FSDP] FSDP collectives 101, "All-gather: everyone shows their piece" and
 *          "Why backward needs a different collective": all-gather concatenates
 *          the shards; reduce-scatter leaves rank k holding slice k of the
 *          reduced result.
 *   [EQ2]  NCCL M2N, Eq. (2), "Local shard bounds": chunk k of an N-element
 *          buffer split W ways starts at floor(k*N/W).
 *
 * Conventions shared by all three collectives:
 *   - send and recv are HOST arrays of W DEVICE pointers.  The library copies
 *     both arrays into the kernel's parameter block before it returns, so the
 *     caller may free or reuse them immediately.
 *   - Buffers are dense 1-D arrays of `dtype` elements: fp32, bf16 (IEEE
 *     bfloat16 bit patterns) or int32.  Every pointer must be non-NULL and
 *     aligned to its element size; 16-byte alignment enables the vectorised
 *     path, anything else runs the element-wise path on the GPU.
 *   - Arithmetic: fp32 and bf16 accumulate in fp32, one IEEE operation per
 *     step, round to nearest even, no fused multiply-add; bf16 results are
 *     rounded to bf16 once, at the end.  int32 sum and prod wrap modulo 2^32;
 *     int32 avg is the C truncating divide of the wrapped sum by W.  min and
 *     max order -0 below +0.
 *   - Accumulation order (this decides float rounding): MR_RING folds chunk k
 *     of the buffer (elements [floor(kN/W), floor((k+1)N/W))) in rank order
 *     k+1, k+2, ..., k (mod W).  MR_TREE reduces elements [0, floor(N/2)) up
 *     tree 1 and the rest up tree 2, each node adding its children's subtotals
 *     to its own contribution (own value first, then the children in tree-1
 *     position order).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and is asynchronous: the call never synchronises, allocates no
 *     device memory and creates no streams.  Execution errors surface at the
 *     caller's next synchronisation.  N == 0 launches nothing and returns MR_OK.
 *   - Kernels are launched with programmatic dependent launch: a launch may
 *     begin while the kernel before it on the stream is finishing, and waits
 *     for that kernel to complete before it reads or writes any buffer, so
 *     stream order holds exactly as for a plain launch (also under CUDA graph
 *     capture).  Setting MR_PDL=0 in the environment before the first call
 *     launches every kernel in plain stream order instead.
 *   - MR_DEBUG=1 in the environment logs each call's plan (the order MR_AUTO
 *     chose, segments, grid) to stderr.
 *   - Errors in arguments return at once and launch nothing; a failed launch
 *     returns MR_ERR_CUDA.  mr_last_error() then describes the failure.
 *   - Allowed aliasing (in place) is listed per call; any other overlap between
 *     the 2W byte ranges returns MR_ERR_ALIAS.
 */
#ifndef MR_H
#define MR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MR_MAX_RANKS 64

typedef enum { MR_FP32 = 0, MR_BF16 = 1, MR_INT32 = 2 } mr_dtype_t;
typedef enum { MR_SUM = 0, MR_PROD = 1, MR_MIN = 2, MR_MAX = 3, MR_AVG = 4 } mr_op_t;
typedef enum { MR_RING = 0, MR_TREE = 1, MR_HIER = 2, MR_AUTO = 3 } mr_algo_t;
typedef enum {
    MR_OK = 0,
    MR_ERR_INVALID_ARGUMENT = 1, /* W out of [1, 64], NULL or misaligned pointer,
                                    N % W != 0 where required, bad enum value */
    MR_ERR_UNSUPPORTED = 2,      /* a well-formed request outside what the call
                                    supports (int32 for the fused RMSNorm) */
    MR_ERR_ALIAS = 3,            /* buffers overlap other than in an allowed form */
    MR_ERR_CUDA = 4              /* the CUDA runtime refused the launch */
} mr_status_t;

/*
 * All-reduce [AR][RING][TREE]: recv[j][e] = result(e) for every rank j.
 *   send[r], recv[r]: N elements each; any N >= 0 (chunks by [EQ2]).
 *   In place: recv[r] == send[r] for every r.
 * One kernel reads W*N and writes W*N elements (reduce-scatter and all-gather
 * fused into one pass).
 */
mr_status_t mr_allreduce(const void* const* send, void* const* recv, int W, size_t N,
                         mr_dtype_t dtype, mr_op_t op, mr_algo_t algo, void* stream);

/*
 * Reduce-scatter [FSDP][RING][TREE]: recv[k][i] = result(k*C + i), C = N / W.
 *   send[r]: N elements; recv[k]: C elements (chunk k).  N % W == 0 required.
 *   The element order of `result` is the all-reduce's (same chunks, same
 *   tree split), so reduce-scatter followed by all-gather equals all-reduce
 *   bit for bit.
 *   In place: recv[r] == send[r] + r*C (in elements) for every r.
 */
mr_status_t mr_reduce_scatter(const void* const* send, void* const* recv, int W, size_t N,
                              mr_dtype_t dtype, mr_op_t op, mr_algo_t algo, void* stream);

/*
 * All-gather [FSDP]: recv[j][k*C + i] = send[k][i] for every j, C = N / W.
 *   send[k]: C elements (shard k); recv[j]: N elements.  N % W == 0 required.
 *   A pure copy: no arithmetic.
 *   In place: send[r] == recv[r] + r*C (in elements) for every r.
 */
mr_status_t mr_all_gather(const void* const* send, void* const* recv, int W, size_t N,
                          mr_dtype_t dtype, void* stream);

/*
 * All-reduce with the residual add and RMSNorm fused after the sum [NORM]:
 * the buffer is `rows` rows of `hidden` elements (N = rows * hidden).  For
 * every element,
 *     s = sum over ranks of send[r][e]   (exactly as mr_allreduce with MR_SUM
 *                                          and `algo`: same chunks, same order,
 *                                          fp32 accumulation)
 *     h = s + residual[e]                  (one fp32 add; skipped if residual
 *                                          is NULL)
 * residual_out[e] (if non-NULL) receives h rounded to `dtype`.  For every row,
 *     ss  = sum of h*h over the row (fp32: a per-thread partial in element
 *           order, then a fixed tree -- the same on every run),
 *     inv = 1 / sqrt(ss / hidden + eps),
 *     recv[j][e] = (h * inv) * weight[e mod hidden], rounded once to dtype,
 * for every rank j.  Each step is one IEEE fp32 operation; no FMA.
 *   send[r], recv[r]: N elements; residual, residual_out: N elements or NULL;
 *   weight: hidden elements (not NULL).  dtype MR_FP32 or MR_BF16 (MR_INT32
 *   returns MR_ERR_UNSUPPORTED).  1 <= hidden <= 49152.  rows == 0 is a no-op.
 *   In place: recv[r] == send[r], and residual_out == residual, are allowed.
 *   The simulated ranks share one residual stream and one weight vector.
 * [NORM] post on NCCL all-reduce, "How this survives ten thousand GPUs": in
 * decoding, the merge (residual add) and the RMSNorm that follow the
 * all-reduce are fused into it.
 */
mr_status_t mr_allreduce_rmsnorm(const void* const* send, void* const* recv, int W, size_t rows, size_t hidden,
                                 const void* residual, void* residual_out, const void* weight, float eps,
                                 mr_dtype_t dtype, mr_algo_t algo, void* stream);

/*
 * 1-bit sign compression with error feedback, then the reduction [SIGN]
 * (fp32 only).  For every rank r and element e:
 *     p = grad[r][e] + err[r][e]                 (one fp32 add)
 *     s_r = ||p_r||_1 / N                        (L1 norm of the whole rank
 *                                                 buffer over N: the exact sum
 *                                                 of the |p| divided exactly by
 *                                                 N, rounded once to the nearest
 *                                                 fp32, ties to even -- a
 *                                                 function of the data alone;
 *                                                 NaN if any p is NaN, else +inf
 *                                                 if any |p| is infinite)
 *     q = +s_r if p >= 0 else -s_r               (the 1-bit code, decoded)
 *     err[r][e] = p - q                          (what was not sent: carried to
 *                                                 the next step)
 * and the q are reduced across ranks exactly as mr_allreduce reduces its
 * contributions (op MR_SUM or MR_AVG -- avg pre-scales each q by fl32(1/W) --,
 * same chunks, same ring or tree order):
 *   mr_allreduce_sign_ef:      recv[j] (N elements) gets the result, every j;
 *                              in place: recv[r] == grad[r].
 *   mr_reduce_scatter_sign_ef: recv[k] (N/W elements) gets chunk k; N % W == 0;
 *                              in place: recv[r] == grad[r] + r*N/W.
 *   grad[r]: N elements (read); err[r]: N elements (read, then overwritten);
 *   scales: W floats of device memory, receives s_r (may be NULL);
 *   workspace: device memory of at least mr_sign_ef_workspace_bytes(W, N)
 *   bytes (at most 90112 for any W and N), owned by the caller, 8-byte
 *   aligned; its contents need no initialisation and are scratch after the
 *   call.  Calls that share a workspace must not run concurrently.  Other ops
 *   return MR_ERR_UNSUPPORTED; N >= 2^37 returns MR_ERR_INVALID_ARGUMENT.
 *   Two kernels are launched on `stream`.
 * [SIGN] "Communication Optimization: Gradient Compression, NCCL ..."
 * (mbrenndoerfer.com): 1-bit SGD sends sign(g) with the scale ||g||_1 / d;
 * error feedback compresses g plus the residual owed from the previous step
 * and keeps the part that was not sent.
 */
size_t mr_sign_ef_workspace_bytes(int W, size_t N);
mr_status_t mr_allreduce_sign_ef(const void* const* grad, void* const* err, void* const* recv, float* scales,
                                 int W, size_t N, mr_op_t op, mr_algo_t algo, void* workspace,
                                 size_t workspace_bytes, void* stream);
mr_status_t mr_reduce_scatter_sign_ef(const void* const* grad, void* const* err, void* const* recv, float* scales,
                                      int W, size_t N, mr_op_t op, mr_algo_t algo, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * mr_reduce_scatter_sign_ef_noalloc: mr_reduce_scatter_sign_ef for callers
 * that cannot allocate device memory -- for example a plugin that is handed
 * only the tensors it works on, a runtime whose device memory belongs to
 * another allocator, or a latency-critical loop that cannot pay for
 * cudaMalloc's implicit synchronisation.  The pages have no counterpart: this
 * is an interface variant, not part of the method.
 *   Same arguments, results and errors as mr_reduce_scatter_sign_ef, without
 *   the workspace: the scratch is a 96 KiB array of device memory inside the
 *   library (every GPU that loads the library holds it until the process
 *   exits).  That is more than any W and N need (at most 90112 bytes of
 *   partials), so no size is refused for want of scratch.  Nothing here calls
 *   cudaMalloc, cudaFree or any allocating routine.
 *   The first call on each device (and the first after a device reset) looks
 *   up the array's device address with that device current; make that first
 *   call before any stream capture.
 *   Every call uses the same array: each call writes all the partials it
 *   later reads, so nothing needs clearing between calls, but calls that
 *   overlap on the GPU (other streams, other threads) race on it.
 */
mr_status_t mr_reduce_scatter_sign_ef_noalloc(const void* const* grad, void* const* err, void* const* recv,
                                              float* scales, int W, size_t N, mr_op_t op, mr_algo_t algo,
                                              void* stream);

/*
 * All-reduce and reduce-scatter with a choice of accumulation order [HIER]:
 *   order->algo == MR_RING or MR_TREE: as mr_allreduce / mr_reduce_scatter.
 *   order->algo == MR_HIER: the ranks form G = W / group groups of `group`
 *     consecutive ranks (rank a*group + i is local rank i of group a);
 *     group must divide W.  Element e lies in chunk c of the buffer cut into
 *     `group` chunks ([EQ2] bounds), and in piece d of chunk c cut into G
 *     pieces.  Each group first folds its own ranks in local ring order
 *     c+1, ..., c (the ring reduce-scatter inside a group), then the G group
 *     totals are folded in group ring order d+1, ..., d (the ring all-reduce
 *     across groups); the all-gather inside the groups copies.  group == W or
 *     group == 1 gives exactly MR_RING.
 *   order->per_hop_rounding == 1 (bf16 only; no effect on fp32 and int32):
 *     the running total is rounded to bf16 after every combine (and a
 *     pre-scaled avg contribution as it is read), as when every partial sum
 *     crosses a wire as bf16 -- NCCL's own bf16 reduction.  0: fp32
 *     accumulation and one final rounding, as in every other call.
 * The other arguments, results, aliasing rules and errors are those of
 * mr_allreduce and mr_reduce_scatter; a NULL order is MR_RING with fp32
 * accumulation.
 * [HIER] "Communication Optimization: Gradient Compression, NCCL ..."
 * (mbrenndoerfer.com): the two-level all-reduce -- local reduce-scatter,
 * node-level all-reduce of the partial sums, local all-gather; FSDP
 * collectives 101: NCCL's bf16 reduction accumulates in bf16.
 */
typedef struct {
    mr_algo_t algo;
    int group;              /* ranks per group, MR_HIER only */
    int per_hop_rounding;   /* 0 or 1 */
} mr_order_t;

mr_status_t mr_allreduce_ex(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                            mr_op_t op, const mr_order_t* order, void* stream);
mr_status_t mr_reduce_scatter_ex(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                                 mr_op_t op, const mr_order_t* order, void* stream);

/* A static, human-readable name of a status code. */
const char* mr_status_string(mr_status_t status);

/* Detail of the last non-OK status returned on the calling thread ("" if none).
 * The string is owned by the library and valid until the thread's next call. */
const char* mr_last_error(void);

/*
 * MR_AUTO [COST]: wherever an algo is taken (except inside mr_order_t's
 * MR_HIER), MR_AUTO picks MR_RING or MR_TREE per call as the argmin of the
 * alpha-beta model  t = alpha + bytes / beta  of each order, with alpha and
 * beta fitted on GB300 per element type and rank count (the table the library
 * is built with; collective_reduction_math_gb300/tune_cost_model.py refits it
 * on another GPU).  bytes is the call's HBM traffic.  The choice depends only
 * on (dtype, W, N, call), so results are reproducible; they equal those of
 * the order chosen, which mr_plan_auto reports.  Integer ops and min / max
 * give the same result in either order.
 *   mr_plan_auto: *algo receives MR_RING or MR_TREE and *predicted_us (if not
 *   NULL) the model's time; reduce_scatter = 0 for all-reduce traffic
 *   (2 W N b bytes), 1 for reduce-scatter ((W + 1) N b).
 * [COST] post on NCCL all-reduce, "How NCCL picks: a cost model, not a
 * threshold": time = lat * latCount + nBytes / bw, argmin per call.
 */
mr_status_t mr_plan_auto(int W, size_t N, mr_dtype_t dtype, int reduce_scatter, mr_algo_t* algo,
                         double* predicted_us);

/*
 * Planner queries (host only; no GPU needed).  They expose the orders the
 * kernels use.
 *   mr_plan_ring_order: order[0..W-1] = the ranks that chunk k visits [RING].
 *   mr_plan_tree: tree `which` (1 or 2) [TREE]; parent[r] (-1 at the root) and
 *     child[2r], child[2r+1] (-1 if absent, tree-1 position order).  Returns
 *     the root rank in *root.
 *   mr_chunk_lo: floor(k*N/W) [EQ2].
 */
mr_status_t mr_plan_ring_order(int W, int k, int* order);
mr_status_t mr_plan_tree(int W, int which, int* parent, int* child, int* root);
size_t mr_chunk_lo(int W, size_t N, int k);

/* Number of kernels this library has launched in this process (all threads,
 * all devices).  Lets a caller count the GPU launches inside a timed region. */
unsigned long long mr_launch_count(void);

/*
 * mr_launch_floor: launch one empty kernel of `ctas` CTAs (1..65535) of the
 * library's block size on `stream`, with the launch attributes every kernel
 * here gets (programmatic dependent launch unless MR_PDL=0).  It reads and
 * writes nothing.  Timed beside a small collective, it separates the cost of
 * a launch from the kernel's own work.  The pages have no counterpart: this
 * is a measuring aid.  Returns MR_ERR_INVALID_ARGUMENT for ctas out of
 * range, MR_ERR_CUDA if the launch fails; counts in mr_launch_count().
 */
mr_status_t mr_launch_floor(unsigned ctas, void* stream);

#ifdef __cplusplus
}
#endif

#endif
