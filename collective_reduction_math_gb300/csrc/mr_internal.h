// mr_internal.h -- kernel parameter blocks and launchers shared by the C ABI
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mr.h"

namespace mr {

constexpr int kMaxRanks = MR_MAX_RANKS;
constexpr int kMaxSegments = 2 * MR_MAX_RANKS + 2;
constexpr int kThreads = 256;       // threads per CTA for every kernel
constexpr int kGatherBytesPerThread = 128;   // bytes each thread loads per all-gather tile
constexpr int kGatherBlocksPerSm = 16;  // all-gather CTAs per SM in the grid (several waves)

// A run of elements with one accumulation order and one output placement:
// a chunk of the ring, or a chunk cut at the tree-1 / tree-2 boundary.
struct Segment {
    uint64_t lo, hi;    // global element range [lo, hi)
    uint64_t out_lo;    // reduce-scatter: element e goes to recv[k][e - out_lo]
    int32_t k;          // the chunk (its owner rank)
    int32_t tree;       // 0: tree 1, 1: tree 2 (tree algorithm only)
    int32_t hc, hd;     // hierarchical order: chunk of `group`, piece of that chunk
};

enum { MODE_ALLREDUCE = 0, MODE_REDUCE_SCATTER = 1 };

struct ReduceParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    Segment seg[kMaxSegments];
    uint64_t tile_start[kMaxSegments + 1];   // tiles of segments [0, i) (prefix count)
    uint64_t tiles_max;                      // most tiles of any one segment
    int W;
    int nseg;
    int mode;
    int vec;        // 1: every pointer (and every reduce-scatter chunk start) is
                    // aligned to the vector width, so the vector path may run
    float scale;    // fl32(1/W): the float avg pre-scale
    int group;      // hierarchical order: ranks per group
    int hop;        // 1: round a bf16 running total to bf16 after every combine
    uint64_t gmask; // hierarchical order: bit p set where order position p starts a group
    uint32_t spread_smem;   // dynamic shared memory every CTA reserves at least, so that a
                            // grid of fewer CTAs than resident slots spreads over the SMs
};

// All-reduce + residual + RMSNorm (rows x hidden elements).
struct NormParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    const void* residual;       // may be null
    void* residual_out;         // may be null
    const void* weight;         // hidden elements
    Segment seg[kMaxSegments];
    uint64_t rows, hidden;
    int W;
    int nseg;
    int vec;                    // 1: 16-byte (or the width's) vectors: pointers aligned, hidden % lanes == 0
    int csize;                  // CTAs per cluster; each takes a slice of a row's columns
    int pipe;                   // 1: one CTA per row (csize 1), 16-byte vectors, two row buffers:
                                //    pass 2 of a row runs in one loop with pass 1 of the CTA's next row
    uint32_t buf_f4;            // pipe: float4s from one row buffer to the next
    float eps;
};

// Largest row the fused RMSNorm keeps in shared memory (fp32 per element).
constexpr uint64_t kMaxNormHidden = 49152;
// Most CTAs in one of its clusters (one row spread over up to 8 SMs).
constexpr int kMaxNormCluster = 8;

// 1-bit sign compression with error feedback (fp32).
struct SignParams {
    const void* grad[kMaxRanks];
    void* err[kMaxRanks];       // read, then overwritten with the new residual
    void* out[kMaxRanks];
    uint32_t* partials;         // workspace: per rank, kL1Words words x nb blocks (word-major)
    float* scales;              // W scales out (device)
    Segment seg[kMaxSegments];
    uint64_t tile_start[kMaxSegments + 1];
    uint64_t tiles_max;
    uint64_t N;
    int W;
    int nseg;
    int mode;
    int vec;                    // 1: every pointer (and reduce-scatter chunk start) aligned to
                                //    sign_vector_bytes(W): the decode kernel's vector path
    int l1_vec;                 // 1: grad and err 16-byte aligned: the L1 kernel's 16-byte loads
    int nb;                     // L1 blocks per rank
    float avg;                  // fl32(1/W)
};

// Exact L1 sums.  The magnitude of a finite fp32 is an integer multiple of
// 2^-149 (the smallest subnormal) below 2^277 of those units, so a sum of up
// to 2^43 magnitudes is an integer below 2^320: ten 32-bit limbs.  A block's
// partial is those ten limbs (carries propagated) and a flags word (bit 0: an
// infinite |p| was seen, bit 1: a NaN).
constexpr int kL1Limbs = 10;
constexpr int kL1Words = kL1Limbs + 1;
// The largest N the sign path takes: the scale's final division keeps the
// sum's top 64 bits, and N below 2^37 leaves at least 26 quotient bits.
constexpr uint64_t kSignMaxN = 1ull << 37;

// L1 blocks per rank: one per 8192 elements, at most 2048 / W (so a call
// never needs more than 2048 partials), at least one.  This sizes the
// workspace; a launch may use fewer blocks (one wave of the GPU).
inline int sign_blocks(int W, uint64_t N) {
    const uint64_t cap = (uint64_t)(2048 / (W < 1 ? 1 : W));
    const uint64_t nb = (N + 8191) / 8192;
    return (int)(nb < 1 ? 1 : nb > cap ? cap : nb);
}
// Workspace of the sign path: the partials, in bytes.
inline uint64_t sign_workspace_bytes(int W, uint64_t N) {
    return (uint64_t)W * (uint64_t)kL1Words * (uint64_t)sign_blocks(W, N) * sizeof(uint32_t);
}
constexpr uint64_t kSignMaxWorkspaceBytes = 2048ull * kL1Words * sizeof(uint32_t);
// Vector width of the decode-and-reduce kernel for a given W.
constexpr int sign_vector_bytes(int W) { return W <= 8 ? 16 : W <= 16 ? 8 : 4; }

struct GatherParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    uint64_t C;     // elements per shard
    int W;
    int esize;      // bytes per element (2 or 4)
    int vec;        // 2: 32-byte vectors, 1: 16-byte vectors (every pointer and
                    // C*esize aligned to the width), 0: element by element
};

// The reduce kernel variant for a given W: register slots for W contributions
// (WCAP), vector width in bytes, vectors per thread per tile (U) and resident
// CTAs per SM.  All-reduce keeps about eight 16-byte loads in flight per
// thread (U*W ~ 8) at 3 CTAs per SM up to W = 8.  Reduce-scatter stores one
// vector per W loads, and at W = 8 runs faster with two vectors per thread at
// 2 CTAs per SM (measured on GB300: 6.8 against 5.8 TB/s).
// Above 16 ranks the tree takes 32 slots (4 batch heads) up to 32 ranks and
// 64 (8 heads) beyond; the left folds take 64 at any W above 16 (their
// batched fold does not depend on the slot count).
constexpr int reduce_wcap(int W, int algo) {
    return W <= 2 ? 2 : W <= 4 ? 4 : W <= 8 ? 8 : W <= 16 ? 16 : (algo == MR_TREE && W <= 32) ? 32 : 64;
}
// Per-hop bf16 sum and avg, and bf16 min and max (on 16-bit order keys; not
// in the plain 16-slot fold), fold packed pairs (two lanes per 32-bit word).
// The host asks this of the batched trees over 32 and 64 slots only.
constexpr bool reduce_pairs(int dtype, int op, bool hop) {
    return dtype == MR_BF16 && ((hop && (op == MR_SUM || op == MR_AVG)) || op == MR_MIN || op == MR_MAX);
}
// Every variant of the reduce kernel moves 16-byte vectors; the host's
// alignment check and the kernel's templates both take the width from here.
constexpr int kReduceVectorBytes = 16;
// The batched trees over 32 and 64 slots keep their batches' in-batch top
// subtotals (one per unit: a lane, or a packed pair of bf16 lanes) in shared
// memory, per thread, instead of registers: each is written once and read
// once.
constexpr bool reduce_top_shared(int wcap, int algo) { return wcap >= 32 && algo == MR_TREE; }
constexpr size_t reduce_top_shared_bytes(int wcap, int units) {
    return (size_t)(wcap / 8) * units * kThreads * sizeof(uint32_t);
}
// The variants whose live state does not fit 80 registers: the 64-slot
// batched trees (8 heads of 4 or 8 units beside a batch of 8 vectors; the
// 32-slot tree keeps 4).
constexpr bool reduce_wide_heads(int wcap, int algo) { return wcap == 64 && algo == MR_TREE; }
// The fused RMSNorm kernel keeps all W values of a lane in registers and so
// narrows its vectors to 4 bytes above 16 ranks.
constexpr int norm_vector_bytes(int W) { return W <= 16 ? 16 : 4; }
constexpr int reduce_unroll_for(int wcap, bool rs) {
    return wcap == 2 ? 4 : wcap == 4 ? 2 : (wcap == 8 && rs) ? 2 : 1;
}
constexpr int reduce_unroll(int W, int algo, bool rs) { return reduce_unroll_for(reduce_wcap(W, algo), rs); }
// Resident CTAs per SM (the kernel's launch bounds and the grid's size): 3 for
// the all-reduce up to 8 ranks and for the batched folds (8 vectors live at a
// time), except the 64-slot trees, else 2.  At 2 per SM the batched W = 16
// folds sat at 24 % of warps active, stalled on loads (ncu, int32 W = 16: 74 %
// of DRAM peak); above 16 ranks 3 per SM took the rings from 5.3-5.6 to
// 6.1-6.2 TB/s at W = 17 and the 32-slot trees from 4.9-5.2 to 5.7-6.0.
constexpr int reduce_blocks_per_sm(int wcap, int u, bool batch, bool wide_heads) {
    return ((wcap <= 8 && wcap * u <= 8) || (batch && !wide_heads)) ? 3 : 2;
}
// Whether the reduce kernel for (W, order, element type, per-hop rounding)
// folds in batches of 8: only 8 vectors and no pointers live in registers, so
// it runs at 3 CTAs per SM (16 slots) where the plain 16-slot fold runs at 2.
// Measured on GB300 at 32 MiB per rank (TB/s, plain -> batched):
//   tree from 9 ranks, every element type: fp32 max W = 9 4.63 -> 6.13,
//     int32 sum W = 11 5.04 -> 5.88, int32 max W = 12 5.90 -> 6.23;
//   rings (and the hierarchical order) at 9 to 11 ranks: bf16 max W = 9
//     5.58 -> 5.92, per-hop bf16 avg W = 10 5.26 -> 6.21;
//   at 12 ranks the plain ring stays 1-3.5 % ahead (bf16 max 6.23 against
//     6.01), except per-hop (5.75 -> 6.03); the hierarchical order does not
//     (groups of 3, 4 or 6: fp32 sum 5.48-5.50 -> 6.27-6.28, bf16 max
//     4.83-4.87 -> 6.16-6.19, int32 sum 5.28-5.32 -> 6.24-6.26);
//   from 13 ranks every order batched (at W = 16 with 3 CTAs per SM: int32
//     sum ring 5.88 -> 6.28 at 16 MiB per rank, per-hop bf16 ring 6.10 ->
//     6.37).
constexpr int kBatchFromRanks = 13;
constexpr bool reduce_batched(int W, int algo, int dtype, bool hop) {
    (void)dtype;
    if (W >= kBatchFromRanks) return true;
    if (W <= 8) return false;
    if (algo == MR_TREE || algo == MR_HIER) return true;
    return W < 12 || hop;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation allowed, so its launch (CTA placement,
// parameter fetch) may begin while the kernel before it on the stream is
// still finishing.  Each kernel therefore first waits on `griddepcontrol.wait`
// (which returns once every grid it depends on has completed and its memory
// is visible) before its first global-memory access, and only then signals
// `griddepcontrol.launch_dependents`, so the next launch may start while this
// one runs but never more than one kernel ahead: signalling before the wait
// lets every queued launch cascade onto the SMs as idle waiting CTAs, which
// was measured on GB300 to halve the all-gather's speed.  Results are the same
// as with plain stream order; only the gap between launches shrinks.  Kernels
// launched without the attribute (or with MR_PDL=0) see both instructions as
// no-ops.
// ---------------------------------------------------------------------------
bool pdl_enabled();     // MR_PDL in the environment ("0" turns it off); default on

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Launch `k` on `s` with programmatic stream serialisation (when enabled)
// and, when cluster > 0, as 1-D thread-block clusters of that many CTAs.
template <class... Exp, class... Act>
inline cudaError_t launch_kernel(void (*k)(Exp...), dim3 grid, size_t smem, cudaStream_t s, unsigned cluster,
                                 Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Act&&>(args)...);
}

#define MR_DECLARE_REDUCE(dt, algo) \
    cudaError_t launch_reduce_##dt##_##algo(const ReduceParams& P, int op, dim3 grid, cudaStream_t s);
MR_DECLARE_REDUCE(fp32, ring)
MR_DECLARE_REDUCE(fp32, tree)
MR_DECLARE_REDUCE(fp32, hier)
MR_DECLARE_REDUCE(bf16, ring)
MR_DECLARE_REDUCE(bf16, tree)
MR_DECLARE_REDUCE(bf16, hier)
MR_DECLARE_REDUCE(bf16, ring_hop)
MR_DECLARE_REDUCE(bf16, tree_hop)
MR_DECLARE_REDUCE(bf16, hier_hop)
MR_DECLARE_REDUCE(int32, ring)
MR_DECLARE_REDUCE(int32, tree)
MR_DECLARE_REDUCE(int32, hier)
#undef MR_DECLARE_REDUCE
// smem: dynamic shared memory each CTA reserves (none used; it caps residency).
cudaError_t launch_all_gather(const GatherParams& P, dim3 grid, size_t smem, cudaStream_t s);
// Resident all-gather CTAs per SM on the current device (its registers' limit).
int all_gather_resident_per_sm();
mr_status_t report_error(mr_status_t st, const char* fmt, ...);
cudaError_t launch_sign_l1(const SignParams& P, cudaStream_t s);
// Supplies a workspace (pointer and size) for the sign path.
using ScratchFn = cudaError_t (*)(void** workspace, size_t* bytes);
mr_status_t run_sign_ef(const char* what, int mode, const void* const* grad, void* const* err, void* const* recv,
                        float* scales, int W, size_t N, mr_op_t op, mr_algo_t algo, void* workspace,
                        size_t workspace_bytes, void* stream, ScratchFn scratch = nullptr);
cudaError_t launch_sign_ef(const SignParams& P, int op, int algo, dim3 grid, cudaStream_t s);
cudaError_t launch_allreduce_rmsnorm(const NormParams& P, int dtype, int algo, dim3 grid, size_t smem, cudaStream_t s);

}  // namespace mr
