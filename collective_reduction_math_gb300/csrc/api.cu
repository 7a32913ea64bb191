// api.cu -- the C ABI: argument validation, alias checks, the chunk-segment
// planner and kernel dispatch.  See include/mr.h for the contract.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <math.h>

#include <algorithm>
#include <atomic>
#include <string>

#include "mr.h"
#include "mr_internal.h"
#include "order.cuh"

namespace {

thread_local std::string g_last_error;
std::atomic<unsigned long long> g_launches{0};

int debug_level() {
    static const int level = [] {
        const char* e = getenv("MR_DEBUG");
        return e ? atoi(e) : 0;
    }();
    return level;
}

mr_status_t fail(mr_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

size_t elem_bytes(mr_dtype_t dt) { return dt == MR_BF16 ? 2u : 4u; }

// The alpha-beta cost model of the orders (t = alpha + bytes / beta), fitted
// on GB300 per element type, rank count and order, and per range of a call's
// buffers: latency-bound, L2-resident, streaming from HBM (as NCCL keeps one
// (lat, bw) pair per protocol, each serving its own range of sizes).
struct CostPair {
    double alpha_us, beta_gbs;
};
struct CostRow {
    int dtype, W, algo;
    CostPair range[3];   // latency, L2, HBM
};
// kCostModelLatencyBytes, kCostModelL2Bytes and kCostModel[].
#include "cost_model.inc"

double model_us(mr_dtype_t dtype, int W, mr_algo_t algo, double bytes, double footprint) {
    // the row of the smallest tabulated W that covers W, else of the largest
    const CostRow* row = nullptr;
    const CostRow* largest = nullptr;
    for (const CostRow& c : kCostModel) {
        if (c.dtype != (int)dtype || c.algo != (int)algo) continue;
        if (c.W >= W && (!row || c.W < row->W)) row = &c;
        if (!largest || c.W > largest->W) largest = &c;
    }
    if (!row) row = largest;
    if (!row) return 1e30;
    const CostPair& p = row->range[footprint <= kCostModelLatencyBytes ? 0 : footprint <= kCostModelL2Bytes ? 1 : 2];
    return p.alpha_us + bytes / (p.beta_gbs * 1e3);
}

// MR_AUTO: the order with the smaller modelled time (ring on a tie).
mr_algo_t resolve_auto(mr_dtype_t dtype, int W, size_t N, bool rs, double* predicted) {
    const double b = (double)elem_bytes(dtype) * (double)N * (rs ? (double)(W + 1) : 2.0 * W);
    // the buffers the call touches: W inputs, and W outputs of N (all-reduce) or N/W (reduce-scatter)
    const double footprint = (double)elem_bytes(dtype) * (double)N * (rs ? (double)(W + 1) : 2.0 * W);
    const double tr = model_us(dtype, W, MR_RING, b, footprint), tt = model_us(dtype, W, MR_TREE, b, footprint);
    if (predicted) *predicted = tt < tr ? tt : tr;
    return tt < tr ? MR_TREE : MR_RING;
}
const char* dtype_name(mr_dtype_t dt) { return dt == MR_FP32 ? "fp32" : dt == MR_BF16 ? "bf16" : "int32"; }
const char* op_name(mr_op_t op) {
    static const char* n[] = {"sum", "prod", "min", "max", "avg"};
    return n[op];
}
const char* algo_name(mr_algo_t a) {
    return a == MR_RING ? "ring" : a == MR_TREE ? "tree" : a == MR_HIER ? "hier" : "auto";
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64) {
        int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 148;
    }
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

mr_status_t check_common(const void* const* send, void* const* recv, int W, mr_dtype_t dtype) {
    if (W < 1 || W > MR_MAX_RANKS)
        return fail(MR_ERR_INVALID_ARGUMENT, "W = %d is outside [1, %d]", W, MR_MAX_RANKS);
    if (dtype != MR_FP32 && dtype != MR_BF16 && dtype != MR_INT32)
        return fail(MR_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dtype);
    if (!send || !recv) return fail(MR_ERR_INVALID_ARGUMENT, "send or recv pointer array is NULL");
    return MR_OK;
}

mr_status_t check_pointers(const void* const* send, void* const* recv, int W, mr_dtype_t dtype) {
    const uintptr_t a = elem_bytes(dtype) - 1;
    for (int r = 0; r < W; ++r) {
        if (!send[r]) return fail(MR_ERR_INVALID_ARGUMENT, "send[%d] is NULL", r);
        if (!recv[r]) return fail(MR_ERR_INVALID_ARGUMENT, "recv[%d] is NULL", r);
        if ((uintptr_t)send[r] & a)
            return fail(MR_ERR_INVALID_ARGUMENT, "send[%d] is not aligned to its %s element", r, dtype_name(dtype));
        if ((uintptr_t)recv[r] & a)
            return fail(MR_ERR_INVALID_ARGUMENT, "recv[%d] is not aligned to its %s element", r, dtype_name(dtype));
    }
    return MR_OK;
}

mr_status_t check_op_algo(mr_op_t op, mr_algo_t algo) {
    if (op < MR_SUM || op > MR_AVG) return fail(MR_ERR_INVALID_ARGUMENT, "unknown op %d", (int)op);
    if (algo == MR_HIER)
        return fail(MR_ERR_INVALID_ARGUMENT, "MR_HIER needs a group size: use mr_allreduce_ex / mr_reduce_scatter_ex");
    if (algo != MR_RING && algo != MR_TREE && algo != MR_AUTO)
        return fail(MR_ERR_INVALID_ARGUMENT, "unknown algo %d", (int)algo);
    return MR_OK;
}

// Overlap check over byte ranges.  Two ranges may overlap only when
// `allowed(a, b)` says so (an in-place form); every other pair of non-empty
// ranges must be disjoint.  Sort by start, then sweep with the set of ranges
// still open (which stays tiny when the buffers are disjoint).
enum RangeKind { SEND = 0, RECV = 1, RESIDUAL = 2, RESIDUAL_OUT = 3, WEIGHT = 4, ERR = 5, SCALES = 6, WORKSPACE = 7 };
const char* kind_name(int k) {
    static const char* n[] = {"send", "recv", "residual", "residual_out", "weight", "err", "scales", "workspace"};
    return n[k];
}

struct Range {
    uintptr_t lo, hi;
    int rank;
    int kind;
};

template <class Allowed>
mr_status_t check_overlaps(Range* rs, int n, Allowed allowed) {
    std::sort(rs, rs + n, [](const Range& a, const Range& b) { return a.lo < b.lo; });
    int open[3 * MR_MAX_RANKS + 8];
    int nopen = 0;
    for (int i = 0; i < n; ++i) {
        int keep = 0;
        for (int j = 0; j < nopen; ++j) {
            const Range& o = rs[open[j]];
            if (o.hi <= rs[i].lo) continue;        // closed before this one starts
            open[keep++] = open[j];
            if (!allowed(o, rs[i]) && !allowed(rs[i], o))
                return fail(MR_ERR_ALIAS, "%s[%d] overlaps %s[%d] in a form that is not an allowed in-place one",
                            kind_name(o.kind), o.rank, kind_name(rs[i].kind), rs[i].rank);
        }
        nopen = keep;
        open[nopen++] = i;
    }
    return MR_OK;
}

// The send/recv ranges of the collectives: rank r's pair may overlap only
// when `inplace(r)` holds.
template <class InPlace>
mr_status_t check_alias(const void* const* send, size_t send_bytes, void* const* recv, size_t recv_bytes,
                        int W, InPlace inplace) {
    Range rs[2 * MR_MAX_RANKS];
    int n = 0;
    for (int r = 0; r < W; ++r) {
        if (send_bytes) rs[n++] = {(uintptr_t)send[r], (uintptr_t)send[r] + send_bytes, r, SEND};
        if (recv_bytes) rs[n++] = {(uintptr_t)recv[r], (uintptr_t)recv[r] + recv_bytes, r, RECV};
    }
    return check_overlaps(rs, n, [&](const Range& a, const Range& b) {
        return a.kind == SEND && b.kind == RECV && a.rank == b.rank && inplace(a.rank);
    });
}

// Segments of [0, N): each chunk k = [floor(kN/W), floor((k+1)N/W)), cut at
// floor(N/2) for the tree algorithm (tree 1 below, tree 2 from there on).
int plan_segments(int W, uint64_t N, mr_algo_t algo, mr::Segment* seg) {
    int n = 0;
    const uint64_t half = N / 2;
    for (int k = 0; k < W; ++k) {
        const uint64_t lo = mr::chunk_lo(W, N, k), hi = mr::chunk_lo(W, N, k + 1);
        if (lo == hi) continue;
        if (algo == MR_TREE && lo < half && half < hi) {
            seg[n++] = {lo, half, lo, k, 0, 0, 0};
            seg[n++] = {half, hi, lo, k, 1, 0, 0};
        } else {
            seg[n++] = {lo, hi, lo, k, (algo == MR_TREE && lo >= half) ? 1 : 0, 0, 0};
        }
    }
    return n;
}

// Tile counts per segment (prefix sums into P.tile_start, the largest in
// P.tiles_max) and the 1-D grid: a few CTAs per SM, never more than there are
// tiles.
// Segments of the hierarchical order: each chunk c of `group` chunks cut into
// its G = W / group pieces; for reduce-scatter also cut at the W chunk bounds,
// which place the output.
int plan_segments_hier(int W, uint64_t N, int group, bool cut_at_chunks, mr::Segment* seg) {
    const int G = W / group;
    uint64_t b[2 * MR_MAX_RANKS + 2];
    int nb = 0;
    for (int c = 0; c < group; ++c) {
        const uint64_t clo = mr::chunk_lo(group, N, c), clen = mr::chunk_lo(group, N, c + 1) - clo;
        for (int d = 0; d < G; ++d) b[nb++] = clo + mr::chunk_lo(G, clen, d);
    }
    b[nb++] = N;
    if (cut_at_chunks)
        for (int k = 1; k < W; ++k) b[nb++] = mr::chunk_lo(W, N, k);
    std::sort(b, b + nb);
    nb = (int)(std::unique(b, b + nb) - b);
    int n = 0, k = 0, c = 0, d = 0;
    for (int i = 0; i + 1 < nb; ++i) {
        const uint64_t lo = b[i], hi = b[i + 1];
        if (lo == hi) continue;
        while (mr::chunk_lo(W, N, k + 1) <= lo) ++k;
        while (mr::chunk_lo(group, N, c + 1) <= lo) { ++c; d = 0; }
        const uint64_t clo = mr::chunk_lo(group, N, c), clen = mr::chunk_lo(group, N, c + 1) - clo;
        while (clo + mr::chunk_lo(G, clen, d + 1) <= lo) ++d;
        seg[n++] = {lo, hi, mr::chunk_lo(W, N, k), k, 0, c, d};
    }
    return n;
}

// Dynamic shared memory each CTA of a one-wave grid reserves so that the
// grid spreads over the SMs: with more than 1.25 CTAs per SM but fewer than
// the resident slots, the block scheduler measured to put up to `resident`
// CTAs on some SMs while others stayed idle; reserving 227 KB / (cap + 1)
// per CTA leaves room for at most cap = ceil(grid / SMs).  Measured (back to
// back, warm L2): the W = 8 fp32 all-reduce at 228-300 tiles 13-17 % faster,
// W = 32 at 200 tiles 11 %, the all-gather at 256 CTAs 17-24 %, the fused
// RMSNorm at 256-300 rows 13-16 %; from 1.05 to 1.25 CTAs per SM it cost
// up to 3 % and is not taken.  0: no reservation.
size_t spread_smem(uint64_t grid, uint64_t resident) {
    const uint64_t sms = (uint64_t)sm_count();
    if (4 * grid <= 5 * sms || grid >= sms * resident) return 0;
    const uint64_t cap = (grid + sms - 1) / sms;
    if (cap >= resident) return 0;
    return (size_t)((227 * 1024) / (cap + 1) + 1024);
}

dim3 plan_tiles(mr::ReduceParams& P, int algo, int lanes, bool batched, bool wide_heads) {
    const bool rs = P.mode == mr::MODE_REDUCE_SCATTER;
    const int u = mr::reduce_unroll(P.W, algo, rs);
    const uint64_t per_tile = P.vec ? (uint64_t)mr::kThreads * u : (uint64_t)mr::kThreads;
    P.tile_start[0] = 0;
    P.tiles_max = 0;
    for (int i = 0; i < P.nseg; ++i) {
        const mr::Segment& g = P.seg[i];
        uint64_t units = g.hi - g.lo;
        if (P.vec) {
            const uint64_t va = (g.lo + lanes - 1) / lanes, vb = g.hi / lanes;
            units = va < vb ? vb - va : 0;
        }
        P.tile_start[i + 1] = P.tile_start[i] + (units + per_tile - 1) / per_tile;
        P.tiles_max = std::max(P.tiles_max, P.tile_start[i + 1] - P.tile_start[i]);
    }
    const uint64_t vtiles = P.vec ? P.tiles_max * P.nseg : P.tile_start[P.nseg];
    const uint64_t tiles = std::max<uint64_t>(vtiles, (uint64_t)P.nseg);
    const int per_sm = mr::reduce_blocks_per_sm(mr::reduce_wcap(P.W, algo), u, batched, wide_heads);
    const uint64_t full = (uint64_t)sm_count() * per_sm;
    uint64_t gx = std::min<uint64_t>(full, tiles);
    // Tile t goes to CTA t mod gx and segment t mod nseg, so with gx a
    // multiple of nseg every CTA stays on one segment for the whole call and
    // no CTA helps a segment that falls behind.  Above 8 segments (the batched
    // folds) that left a tail that grew with the call (W = 57 fp32 ring at 64
    // MiB per rank 5082 GB/s, W = 24 5668, W = 19 5607); a grid one or more
    // CTAs smaller, sharing no factor with nseg, deals every CTA's tiles
    // across all segments (5960, 6206, 6328).  Up to 8 segments (57 or more
    // CTAs per segment, the plain folds) the fixed assignment measured 3.6 %
    // faster (W = 8 fp32 ring) and stays.  A grid capped by the tile count
    // (a small call: one tile per CTA, or a few) keeps one CTA per tile.
    if (P.vec && P.nseg > 8 && gx == full && gx % (uint64_t)P.nseg == 0) {
        auto gcd = [](uint64_t a, uint64_t b) {
            while (b) {
                const uint64_t t = a % b;
                a = b;
                b = t;
            }
            return a;
        };
        while (gx > 1 && gcd(gx, (uint64_t)P.nseg) != 1) --gx;
    }
    // A one-wave grid with more CTAs than SMs is spread over them (at 1 MiB
    // per rank, 256 CTAs: W = 8 fp32 ring 3.43 -> 3.02 us, W = 16 5.67 ->
    // 4.83, W = 32 10.08 -> 8.52, W = 64 26.1 -> 23.3).
    P.spread_smem = (uint32_t)spread_smem(gx, (uint64_t)per_sm);
    return dim3((unsigned)std::max<uint64_t>(gx, 1), 1, 1);
}

cudaError_t launch_reduce(mr_dtype_t dtype, const mr::ReduceParams& P, mr_op_t op, mr_algo_t algo,
                          dim3 grid, cudaStream_t s) {
    switch (dtype) {
        case MR_FP32:
            return algo == MR_RING ? mr::launch_reduce_fp32_ring(P, op, grid, s)
                 : algo == MR_TREE ? mr::launch_reduce_fp32_tree(P, op, grid, s)
                                   : mr::launch_reduce_fp32_hier(P, op, grid, s);
        case MR_BF16:
            if (P.hop)
                return algo == MR_RING ? mr::launch_reduce_bf16_ring_hop(P, op, grid, s)
                     : algo == MR_TREE ? mr::launch_reduce_bf16_tree_hop(P, op, grid, s)
                                       : mr::launch_reduce_bf16_hier_hop(P, op, grid, s);
            return algo == MR_RING ? mr::launch_reduce_bf16_ring(P, op, grid, s)
                 : algo == MR_TREE ? mr::launch_reduce_bf16_tree(P, op, grid, s)
                                   : mr::launch_reduce_bf16_hier(P, op, grid, s);
        case MR_INT32:
            return algo == MR_RING ? mr::launch_reduce_int32_ring(P, op, grid, s)
                 : algo == MR_TREE ? mr::launch_reduce_int32_tree(P, op, grid, s)
                                   : mr::launch_reduce_int32_hier(P, op, grid, s);
    }
    return cudaErrorInvalidValue;
}

mr_status_t run_reduce(const char* what, int mode, const void* const* send, void* const* recv, int W, size_t N,
                       mr_dtype_t dtype, mr_op_t op, mr_algo_t algo, void* stream, int group = 0, int hop = 0) {
    const bool is_auto = algo == MR_AUTO;
    double predicted = 0.0;
    if (is_auto) algo = resolve_auto(dtype, W, N, mode == mr::MODE_REDUCE_SCATTER, &predicted);
    mr::ReduceParams P;
    for (int r = 0; r < W; ++r) {
        P.in[r] = send[r];
        P.out[r] = recv[r];
    }
    P.W = W;
    P.mode = mode;
    P.scale = (float)(1.0 / (double)W);
    P.group = algo == MR_HIER ? group : W;
    P.hop = hop;
    P.gmask = 0;
    for (int p = 0; p < W; p += P.group) P.gmask |= 1ull << p;
    P.nseg = algo == MR_HIER ? plan_segments_hier(W, N, group, mode == mr::MODE_REDUCE_SCATTER, P.seg)
                             : plan_segments(W, N, algo, P.seg);
    const int eb = (int)elem_bytes(dtype);
    const int vb = mr::kReduceVectorBytes;
    bool vec = true;
    for (int r = 0; r < W; ++r)
        vec = vec && ((uintptr_t)send[r] % vb == 0) && ((uintptr_t)recv[r] % vb == 0);
    if (mode == mr::MODE_REDUCE_SCATTER) vec = vec && ((N / W) * eb) % vb == 0;
    P.vec = vec ? 1 : 0;
    const dim3 grid = plan_tiles(P, algo, vb / eb, mr::reduce_batched(W, algo, dtype, hop != 0),
                                 mr::reduce_wide_heads(mr::reduce_wcap(W, algo), algo));
    const cudaError_t err = launch_reduce(dtype, P, op, algo, grid, (cudaStream_t)stream);
    if (err != cudaSuccess)
        return fail(MR_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(err));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (debug_level() > 0 && is_auto)
        fprintf(stderr, "[mr] %s auto -> %s (model %.2f us)\n", what, algo_name(algo), predicted);
    if (debug_level() > 0)
        fprintf(stderr, "[mr] %s dtype=%s op=%s algo=%s group=%d per_hop=%d W=%d N=%zu segments=%d tiles=%llu "
                "vector=%d grid=%u threads=%d spread_smem=%u sms=%d\n",
                what, dtype_name(dtype), op_name(op), algo_name(algo), P.group, P.hop, W, N, P.nseg,
                (unsigned long long)P.tile_start[P.nseg], P.vec, grid.x, mr::kThreads, P.spread_smem, sm_count());
    return MR_OK;
}

}  // namespace

namespace mr {
// A kernel that does nothing but enter and leave like every other kernel here
// (the programmatic-dependent-launch wait and signal): the launch floor.
__global__ void __launch_bounds__(kThreads) empty_kernel(int) { pdl_enter(); }

bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("MR_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// Records `fmt` as the calling thread's last error and returns `st` (for
// entry points defined in other translation units).
mr_status_t report_error(mr_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}
}  // namespace mr

extern "C" {

mr_status_t mr_allreduce(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                         mr_op_t op, mr_algo_t algo, void* stream) {
    g_last_error.clear();
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st == MR_OK) st = check_op_algo(op, algo);
    if (st != MR_OK || N == 0) return st;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const size_t bytes = N * elem_bytes(dtype);
    st = check_alias(send, bytes, recv, bytes, W, [&](int r) { return send[r] == recv[r]; });
    if (st != MR_OK) return st;
    return run_reduce("allreduce", mr::MODE_ALLREDUCE, send, recv, W, N, dtype, op, algo, stream);
}

mr_status_t mr_reduce_scatter(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                              mr_op_t op, mr_algo_t algo, void* stream) {
    g_last_error.clear();
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st == MR_OK) st = check_op_algo(op, algo);
    if (st != MR_OK) return st;
    if (N % (size_t)W != 0)
        return fail(MR_ERR_INVALID_ARGUMENT, "reduce_scatter needs N (%zu) divisible by W (%d)", N, W);
    if (N == 0) return MR_OK;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const size_t b = elem_bytes(dtype), C = N / (size_t)W;
    st = check_alias(send, N * b, recv, C * b, W, [&](int r) {
        return (const char*)recv[r] == (const char*)send[r] + (size_t)r * C * b;
    });
    if (st != MR_OK) return st;
    return run_reduce("reduce_scatter", mr::MODE_REDUCE_SCATTER, send, recv, W, N, dtype, op, algo, stream);
}

mr_status_t mr_all_gather(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                          void* stream) {
    g_last_error.clear();
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st != MR_OK) return st;
    if (N % (size_t)W != 0)
        return fail(MR_ERR_INVALID_ARGUMENT, "all_gather needs N (%zu) divisible by W (%d)", N, W);
    if (N == 0) return MR_OK;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const size_t b = elem_bytes(dtype), C = N / (size_t)W;
    st = check_alias(send, C * b, recv, N * b, W, [&](int r) {
        return (const char*)send[r] == (const char*)recv[r] + (size_t)r * C * b;
    });
    if (st != MR_OK) return st;

    mr::GatherParams P;
    for (int r = 0; r < W; ++r) {
        P.in[r] = send[r];
        P.out[r] = recv[r];
    }
    P.W = W;
    P.C = C;
    P.esize = (int)b;
    auto aligned = [&](size_t a) {
        bool ok = (C * b) % a == 0;
        for (int r = 0; r < W; ++r) ok = ok && ((uintptr_t)send[r] % a == 0) && ((uintptr_t)recv[r] % a == 0);
        return ok;
    };
    P.vec = aligned(32) ? 2 : aligned(16) ? 1 : 0;
    const int vb = P.vec == 2 ? 32 : 16;
    const uint64_t per_tile = P.vec ? (uint64_t)mr::kThreads * (mr::kGatherBytesPerThread / vb) : (uint64_t)mr::kThreads;
    const uint64_t units = P.vec ? (C * b) / vb : C;
    const uint64_t tiles = std::max<uint64_t>(1, (units + per_tile - 1) / per_tile) * (uint64_t)W;
    const uint64_t sms = (uint64_t)sm_count();
    const uint64_t gx = std::min<uint64_t>(sms * mr::kGatherBlocksPerSm, tiles);
    const dim3 grid((unsigned)gx, 1, 1);
    // A one-wave grid of more CTAs than SMs is spread over them.
    const size_t smem = spread_smem(gx, (uint64_t)mr::all_gather_resident_per_sm());
    const cudaError_t err = mr::launch_all_gather(P, grid, smem, (cudaStream_t)stream);
    if (err != cudaSuccess) return fail(MR_ERR_CUDA, "all_gather launch failed: %s", cudaGetErrorString(err));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (debug_level() > 0)
        fprintf(stderr, "[mr] all_gather dtype=%s W=%d N=%zu vector=%d grid=%u threads=%d\n", dtype_name(dtype),
                W, N, P.vec, grid.x, mr::kThreads);
    return MR_OK;
}

static mr_status_t check_order(const mr_order_t* order, int W, mr_algo_t* algo, int* group, int* hop) {
    *algo = MR_RING;
    *group = W;
    *hop = 0;
    if (!order) return MR_OK;
    if (order->algo != MR_RING && order->algo != MR_TREE && order->algo != MR_HIER && order->algo != MR_AUTO)
        return fail(MR_ERR_INVALID_ARGUMENT, "unknown algo %d", (int)order->algo);
    if (order->per_hop_rounding != 0 && order->per_hop_rounding != 1)
        return fail(MR_ERR_INVALID_ARGUMENT, "per_hop_rounding must be 0 or 1");
    if (order->algo == MR_HIER && (order->group < 1 || order->group > W || W % order->group != 0))
        return fail(MR_ERR_INVALID_ARGUMENT, "group = %d must divide W = %d", order->group, W);
    *algo = order->algo;
    *group = order->algo == MR_HIER ? order->group : W;
    *hop = order->per_hop_rounding;
    return MR_OK;
}

mr_status_t mr_allreduce_ex(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                            mr_op_t op, const mr_order_t* order, void* stream) {
    g_last_error.clear();
    mr_algo_t algo;
    int group, hop;
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st == MR_OK) st = check_op_algo(op, MR_RING);
    if (st == MR_OK) st = check_order(order, W, &algo, &group, &hop);
    if (st != MR_OK || N == 0) return st;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const size_t bytes = N * elem_bytes(dtype);
    st = check_alias(send, bytes, recv, bytes, W, [&](int r) { return send[r] == recv[r]; });
    if (st != MR_OK) return st;
    return run_reduce("allreduce_ex", mr::MODE_ALLREDUCE, send, recv, W, N, dtype, op, algo, stream, group, hop);
}

mr_status_t mr_reduce_scatter_ex(const void* const* send, void* const* recv, int W, size_t N, mr_dtype_t dtype,
                                 mr_op_t op, const mr_order_t* order, void* stream) {
    g_last_error.clear();
    mr_algo_t algo;
    int group, hop;
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st == MR_OK) st = check_op_algo(op, MR_RING);
    if (st == MR_OK) st = check_order(order, W, &algo, &group, &hop);
    if (st != MR_OK) return st;
    if (N % (size_t)W != 0)
        return fail(MR_ERR_INVALID_ARGUMENT, "reduce_scatter needs N (%zu) divisible by W (%d)", N, W);
    if (N == 0) return MR_OK;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const size_t b = elem_bytes(dtype), C = N / (size_t)W;
    st = check_alias(send, N * b, recv, C * b, W, [&](int r) {
        return (const char*)recv[r] == (const char*)send[r] + (size_t)r * C * b;
    });
    if (st != MR_OK) return st;
    return run_reduce("reduce_scatter_ex", mr::MODE_REDUCE_SCATTER, send, recv, W, N, dtype, op, algo, stream, group,
                      hop);
}

// Shared memory a fused-RMSNorm CTA of a multi-CTA cluster reserves, so that
// no more than two fit on one SM (228 KB of shared memory per SM, 1 KB of it
// reserved per CTA).
constexpr size_t kNormSpreadSmem = 80 * 1024;

mr_status_t mr_allreduce_rmsnorm(const void* const* send, void* const* recv, int W, size_t rows, size_t hidden,
                                 const void* residual, void* residual_out, const void* weight, float eps,
                                 mr_dtype_t dtype, mr_algo_t algo, void* stream) {
    g_last_error.clear();
    mr_status_t st = check_common(send, recv, W, dtype);
    if (st == MR_OK) st = check_op_algo(MR_SUM, algo);
    if (st != MR_OK) return st;
    if (dtype == MR_INT32) return fail(MR_ERR_UNSUPPORTED, "allreduce_rmsnorm takes fp32 or bf16, not int32");
    if (hidden < 1 || hidden > mr::kMaxNormHidden)
        return fail(MR_ERR_INVALID_ARGUMENT, "hidden = %zu is outside [1, %llu]", hidden,
                    (unsigned long long)mr::kMaxNormHidden);
    if (!(eps >= 0.0f) || eps == INFINITY)
        return fail(MR_ERR_INVALID_ARGUMENT, "eps must be finite and >= 0");
    if (rows > (SIZE_MAX / 4) / hidden) return fail(MR_ERR_INVALID_ARGUMENT, "rows * hidden overflows");
    if (rows == 0) return MR_OK;
    if ((st = check_pointers(send, recv, W, dtype)) != MR_OK) return st;
    const uintptr_t a = elem_bytes(dtype) - 1;
    if (!weight) return fail(MR_ERR_INVALID_ARGUMENT, "weight is NULL");
    if (((uintptr_t)weight & a) || ((uintptr_t)residual & a) || ((uintptr_t)residual_out & a))
        return fail(MR_ERR_INVALID_ARGUMENT, "weight, residual or residual_out is not aligned to its element");
    const size_t N = rows * hidden, b = elem_bytes(dtype), bytes = N * b;

    Range rs[2 * MR_MAX_RANKS + 3];
    int n = 0;
    for (int r = 0; r < W; ++r) {
        rs[n++] = {(uintptr_t)send[r], (uintptr_t)send[r] + bytes, r, SEND};
        rs[n++] = {(uintptr_t)recv[r], (uintptr_t)recv[r] + bytes, r, RECV};
    }
    if (residual) rs[n++] = {(uintptr_t)residual, (uintptr_t)residual + bytes, 0, RESIDUAL};
    if (residual_out) rs[n++] = {(uintptr_t)residual_out, (uintptr_t)residual_out + bytes, 0, RESIDUAL_OUT};
    rs[n++] = {(uintptr_t)weight, (uintptr_t)weight + hidden * b, 0, WEIGHT};
    st = check_overlaps(rs, n, [](const Range& x, const Range& y) {
        const bool same = x.lo == y.lo && x.hi == y.hi;
        return same && ((x.kind == SEND && y.kind == RECV && x.rank == y.rank) ||
                        (x.kind == RESIDUAL && y.kind == RESIDUAL_OUT));
    });
    if (st != MR_OK) return st;

    if (algo == MR_AUTO) algo = resolve_auto(dtype, W, N, false, nullptr);
    mr::NormParams P;
    for (int r = 0; r < W; ++r) {
        P.in[r] = send[r];
        P.out[r] = recv[r];
    }
    P.residual = residual;
    P.residual_out = residual_out;
    P.weight = weight;
    P.rows = rows;
    P.hidden = hidden;
    P.W = W;
    P.eps = eps;
    P.nseg = plan_segments(W, N, algo, P.seg);
    const int vb = mr::norm_vector_bytes(W);
    const size_t lanes = vb / b;
    bool vec = hidden % lanes == 0;
    for (int r = 0; r < W; ++r) vec = vec && ((uintptr_t)send[r] % vb == 0) && ((uintptr_t)recv[r] % vb == 0);
    vec = vec && ((uintptr_t)weight % vb == 0) && ((uintptr_t)residual % vb == 0) && ((uintptr_t)residual_out % vb == 0);
    P.vec = vec ? 1 : 0;
    // A cluster of csize CTAs per row at a time; each CTA keeps its slice of
    // the row's fp32 values in shared memory.  Few rows (decode): spread each
    // row over up to 8 SMs, as long as every CTA keeps at least one vector
    // per thread.
    const size_t sms = (size_t)sm_count();
    int csize = 1;
    while (csize < 8 && rows * (size_t)(csize * 2) <= 2 * sms && hidden / lanes / (size_t)(csize * 2) >= mr::kThreads)
        csize *= 2;
    P.csize = csize;
    const size_t slice = (hidden + csize - 1) / csize + lanes;
    // The row slice in shared memory.  Spread over a cluster (few rows), a
    // CTA also reserves enough shared memory that at most two of them share
    // an SM: three of the 256 decode CTAs on one SM left it with half as much
    // again to load and store as the rest (per-phase timestamps, W = 8, 64 x
    // 8192 bf16: 5.97 against 5.50 us per step).
    const size_t buf_bytes = ((slice * 4 + 15) / 16) * 16;
    size_t smem = buf_bytes;
    if (csize > 1) smem = std::max<size_t>(smem, kNormSpreadSmem);
    // One whole wave of resident CTAs, looping over the rows.  Residency is
    // the smaller of what the kernel's register budget allows (3 per SM up to
    // 8 ranks, 2 up to 16, else 1: its launch bounds) and what shared memory
    // allows (227 KB per SM, the row slice plus about 1 KB per CTA).  A grid
    // that left a partial last wave measured up to 10 % slower on GB300
    // (W = 8 bf16, hidden 12288: 5032 against 5546 GB/s).
    const size_t reg_resident = W <= 8 ? 3 : W <= 16 ? 2 : 1;
    auto resident = [&](size_t bytes) {
        return std::min(reg_resident, std::max<size_t>(1, (227 * 1024) / (bytes + 1024)));
    };
    size_t per_sm = resident(smem);
    // One CTA per row with several rows each (up to 16 ranks): a second row
    // buffer lets pass 2 of a row and pass 1 of the next share one loop.  That
    // variant runs at 2 CTAs per SM (its launch bounds), and is taken where
    // both buffers fit twice per SM and an element's W contributions take more
    // than 8 bytes.  Measured on GB300, 4096 x 8192 rows (GB/s, one row loop
    // at 3 CTAs per SM -> pipelined at 2): bf16 W = 8 5969 -> 6158, W = 5
    // 5209 -> 5285, fp32 W = 8 6038 -> 6547, W = 3 4983 -> 5106; with 8
    // bytes or fewer it loses or ties (bf16 W = 4 5137 -> 4891, fp32 W = 2
    // 4354 -> 4375).
    P.buf_f4 = (uint32_t)(buf_bytes / 16);
    P.pipe = 0;
    const size_t pipe_per_sm = std::min<size_t>(2, std::max<size_t>(1, (227 * 1024) / (2 * buf_bytes + 1024)));
    if (csize == 1 && P.vec && vb == 16 && W <= 16 && (size_t)W * b > 8 && pipe_per_sm == 2 &&
        rows > sms * pipe_per_sm) {
        P.pipe = 1;
        smem = 2 * buf_bytes;
        per_sm = pipe_per_sm;
    }
    const size_t clusters = std::min<size_t>(rows, std::max<size_t>(1, sms * per_sm / csize));
    const dim3 grid((unsigned)(clusters * csize), 1, 1);
    // A one-wave grid of more CTAs than SMs is spread over them (W = 8 bf16,
    // hidden 8192, 256 and 300 rows: 17.3 -> 15.1 us, 19.9 -> 16.7 us).
    smem = std::max<size_t>(smem, spread_smem(grid.x, per_sm));
    const cudaError_t err = mr::launch_allreduce_rmsnorm(P, dtype, algo, grid, smem, (cudaStream_t)stream);
    if (err != cudaSuccess) return fail(MR_ERR_CUDA, "allreduce_rmsnorm launch failed: %s", cudaGetErrorString(err));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (debug_level() > 0)
        fprintf(stderr, "[mr] allreduce_rmsnorm dtype=%s algo=%s W=%d rows=%zu hidden=%zu vector=%d grid=%u "
                "cluster=%d smem=%zu pipelined=%d\n", dtype_name(dtype), algo_name(algo), W, rows, hidden, P.vec,
                grid.x, csize, smem, P.pipe);
    return MR_OK;
}

size_t mr_sign_ef_workspace_bytes(int W, size_t N) {
    if (W < 1 || W > MR_MAX_RANKS) return 0;
    return (size_t)mr::sign_workspace_bytes(W, N);
}

}  // extern "C"

// The sign-compressed reductions.  `scratch`, when given, supplies the
// workspace once every argument has been checked (the allocation-free entry
// point); otherwise the caller's workspace is used.
mr_status_t mr::run_sign_ef(const char* what, int mode, const void* const* grad, void* const* err,
                            void* const* recv, float* scales, int W, size_t N, mr_op_t op, mr_algo_t algo,
                            void* workspace, size_t workspace_bytes, void* stream, ScratchFn scratch) {
    g_last_error.clear();
    mr_status_t st = check_common(grad, recv, W, MR_FP32);
    if (st == MR_OK) st = check_op_algo(op, algo);
    if (st != MR_OK) return st;
    if (op != MR_SUM && op != MR_AVG) return fail(MR_ERR_UNSUPPORTED, "%s reduces with sum or avg only", what);
    if (!err) return fail(MR_ERR_INVALID_ARGUMENT, "err pointer array is NULL");
    if (mode == mr::MODE_REDUCE_SCATTER && N % (size_t)W != 0)
        return fail(MR_ERR_INVALID_ARGUMENT, "%s needs N (%zu) divisible by W (%d)", what, N, W);
    if (N == 0) return MR_OK;
    if (N >= mr::kSignMaxN)
        return fail(MR_ERR_INVALID_ARGUMENT, "%s takes N below 2^37 elements per rank (N = %zu)", what, N);
    if ((st = check_pointers(grad, recv, W, MR_FP32)) != MR_OK) return st;
    for (int r = 0; r < W; ++r)
        if (!err[r] || ((uintptr_t)err[r] & 3u)) return fail(MR_ERR_INVALID_ARGUMENT, "err[%d] is NULL or misaligned", r);
    if ((uintptr_t)scales & 3u) return fail(MR_ERR_INVALID_ARGUMENT, "scales is misaligned");
    const size_t need = mr_sign_ef_workspace_bytes(W, N);
    if (!scratch && (!workspace || ((uintptr_t)workspace & 7u) || workspace_bytes < need))
        return fail(MR_ERR_INVALID_ARGUMENT, "workspace must be 8-byte aligned and hold %zu bytes", need);

    const size_t bytes = N * 4, C = N / (size_t)W, out_bytes = mode == mr::MODE_REDUCE_SCATTER ? C * 4 : bytes;
    Range rs[3 * MR_MAX_RANKS + 2];
    int n = 0;
    for (int r = 0; r < W; ++r) {
        rs[n++] = {(uintptr_t)grad[r], (uintptr_t)grad[r] + bytes, r, SEND};
        rs[n++] = {(uintptr_t)recv[r], (uintptr_t)recv[r] + out_bytes, r, RECV};
        rs[n++] = {(uintptr_t)err[r], (uintptr_t)err[r] + bytes, r, ERR};
    }
    if (scales) rs[n++] = {(uintptr_t)scales, (uintptr_t)scales + (size_t)W * 4, 0, SCALES};
    if (!scratch) rs[n++] = {(uintptr_t)workspace, (uintptr_t)workspace + need, 0, WORKSPACE};
    st = check_overlaps(rs, n, [&](const Range& x, const Range& y) {
        if (!(x.kind == SEND && y.kind == RECV && x.rank == y.rank)) return false;
        if (mode == mr::MODE_REDUCE_SCATTER) return y.lo == x.lo + (size_t)x.rank * C * 4;
        return y.lo == x.lo;
    });
    if (st != MR_OK) return st;
    if (scratch) {
        // The library's own scratch (no caller buffer can overlap it).
        const cudaError_t e = scratch(&workspace, &workspace_bytes);
        if (e != cudaSuccess)
            return fail(MR_ERR_CUDA, "%s: locating the static scratch failed: %s", what, cudaGetErrorString(e));
        if (workspace_bytes < need)
            return fail(MR_ERR_INVALID_ARGUMENT, "%s: the static scratch holds %zu bytes, the call needs %zu", what,
                        workspace_bytes, need);
    }

    if (algo == MR_AUTO) algo = resolve_auto(MR_FP32, W, N, mode == mr::MODE_REDUCE_SCATTER, nullptr);
    mr::SignParams P;
    for (int r = 0; r < W; ++r) {
        P.grad[r] = grad[r];
        P.err[r] = err[r];
        P.out[r] = recv[r];
    }
    P.partials = static_cast<uint32_t*>(workspace);
    P.scales = scales;
    P.N = N;
    P.W = W;
    P.mode = mode;
    // L1 blocks per rank: at most one full wave of the L1 kernel over all
    // ranks (8 blocks of 256 threads per SM).  2048 blocks at W = 8 made 1.7
    // waves, the last two-thirds full; one wave measured 6342 -> 6457 GB/s for
    // the W = 8, 2^24 reduce-scatter step.  The partials are exact integer
    // sums, so the scale does not depend on the block count.
    P.nb = std::min<int>(mr::sign_blocks(W, N), std::max(1, sm_count() * 8 / W));
    P.avg = (float)(1.0 / (double)W);
    P.nseg = plan_segments(W, N, algo, P.seg);
    const int vb = mr::sign_vector_bytes(W);
    bool vec = true, l1_vec = true;
    for (int r = 0; r < W; ++r) {
        vec = vec && ((uintptr_t)grad[r] % vb == 0) && ((uintptr_t)err[r] % vb == 0) && ((uintptr_t)recv[r] % vb == 0);
        l1_vec = l1_vec && ((uintptr_t)grad[r] % 16 == 0) && ((uintptr_t)err[r] % 16 == 0);
    }
    if (mode == mr::MODE_REDUCE_SCATTER) vec = vec && (C * 4) % vb == 0;
    P.vec = vec ? 1 : 0;
    P.l1_vec = l1_vec ? 1 : 0;
    // tiles of kThreads vectors (or elements), round-robin across segments
    const uint64_t lanes = vb / 4;
    P.tile_start[0] = 0;
    P.tiles_max = 0;
    for (int i = 0; i < P.nseg; ++i) {
        const mr::Segment& g = P.seg[i];
        uint64_t units = g.hi - g.lo;
        if (P.vec) {
            const uint64_t va = (g.lo + lanes - 1) / lanes, vb2 = g.hi / lanes;
            units = va < vb2 ? vb2 - va : 0;
        }
        P.tile_start[i + 1] = P.tile_start[i] + (units + mr::kThreads - 1) / mr::kThreads;
        P.tiles_max = std::max(P.tiles_max, P.tile_start[i + 1] - P.tile_start[i]);
    }
    const uint64_t tiles = std::max<uint64_t>(P.vec ? P.tiles_max * P.nseg : P.tile_start[P.nseg], P.nseg);
    const dim3 grid((unsigned)std::min<uint64_t>((uint64_t)sm_count() * 2, tiles), 1, 1);
    cudaError_t e = mr::launch_sign_l1(P, (cudaStream_t)stream);
    if (e == cudaSuccess) {
        g_launches.fetch_add(1, std::memory_order_relaxed);
        e = mr::launch_sign_ef(P, op, algo, grid, (cudaStream_t)stream);
        if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (e != cudaSuccess) return fail(MR_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    if (debug_level() > 0)
        fprintf(stderr, "[mr] %s op=%s algo=%s W=%d N=%zu l1_blocks=%d vector=%d grid=%u\n", what, op_name(op),
                algo_name(algo), W, N, P.nb, P.vec, grid.x);
    return MR_OK;
}

extern "C" {

mr_status_t mr_allreduce_sign_ef(const void* const* grad, void* const* err, void* const* recv, float* scales,
                                 int W, size_t N, mr_op_t op, mr_algo_t algo, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    return mr::run_sign_ef("allreduce_sign_ef", mr::MODE_ALLREDUCE, grad, err, recv, scales, W, N, op, algo, workspace,
                       workspace_bytes, stream);
}

mr_status_t mr_reduce_scatter_sign_ef(const void* const* grad, void* const* err, void* const* recv, float* scales,
                                      int W, size_t N, mr_op_t op, mr_algo_t algo, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    return mr::run_sign_ef("reduce_scatter_sign_ef", mr::MODE_REDUCE_SCATTER, grad, err, recv, scales, W, N, op, algo,
                       workspace, workspace_bytes, stream);
}

const char* mr_status_string(mr_status_t status) {
    switch (status) {
        case MR_OK: return "MR_OK";
        case MR_ERR_INVALID_ARGUMENT: return "MR_ERR_INVALID_ARGUMENT";
        case MR_ERR_UNSUPPORTED: return "MR_ERR_UNSUPPORTED";
        case MR_ERR_ALIAS: return "MR_ERR_ALIAS";
        case MR_ERR_CUDA: return "MR_ERR_CUDA";
    }
    return "MR_UNKNOWN_STATUS";
}

const char* mr_last_error(void) { return g_last_error.c_str(); }

mr_status_t mr_plan_ring_order(int W, int k, int* order) {
    g_last_error.clear();
    if (W < 1 || W > MR_MAX_RANKS || k < 0 || k >= W || !order)
        return fail(MR_ERR_INVALID_ARGUMENT, "mr_plan_ring_order: bad W, k or order");
    for (int i = 0; i < W; ++i) order[i] = mr::ring_rank(W, k, i);
    return MR_OK;
}

mr_status_t mr_plan_tree(int W, int which, int* parent, int* child, int* root) {
    g_last_error.clear();
    if (W < 1 || W > MR_MAX_RANKS || (which != 1 && which != 2) || !parent || !child || !root)
        return fail(MR_ERR_INVALID_ARGUMENT, "mr_plan_tree: bad W, which or output pointer");
    const int t = which - 1;
    for (int p = 0; p < W; ++p) {
        const int r = mr::tree_rank(W, t, p);
        const int q = mr::tree_parent(W, p);
        const int lo = mr::tree_lower_child(W, p), up = mr::tree_upper_child(W, p);
        parent[r] = q < 0 ? -1 : mr::tree_rank(W, t, q);
        int n = 0;
        child[2 * r] = child[2 * r + 1] = -1;
        if (lo >= 0) child[2 * r + n++] = mr::tree_rank(W, t, lo);
        if (up >= 0) child[2 * r + n++] = mr::tree_rank(W, t, up);
    }
    *root = mr::tree_rank(W, t, 0);
    return MR_OK;
}

mr_status_t mr_plan_auto(int W, size_t N, mr_dtype_t dtype, int reduce_scatter, mr_algo_t* algo,
                         double* predicted_us) {
    g_last_error.clear();
    if (W < 1 || W > MR_MAX_RANKS || !algo || (dtype != MR_FP32 && dtype != MR_BF16 && dtype != MR_INT32))
        return fail(MR_ERR_INVALID_ARGUMENT, "mr_plan_auto: bad W, dtype or algo pointer");
    *algo = resolve_auto(dtype, W, N, reduce_scatter != 0, predicted_us);
    return MR_OK;
}

size_t mr_chunk_lo(int W, size_t N, int k) {
    if (W < 1 || k < 0 || k > W) return 0;
    return (size_t)mr::chunk_lo(W, N, k);
}

unsigned long long mr_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

mr_status_t mr_launch_floor(unsigned ctas, void* stream) {
    g_last_error.clear();
    if (ctas < 1 || ctas > 65535) return fail(MR_ERR_INVALID_ARGUMENT, "mr_launch_floor: ctas = %u is outside [1, 65535]", ctas);
    const cudaError_t e = mr::launch_kernel(mr::empty_kernel, dim3(ctas, 1, 1), 0, (cudaStream_t)stream, 0, 0);
    if (e != cudaSuccess) return fail(MR_ERR_CUDA, "launch_floor launch failed: %s", cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return MR_OK;
}

}  // extern "C"
