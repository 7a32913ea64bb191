// order.cuh -- the accumulation orders, usable on host (planner) and device
// (kernels).
//
// Ring ("The ring, exactly as the kernel runs it", post on NCCL all-reduce):
// ranks form the ring 0 -> 1 -> ... -> W-1 -> 0; chunk k's running total
// starts on rank k+1 and gains one neighbour per hop until it completes on
// rank k, its owner.  Position i of chunk k's order is rank (k+1+i) mod W.
//
// Tree ("The double binary tree", same post): tree 1 is described by tree
// POSITIONS p in [0, W).  The lowest set bit b of p fixes its level (the root,
// p = 0, sits above every level).  Position p has a lower child p - b/2 (when
// b > 1) and an upper child p + h for the largest h in {b/2, b/4, ..., 1} that
// stays inside [0, W); the root's only child is the largest power of two
// below W.  Its parent is p with b cleared and the next bit set, or just with
// b cleared when that falls outside the ranks.  Tree 1 puts rank p at
// position p.  Tree 2 puts rank W-1-p at position p when W is even (the
// mirror image) and rank (p+1) mod W when W is odd (the shift by one), so
// leaves of one tree are interior in the other.
//
// A node's subtotal is its own contribution, then (+) the lower child's
// subtotal, then (+) the upper child's.  Elements [0, floor(N/2)) use tree 1,
// the rest tree 2.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define MR_HD __host__ __device__ __forceinline__
#else
#define MR_HD inline
#endif

namespace mr {

MR_HD int pow2_at_least(int W) {
    int B = 1;
    while (B < W) B <<= 1;
    return B;
}

MR_HD int ring_rank(int W, int k, int i) {
    int r = k + 1 + i;
    while (r >= W) r -= W;
    return r;
}

// Rank that sits at tree-1 position p in tree t (0 = tree 1, 1 = tree 2).
MR_HD int tree_rank(int W, int t, int p) {
    if (t == 0) return p;
    if ((W & 1) == 0) return W - 1 - p;
    return (p + 1 == W) ? 0 : p + 1;
}

// Level bit of position p (the root takes the smallest power of two >= W).
MR_HD int tree_level(int W, int p) { return p == 0 ? pow2_at_least(W) : (p & -p); }

MR_HD int tree_lower_child(int W, int p) {
    int b = tree_level(W, p);
    return (p > 0 && b > 1) ? p - (b >> 1) : -1;
}

MR_HD int tree_upper_child(int W, int p) {
    int b = tree_level(W, p);
    for (int h = b >> 1; h >= 1; h >>= 1)
        if (p + h < W) return p + h;
    return -1;
}

MR_HD int tree_parent(int W, int p) {
    if (p == 0) return -1;
    int b = p & -p;
    int q = (p & ~b) | (b << 1);
    return q < W ? q : (p & ~b);
}

// Hierarchical order (groups of g consecutive ranks, G = W/g groups):
// position p = (group position) * g + (local position); the group at group
// position j is (d+1+j) mod G, the local rank at local position i is
// (c+1+i) mod g, where c is the element's chunk of g and d its piece of G.
MR_HD int hier_rank(int W, int g, int c, int d, int p) {
    const int G = W / g;
    return ring_rank(G, d, p / g) * g + ring_rank(g, c, p % g);
}

// floor(k*N/W) without forming k*N.
MR_HD uint64_t chunk_lo(int W, uint64_t N, int k) {
    uint64_t q = N / (uint64_t)W, r = N % (uint64_t)W;
    return (uint64_t)k * q + ((uint64_t)k * r) / (uint64_t)W;
}

}  // namespace mr
