"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas: each compares it with a
worked example the pages print, a literal simulation of the ring schedule, the
tree diagram the pages draw, brute force over every accumulation order, an
independent library (torch) or a closed-form error bound.
"""
import itertools
import math

import numpy as np
import pytest

import synth
from golden_io import read_blocks, read_tree
from ring_sim import simulate

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _f32(xs):
    return np.array([float(x) for x in xs.split()], np.float32)


# --------------------------------------------------------------------------
# Worked examples printed on the pages
# --------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_worked_examples(oracle_mod, algo):
    blocks = read_blocks("worked_examples.txt")
    assert len(blocks) == 4
    for b in blocks:
        ins = [_f32(b["rank0"]), _f32(b["rank1"])]
        exp = [_f32(b["expect0"]), _f32(b["expect1"])]
        if b["collective"] == "allreduce":
            got = oracle_mod.allreduce("fp32", b["op"], algo, ins, all_ranks=True)
        elif b["collective"] == "reduce_scatter":
            got = oracle_mod.reduce_scatter("fp32", b["op"], algo, ins)
        else:
            got = oracle_mod.all_gather("fp32", ins, all_ranks=True)
        for g, e in zip(got, exp):
            assert g.tobytes() == e.tobytes(), (b["case"], g, e)


def test_worked_examples_other_dtypes(oracle_mod):
    """The same examples are exact in int32 and bf16."""
    a = np.array([8, 0, 4, 2], np.int32)
    b = np.array([0, 4, 8, 6], np.int32)
    assert oracle_mod.allreduce("int32", "sum", "ring", [a, b]).tolist() == [8, 4, 12, 8]
    assert oracle_mod.allreduce("int32", "avg", "ring", [a, b]).tolist() == [4, 2, 6, 4]
    rs = oracle_mod.reduce_scatter("int32", "avg", "tree", [a, b])
    assert [x.tolist() for x in rs] == [[4, 2], [6, 4]]
    bf = [synth._to_bf16_bits(a.astype(np.float32)), synth._to_bf16_bits(b.astype(np.float32))]
    out = oracle_mod.allreduce("bf16", "avg", "ring", bf)
    assert ((out.astype(np.uint32) << 16).view(np.float32)).tolist() == [4, 2, 6, 4]


# --------------------------------------------------------------------------
# The ring order against a literal simulation of the ring schedule
# --------------------------------------------------------------------------

@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("dtype,op", [("fp32", "sum"), ("fp32", "avg"), ("fp32", "prod"),
                                       ("bf16", "sum"), ("bf16", "avg"), ("bf16", "prod"),
                                       ("int32", "sum"), ("int32", "avg"), ("int32", "prod")])
@pytest.mark.parametrize("N", [6, 60, 97])
def test_ring_matches_step_simulation(oracle_mod, W, dtype, op, N):
    ins = synth.random_values(100 + W, W, N, dtype)
    sim, transfers, finisher = simulate(dtype, op, ins)
    assert transfers == 2 * (W - 1)
    assert finisher == list(range(W))          # chunk k completes on its owner, rank k
    got = oracle_mod.allreduce(dtype, op, "ring", ins, all_ranks=True)
    for r in range(W):
        assert got[r].tobytes() == sim[r].tobytes(), (r, got[r], sim[r])


def test_ring_order_examples(oracle_mod):
    # chunk k starts at rank k+1 and completes on rank k
    assert oracle_mod.ring_order(4, 0) == [1, 2, 3, 0]
    assert oracle_mod.ring_order(4, 3) == [0, 1, 2, 3]
    assert oracle_mod.ring_order(1, 0) == [0]


# --------------------------------------------------------------------------
# The trees
# --------------------------------------------------------------------------

def test_tree_matches_diagram(oracle_mod):
    parent, kids = read_tree("tree14.txt")
    root, p, c = oracle_mod.tree(14, 1)
    assert root == 0
    assert p == parent
    assert c == kids


def _check_tree(W, root, parent, kids):
    assert parent[root] == -1
    assert sum(1 for r in range(W) if parent[r] == -1) == 1
    assert sum(len(k) for k in kids) == W - 1
    for r in range(W):
        assert len(kids[r]) <= 2
        for ch in kids[r]:
            assert parent[ch] == r
    seen, stack = set(), [root]
    while stack:
        v = stack.pop()
        assert v not in seen
        seen.add(v)
        stack.extend(kids[v])
    assert seen == set(range(W))


@pytest.mark.parametrize("W", range(1, 65))
def test_trees_are_trees(oracle_mod, W):
    for which in (1, 2):
        root, parent, kids = oracle_mod.tree(W, which)
        _check_tree(W, root, parent, kids)
    # depth of tree 1 is logarithmic: at most ceil(log2 W) + 1 levels
    root, parent, kids = oracle_mod.tree(W, 1)
    depth = 0
    for r in range(W):
        d, v = 0, r
        while parent[v] != -1:
            v, d = parent[v], d + 1
        depth = max(depth, d)
    assert depth <= max(1, math.ceil(math.log2(W))) + 1


@pytest.mark.parametrize("W", range(2, 65))
def test_double_tree_complementarity(oracle_mod, W):
    """Tree 1's leaves are the odd ranks.  Tree 2 is the mirror (even W) or the
    shift by one (odd W); a leaf of one is interior in the other, give or take
    one boundary rank when W is odd."""
    _, _, k1 = oracle_mod.tree(W, 1)
    _, _, k2 = oracle_mod.tree(W, 2)
    leaves1 = {r for r in range(W) if not k1[r]}
    leaves2 = {r for r in range(W) if not k2[r]}
    assert leaves1 == {r for r in range(W) if r % 2 == 1}
    interior_both = {r for r in range(W) if k1[r] and k2[r]}
    if W % 2 == 0:
        assert leaves2 == {r for r in range(W) if r % 2 == 0}
        assert not (leaves1 & leaves2)
        assert not interior_both
    else:
        assert len(interior_both) <= 1
        assert not (leaves1 & leaves2) or W == 1


def _fold_over_tree(op, root, kids, y):
    """Reduce up a tree given as a child table: each node adds its children's
    subtotals, in ascending order, to its own value (numpy fp32)."""
    def sub(v):
        acc = y[v]
        for c in kids[v]:
            acc = acc + sub(c) if op in ("sum", "avg") else acc * sub(c)
        return acc
    return sub(root)


@pytest.mark.parametrize("op", ["sum", "prod"])
def test_tree_reduction_on_diagram(oracle_mod, op):
    """Fold the page's 14-rank tree by hand (tree 1 for the first half of the
    buffer, its mirror image for the second half) and compare bit for bit."""
    W, N = 14, 64
    parent, kids = read_tree("tree14.txt")
    ins = synth.random_values(7, W, N, "fp32")
    got = oracle_mod.allreduce("fp32", op, "tree", ins)
    # mirror image: rank 13 - r takes the place of r
    kids2 = [None] * W
    for r in range(W):
        kids2[W - 1 - r] = [W - 1 - c for c in kids[r]]
    for e in range(N):
        y = [np.float32(ins[r][e]) for r in range(W)]
        if e < N // 2:
            want = _fold_over_tree(op, 0, kids, y)
        else:
            want = _fold_over_tree(op, W - 1, kids2, y)
        assert np.float32(want).tobytes() == got[e:e + 1].tobytes(), e


def test_tree_shift_for_odd_w(oracle_mod):
    """For odd W the second tree is the first shifted by one rank."""
    W = 7
    r1, p1, k1 = oracle_mod.tree(W, 1)
    r2, p2, k2 = oracle_mod.tree(W, 2)
    assert r2 == (r1 + 1) % W
    for r in range(W):
        m = (r + 1) % W
        assert p2[m] == (-1 if p1[r] == -1 else (p1[r] + 1) % W)
        assert k2[m] == [(c + 1) % W for c in k1[r]]


# --------------------------------------------------------------------------
# Order-free ops: every accumulation order gives the same result
# --------------------------------------------------------------------------

def _key(v):
    v = float(v)
    return (v, 1 if math.copysign(1.0, v) > 0 else 0)   # -0 below +0


def _fold_any_order(dtype, op, vals):
    if op == "min":
        return min(vals, key=_key) if dtype != "int32" else min(vals)
    if op == "max":
        return max(vals, key=_key) if dtype != "int32" else max(vals)
    acc = np.int32(vals[0])
    for v in vals[1:]:
        acc = np.int32(acc + np.int32(v)) if op in ("sum", "avg") else np.int32(acc * np.int32(v))
    return acc


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_order_free_ops_brute_force(oracle_mod, W, algo):
    N = 24
    big = [synth.uniform_int(3, W, N, -2**31, 2**31 - 1, "int32")[r] for r in range(W)]
    small = synth.uniform_int(4, W, N, -1000, 1000, "int32")
    for ins in (big, small):
        for op in ("sum", "prod", "min", "max", "avg"):
            got = oracle_mod.allreduce("int32", op, algo, ins)
            for e in range(N):
                vals = [int(ins[r][e]) for r in range(W)]
                results = set()
                with np.errstate(over="ignore"):
                    for perm in itertools.permutations(vals):
                        results.add(int(_fold_any_order("int32", op, list(perm))))
                assert len(results) == 1
                want = results.pop()
                if op == "avg":                      # truncating divide of the wrapped sum
                    want = abs(want) // W if want >= 0 else -(abs(want) // W)
                assert int(got[e]) == want, (op, e, vals)
    # float min/max including signed zeros
    fl = synth.random_values(5, W, N, "fp32", kind="small_int")
    for r in range(W):
        fl[r][::3] = 0.0
        fl[r][1::5] = -0.0
    for op in ("min", "max"):
        got = oracle_mod.allreduce("fp32", op, algo, fl)
        for e in range(N):
            vals = [np.float32(fl[r][e]) for r in range(W)]
            outs = {np.float32(_fold_any_order("fp32", op, list(p))).tobytes()
                    for p in itertools.permutations(vals)}
            assert len(outs) == 1
            assert got[e:e + 1].tobytes() == outs.pop()


def test_signed_zero_rule(oracle_mod):
    a = np.array([-0.0, 0.0], np.float32)
    b = np.array([0.0, -0.0], np.float32)
    for algo in ("ring", "tree"):
        mn = oracle_mod.allreduce("fp32", "min", algo, [a, b])
        mx = oracle_mod.allreduce("fp32", "max", algo, [a, b])
        assert [math.copysign(1, v) for v in mn] == [-1, -1]
        assert [math.copysign(1, v) for v in mx] == [1, 1]


# --------------------------------------------------------------------------
# Integer details: wrapping product, truncating average
# --------------------------------------------------------------------------

def test_int_wrap_and_truncating_avg(oracle_mod):
    a = np.array([65536, 46341, -3, 3, -7, 2**31 - 1], np.int32)
    b = np.array([65536, 46341, 0, 0, 0, 1], np.int32)
    prod = oracle_mod.allreduce("int32", "prod", "ring", [a, b])
    assert prod[0] == 0                                   # 2^32 wraps to 0
    assert prod[1] == 46341 * 46341 - 2**32               # wraps negative
    s = oracle_mod.allreduce("int32", "sum", "ring", [a, b])
    assert s[5] == -2**31                                 # INT_MAX + 1 wraps
    avg = oracle_mod.allreduce("int32", "avg", "tree", [a, b])
    assert avg[2] == -1 and avg[3] == 1 and avg[4] == -3  # truncation toward zero
    assert avg[5] == -2**30                               # divide of the wrapped sum


# --------------------------------------------------------------------------
# Float details: exact sums, pre-scaled average, error bound
# --------------------------------------------------------------------------

def test_exact_integer_valued_floats(oracle_mod):
    """Integer-valued fp32 data in [-8, 8] sums exactly in every order, so ring,
    tree and torch's sum over the stacked ranks agree bit for bit."""
    import torch
    ins = synth.workload_inputs("small_int_fp32_w2")
    W = len(ins)
    ring = oracle_mod.allreduce("fp32", "sum", "ring", ins)
    tree = oracle_mod.allreduce("fp32", "sum", "tree", ins)
    lib = torch.stack([torch.from_numpy(x) for x in ins]).sum(0).numpy()
    assert ring.tobytes() == tree.tobytes() == lib.tobytes()
    avg = oracle_mod.allreduce("fp32", "avg", "ring", ins)
    assert avg.tobytes() == (lib * np.float32(1.0 / W)).astype(np.float32).tobytes()
    # W = 16 integer-valued data, still exact
    ins16 = synth.uniform_int(9, 16, 1000, -8, 8, "fp32")
    lib16 = torch.stack([torch.from_numpy(x) for x in ins16]).sum(0).numpy()
    for algo in ("ring", "tree"):
        assert oracle_mod.allreduce("fp32", "sum", algo, ins16).tobytes() == lib16.tobytes()


def test_avg_is_prescaled(oracle_mod):
    """The float average scales each contribution by 1/n as it is read, so a
    sum that would overflow before a final divide stays finite."""
    a = np.array([3.0e38, -3.0e38], np.float32)
    b = np.array([3.0e38, -3.0e38], np.float32)
    for algo in ("ring", "tree"):
        out = oracle_mod.allreduce("fp32", "avg", algo, [a, b])
        assert out.tolist() == [np.float32(3.0e38), np.float32(-3.0e38)]
    # with W = 3 the scale is fl32(1/3) applied before the sum
    x = [np.array([1.0], np.float32)] * 3
    out = oracle_mod.allreduce("fp32", "avg", "ring", x)
    s = np.float32(1.0 / 3.0)
    assert out[0] == np.float32(np.float32(s + s) + s)


@pytest.mark.parametrize("W", [2, 3, 8, 16, 64])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_float_sum_error_bound(oracle_mod, W, algo):
    """Any order of W-1 rounded adds lies within gamma_{W-1} * sum|y| of the
    exact sum; ring and tree therefore lie within twice that of each other."""
    N = 4096
    ins = synth.normal(11, W, N, 1.0, "fp32")
    got = oracle_mod.allreduce("fp32", "sum", algo, ins).astype(np.float64)
    stack = np.stack([x.astype(np.float64) for x in ins])
    exact = stack.sum(0)
    mag = np.abs(stack).sum(0)
    u = 2.0 ** -24
    gamma = (W - 1) * u / (1 - (W - 1) * u)
    assert np.all(np.abs(got - exact) <= gamma * mag + 1e-45)
    other = oracle_mod.allreduce("fp32", "sum", "tree" if algo == "ring" else "ring", ins).astype(np.float64)
    assert np.all(np.abs(got - other) <= 2 * W * u * mag)


def test_bf16_accumulates_in_fp32(oracle_mod):
    """bf16 inputs are widened exactly, summed in fp32 and rounded once: the
    result equals the fp32 sum of the widened values, rounded to bf16 by torch."""
    import torch
    W, N = 8, 2048
    ins = synth.normal(12, W, N, 1e-2, "bf16")
    got = oracle_mod.allreduce("bf16", "sum", "ring", ins)
    wide = [(x.astype(np.uint32) << 16).view(np.float32) for x in ins]
    # ring order of chunk k: k+1, ..., k; fp32 adds in numpy
    ref = np.empty(N, np.float32)
    for k in range(W):
        lo, hi = k * N // W, (k + 1) * N // W
        acc = wide[(k + 1) % W][lo:hi].copy()
        for i in range(1, W):
            acc = acc + wide[(k + 1 + i) % W][lo:hi]
        ref[lo:hi] = acc
    want = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert got.tobytes() == want.tobytes()


# --------------------------------------------------------------------------
# bf16 rounding against torch's conversion
# --------------------------------------------------------------------------

def test_bf16_rne_against_torch(oracle_mod):
    """Every high half, combined with low halves covering below/at/above the
    halfway point (ties to even decided by the high half), plus a random sample."""
    import torch
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(1)
    pats = np.concatenate([pats, rng.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32)])
    f = pats.view(np.float32)
    pats = pats[~np.isnan(f)]
    got = oracle_mod.bf16_rne(pats)
    want = torch.from_numpy(pats.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    # NaN stays NaN with its sign (payload itself unpinned)
    nan = np.array([0x7FC00000, 0xFF800001, 0x7F800001], np.uint32)
    r = oracle_mod.bf16_rne(nan)
    assert all(((x & 0x7F80) == 0x7F80) and (x & 0x7F) for x in r.tolist())
    assert [x >> 15 for x in r.tolist()] == [0, 1, 0]


# --------------------------------------------------------------------------
# Chunk bounds, compositions, sampled reduction, argument checks
# --------------------------------------------------------------------------

def test_chunk_bounds(oracle_mod):
    for W in (1, 2, 3, 7, 8, 16, 64):
        for N in (0, 1, 5, 63, 64, 1000, 2**40 + 3):
            lo = [oracle_mod.chunk_lo(W, N, k) for k in range(W + 1)]
            assert lo[0] == 0 and lo[W] == N
            assert lo == [(k * N) // W for k in range(W + 1)]
            sizes = [lo[k + 1] - lo[k] for k in range(W)]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int32"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max", "avg"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_rs_then_ag_is_allreduce(oracle_mod, dtype, op, algo):
    W, N = 6, 6 * 37
    ins = synth.random_values(13, W, N, dtype)
    ar = oracle_mod.allreduce(dtype, op, algo, ins)
    shards = oracle_mod.reduce_scatter(dtype, op, algo, ins)
    full = oracle_mod.all_gather(dtype, shards, all_ranks=True)
    for j in range(W):
        assert full[j].tobytes() == ar.tobytes()


@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_reduce_one_matches(oracle_mod, algo):
    W, N = 5, 203
    for dtype in ("fp32", "bf16", "int32"):
        ins = synth.random_values(14, W, N, dtype)
        ar = oracle_mod.allreduce(dtype, "avg", algo, ins)
        for e in (0, 1, 40, 100, 101, 102, 202):
            y = np.array([ins[r][e] for r in range(W)], ins[0].dtype)
            assert oracle_mod.reduce_one(dtype, "avg", algo, N, e, y) == ar[e]


def test_single_rank_is_copy(oracle_mod):
    x = synth.normal(15, 1, 33, 1.0, "fp32")
    for op in ("sum", "prod", "min", "max", "avg"):
        for algo in ("ring", "tree"):
            assert oracle_mod.allreduce("fp32", op, algo, x).tobytes() == x[0].tobytes()


def test_rejects_bad_arguments(oracle_mod):
    x = synth.normal(16, 3, 10, 1.0, "fp32")
    with pytest.raises(ValueError):
        oracle_mod.reduce_scatter("fp32", "sum", "ring", x)   # 10 % 3 != 0
    lib = oracle_mod.lib()
    assert lib.or_allreduce(0, 0, 0, 0, 4, None, None) == -1
    assert lib.or_allreduce(0, 0, 0, 65, 4, None, None) == -1
    assert lib.or_allreduce(3, 0, 0, 2, 4, None, None) == -1
    assert lib.or_allreduce(0, 5, 0, 2, 4, None, None) == -1
    assert lib.or_allreduce(0, 0, 2, 2, 4, None, None) == -1


def _host_reduce_one(oracle_mod, dtype, op, algo, W, N, e, y):
    """Element e of an N-element all-reduce recomputed plainly on the host:
    the chunk from floor(k*N/W) in Python integers, the ring order k+1, ...,
    k or the oracle's tree (tree 1 below floor(N/2), tree 2 from there), and
    the fold in numpy fp32 or wrapping 32-bit integers."""
    k = max(j for j in range(W) if (j * N) // W <= e)
    if dtype == "int32":
        vals = [int(v) & 0xFFFFFFFF for v in y]
        comb = {"sum": lambda a, b: (a + b) & 0xFFFFFFFF, "avg": lambda a, b: (a + b) & 0xFFFFFFFF,
                "max": lambda a, b: b if _s32(b) > _s32(a) else a}[op]
    else:
        vals = [np.float32(v) for v in y]
        if op == "avg":
            vals = [np.float32(v * np.float32(1.0 / W)) for v in vals]
        comb = {"sum": lambda a, b: np.float32(a + b), "avg": lambda a, b: np.float32(a + b)}[op]
    if algo == "ring":
        order = [(k + 1 + i) % W for i in range(W)]
        acc = vals[order[0]]
        for r in order[1:]:
            acc = comb(acc, vals[r])
    else:
        root, _, kids = oracle_mod.tree(W, 1 if e < N // 2 else 2)

        def sub(v):
            a = vals[v]
            for c in kids[v]:
                a = comb(a, sub(c))
            return a
        acc = sub(root)
    if dtype == "int32":
        acc = _s32(acc)
        if op == "avg":
            acc = int(acc / W)          # one truncating divide of the wrapped sum
        return np.int32(acc)
    return np.float32(acc)


def _s32(u):
    return u - (1 << 32) if u & 0x80000000 else u


@pytest.mark.parametrize("N", [2**31 + 9, 2**40 + 3, 2**62 + 5])
@pytest.mark.parametrize("W", [2, 4, 7])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_reduce_one_at_large_n(oracle_mod, N, W, algo):
    """or_reduce_one (the oracle's one-position reduction behind the GPU's
    checks past 2^31 elements) at positions on both sides of every chunk
    bound and of the tree split, for N far beyond what can be allocated."""
    rng = np.random.default_rng(N % 1000 + W)
    es = {0, N - 1, N // 2 - 1, N // 2, N // 2 + 1}
    for kk in range(1, W):
        lo = (kk * N) // W
        es |= {lo - 1, lo, lo + 1}
    es |= {int(x) for x in rng.integers(0, N, size=5, dtype=np.uint64)}
    for e in sorted(es):
        yf = rng.standard_normal(W).astype(np.float32)
        yi = rng.integers(-2**31, 2**31, size=W, dtype=np.int64).astype(np.int32)
        for dtype, op, y in (("fp32", "sum", yf), ("fp32", "avg", yf), ("int32", "sum", yi), ("int32", "max", yi),
                             ("int32", "avg", yi)):
            got = oracle_mod.reduce_one(dtype, op, algo, N, e, y)
            want = _host_reduce_one(oracle_mod, dtype, op, algo, W, N, e, y)
            assert np.array(got).tobytes() == np.array(want).tobytes(), (dtype, op, e)
