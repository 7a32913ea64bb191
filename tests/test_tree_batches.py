"""The tree order folded in batches of 8 positions gives exactly the oracle's
tree fold.

From 13 ranks up the CUDA kernel does not hold all W contributions of an
element at once.  It loads the positions in batches [8m, 8m+8), folds each
batch up to the node that the batch head's upper-child search finds inside it,
and then folds the batch heads 8m as the same bit-trick tree one level up.
The int32 trees over 16 slots run a second schedule when W is not a
multiple of 8: the positions past W padded with the op's exact identity and
the whole tree folded with no condition on W.  This test restates both schedules on symbols and checks,
for every W from 9 to 64, that they perform the oracle's combines in the
oracle's order (the padded one once its identities drop): each node's
own value first, then its children's subtotals in the order the oracle lists
them (double binary tree, "The double binary tree", post on NCCL all-reduce).
Positions, not ranks, are folded, so one check covers both trees.
"""
import pytest


def oracle_fold(W, oracle_mod):
    """The symbolic fold of tree 1 over positions, from the oracle's tree."""
    root, _parent, kids = oracle_mod.tree(W, 1)

    def sub(v):
        e = f"y{v}"
        for c in kids[v]:
            e = f"({e}+{sub(c)})"
        return e
    return sub(root)


def batch_top(yb, Wb):
    """Levels 2 and 4 inside one batch (yb[0] is the head), then the subtotal
    of the largest h in {4, 2, 1} with h < Wb."""
    y = list(yb)
    b = 2
    while b < 8:
        for p in range(b, 8, 2 * b):
            if p < Wb:
                a = f"({y[p]}+{y[p - b // 2]})"
                h = b // 2
                while h >= 1:
                    if p + h < Wb:
                        a = f"({a}+{y[p + h]})"
                        break
                    h //= 2
                y[p] = a
        b *= 2
    for h in (4, 2, 1):
        if h < Wb:
            return y[h]
    return None


def batched_fold(W, slots, swap_children=False):
    """The kernel's schedule with `slots` register slots (16, 32 or 64).
    swap_children plants a mistake: a head adds its upper child first."""
    y = [f"y{i}" for i in range(W)] + [None] * (slots + 8 - W)
    NB, M = slots // 8, (W + 7) // 8
    head, top = [None] * NB, [None] * NB
    for m in range(min(NB, M)):
        Wb = min(8, W - 8 * m)
        head[m] = y[8 * m]
        top[m] = batch_top(y[8 * m:8 * m + 8], Wb)
    B = 1
    while B < NB:
        for m in range(B, NB, 2 * B):
            if m < M:
                lower = top[m - 1] if B == 1 else head[m - B // 2]
                upper = None
                h = B // 2
                while h >= 1:
                    if m + h < M:
                        upper = head[m + h]
                        break
                    h //= 2
                if upper is None and 8 * m + 1 < W:
                    upper = top[m]
                first, second = (upper, lower) if swap_children and upper is not None else (lower, upper)
                a = f"({head[m]}+{first})"
                if second is not None:
                    a = f"({a}+{second})"
                head[m] = a
        B *= 2
    a, h = head[0], NB // 2
    while h >= 1:
        if h < M:
            return f"({a}+{head[h]})"
        h //= 2
    return a


def cmb(a, b):
    """One combine, written out; the identity e drops (a + e = e + a = a)."""
    if a == "e":
        return b
    if b == "e":
        return a
    return f"({a}+{b})"


def padded_fold(W, slots, swap_children=False):
    """The kernel's schedule: positions past W padded with the identity e and
    the whole bit-trick tree over slots // 8 batches of 8 folded with no
    condition on W (in-batch nodes 2, 6, 4; head m's lower child the previous
    batch's node 4 or head m - B/2, its upper child its own batch's node 4 or
    head m + B/2; the root's child head NB/2).  swap_children plants a
    mistake: a head adds its upper child first."""
    NB = slots // 8
    y = [f"y{i}" if i < W else "e" for i in range(slots)]
    head, top = [None] * NB, [None] * NB
    for m in range(NB):
        b = y[8 * m:8 * m + 8]
        n2 = cmb(cmb(b[2], b[1]), b[3])
        n6 = cmb(cmb(b[6], b[5]), b[7])
        top[m] = cmb(cmb(b[4], n2), n6)
        head[m] = b[0]
    B = 1
    while B < NB:
        for m in range(B, NB, 2 * B):
            lower = top[m - 1] if B == 1 else head[m - B // 2]
            upper = top[m] if B == 1 else head[m + B // 2]
            first, second = (upper, lower) if swap_children else (lower, upper)
            head[m] = cmb(cmb(head[m], first), second)
        B *= 2
    return cmb(head[0], head[NB // 2])


def kernel_slots(W):
    """The slots of the kernel the host runs for the tree: 16 up to 16 ranks,
    32 (4 batch heads) up to 32, else 64 (8 heads)."""
    return 16 if W <= 16 else 32 if W <= 32 else 64


@pytest.mark.parametrize("W", range(9, 65))
def test_batched_tree_is_the_oracle_tree(oracle_mod, W):
    assert batched_fold(W, kernel_slots(W)) == oracle_fold(W, oracle_mod)


@pytest.mark.parametrize("W", range(17, 33))
def test_the_64_slot_tree_also_folds_17_to_32_ranks(oracle_mod, W):
    """The 64-slot schedule over at most 4 batches is the 32-slot one."""
    assert batched_fold(W, 64) == batched_fold(W, 32) == oracle_fold(W, oracle_mod)


@pytest.mark.parametrize("W", [12, 24, 64])
def test_a_planted_mistake_is_caught(oracle_mod, W):
    """A head that adds its upper child before its lower one is caught."""
    slots = kernel_slots(W)
    assert batched_fold(W, slots) == oracle_fold(W, oracle_mod)
    assert batched_fold(W, slots, swap_children=True) != oracle_fold(W, oracle_mod)


@pytest.mark.parametrize("W", range(9, 65))
def test_padded_tree_is_the_oracle_tree(oracle_mod, W):
    """The identity-padded schedule the kernel runs gives the oracle's tree
    fold once the identities drop, at the host's slot count and at 64."""
    want = oracle_fold(W, oracle_mod)
    assert padded_fold(W, kernel_slots(W)) == want
    assert padded_fold(W, 64) == want


@pytest.mark.parametrize("W", [10, 12, 24, 40, 64])
def test_a_planted_mistake_in_the_padded_tree_is_caught(oracle_mod, W):
    assert padded_fold(W, kernel_slots(W), swap_children=True) != oracle_fold(W, oracle_mod)
