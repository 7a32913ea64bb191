"""Pins of the oracle's hierarchical order and per-hop bf16 rounding.

The hierarchical all-reduce ("Communication Optimization ...", the five-step
topology-aware all-reduce) is checked against a literal two-level pipeline:
the ring schedule simulator run inside every group, then across the groups on
every chunk.  Per-hop bf16 rounding is checked against the same simulator
with the partials rounded as they cross each hop, and against torch's own
bf16 addition."""
import numpy as np
import pytest

import synth
from ring_sim import simulate

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _widen(dtype, a):
    return (a.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else a


def hier_sim(dtype, op, inputs, g, hop=False):
    """Ring reduce-scatter + all-gather inside each group of g ranks, then a
    ring all-reduce across the groups on every g-chunk, literally."""
    W, N = len(inputs), inputs[0].size
    G = W // g
    y = [_widen(dtype, a) for a in inputs]
    if op == "avg" and dtype != "int32":
        s = np.float32(1.0 / W)
        y = [(v * s).astype(np.float32) for v in y]
        if hop and dtype == "bf16":
            import ring_sim
            y = [ring_sim._to_bf16_and_back(v) for v in y]
    inner_op = "sum" if op == "avg" else op
    dt = "fp32" if dtype == "bf16" else dtype
    group_total = [simulate(dt, inner_op, y[a * g:(a + 1) * g], raw=True)[0][0] if not hop else
                   simulate_hop(inner_op, y[a * g:(a + 1) * g]) for a in range(G)]
    out = np.empty(N, np.float32 if dtype != "int32" else np.int32)
    for c in range(g):
        lo, hi = (c * N) // g, ((c + 1) * N) // g
        parts = [gt[lo:hi].copy() for gt in group_total]
        out[lo:hi] = (simulate(dt, inner_op, parts, raw=True)[0][0] if not hop else simulate_hop(inner_op, parts))
    return out


def simulate_hop(op, y):
    # bf16 per-hop simulation on already-widened fp32 values
    return simulate("bf16", op, y, hop=True, raw=True)[0][0]


def _post(dtype, op, W, acc):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "int32" and op == "avg":
        wide = acc.astype(np.int64)
        q = np.abs(wide) // W
        return np.where(wide < 0, -q, q).astype(np.int32)
    return acc


@pytest.mark.parametrize("dtype,op", [("fp32", "sum"), ("fp32", "avg"), ("fp32", "prod"), ("bf16", "sum"),
                                       ("bf16", "avg"), ("int32", "sum"), ("int32", "avg")])
@pytest.mark.parametrize("W,g", [(4, 2), (6, 3), (6, 2), (8, 4), (8, 2), (9, 3), (12, 4)])
@pytest.mark.parametrize("N", [60, 97])
def test_hier_matches_two_level_pipeline(oracle_mod, dtype, op, W, g, N):
    ins = synth.random_values(200 + W + g, W, N, dtype, kind="near_one" if op == "prod" else "normal")
    want = _post(dtype, op, W, hier_sim(dtype, op, ins, g))
    got = oracle_mod.allreduce_ex(dtype, op, "hier", ins, group=g)
    assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("W", [1, 2, 5, 8])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int32"])
def test_hier_degenerates_to_ring(oracle_mod, W, dtype):
    """One group of W, or W groups of one: the hierarchy is the plain ring."""
    ins = synth.random_values(300 + W, W, 4 * W + 3, dtype)
    ring = oracle_mod.allreduce(dtype, "avg", "ring", ins)
    for g in (1, W):
        assert oracle_mod.allreduce_ex(dtype, "avg", "hier", ins, group=g).tobytes() == ring.tobytes()


def test_hier_integer_ops_are_order_free(oracle_mod):
    ins = synth.random_values(301, 8, 1000, "int32")
    for op in ("sum", "prod", "min", "max", "avg"):
        ring = oracle_mod.allreduce("int32", op, "ring", ins)
        assert oracle_mod.allreduce_ex("int32", op, "hier", ins, group=4).tobytes() == ring.tobytes()


@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("W", [2, 3, 5, 8])
def test_per_hop_bf16_ring_matches_simulation(oracle_mod, op, W):
    ins = synth.random_values(400 + W, W, 101, "bf16")
    y = [_widen("bf16", a) for a in ins]
    if op == "avg":
        import ring_sim
        y = [ring_sim._to_bf16_and_back((v * np.float32(1.0 / W)).astype(np.float32)) for v in y]
    want = _post("bf16", "sum", W, simulate_hop("sum", y))
    got = oracle_mod.allreduce_ex("bf16", op, "ring", ins, hop=True)
    assert got.tobytes() == want.tobytes()
    # per-hop rounding of a hierarchical order, too
    if W % 2 == 0 and W > 2:
        want_h = _post("bf16", op, W, hier_sim("bf16", op, ins, 2, hop=True))
        assert oracle_mod.allreduce_ex("bf16", op, "hier", ins, group=2, hop=True).tobytes() == want_h.tobytes()


def test_per_hop_two_ranks_is_torch_bf16_add(oracle_mod):
    """With two ranks a ring hop is one bf16 addition: torch's bf16 + bf16."""
    import torch
    a, b = synth.random_values(402, 2, 5000, "bf16")
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    want = (tb + ta).view(torch.int16).numpy().view(np.uint16)       # chunk 0: rank 1 then rank 0
    got = oracle_mod.allreduce_ex("bf16", "sum", "ring", [a, b], hop=True)
    assert np.array_equal(got, want)
    # and without per-hop rounding the fp32 sum rounds once: the same for two terms
    assert np.array_equal(oracle_mod.allreduce("bf16", "sum", "ring", [a, b]), want)


def test_per_hop_changes_bf16_results(oracle_mod):
    """Rounding every hop differs from accumulating in fp32 (the reason the
    FSDP page gives for reducing in fp32), and is no-op for fp32 and int32."""
    ins = synth.random_values(403, 8, 4096, "bf16")
    a = oracle_mod.allreduce_ex("bf16", "sum", "ring", ins, hop=True)
    b = oracle_mod.allreduce("bf16", "sum", "ring", ins)
    assert not np.array_equal(a, b)
    f = synth.random_values(404, 8, 999, "fp32")
    assert oracle_mod.allreduce_ex("fp32", "sum", "ring", f, hop=True).tobytes() == \
        oracle_mod.allreduce("fp32", "sum", "ring", f).tobytes()


def test_rs_ex_is_allreduce_ex_chunks(oracle_mod):
    ins = synth.random_values(405, 8, 8 * 77, "bf16")
    ar = oracle_mod.allreduce_ex("bf16", "avg", "hier", ins, group=4, hop=True)
    rs = oracle_mod.reduce_scatter_ex("bf16", "avg", "hier", ins, group=4, hop=True)
    assert np.concatenate(rs).tobytes() == ar.tobytes()
