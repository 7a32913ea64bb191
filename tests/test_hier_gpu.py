"""GPU parity of the hierarchical order and of per-hop bf16 rounding, through
mr_allreduce_ex / mr_reduce_scatter_ex, bit for bit against the oracle."""
import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_same, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import collective_reduction_math_gb300 as m
    m.load()
    return m


def _data(seed, W, N, dtype, op):
    return synth.random_values(seed, W, N, dtype, kind="near_one" if op == "prod" else "normal")


def check(mr, dtype, op, algo, group, hop, W, N):
    import oracle
    import torch
    host = _data(700 + W + (group or 0), W, N, dtype, op)
    xs = [to_device(h, dtype) for h in host]
    g = Guarded(W, N, dtype)
    mr.mr_allreduce_ex(xs, g.views, op=op, algo=algo, group=group, per_hop=hop)
    torch.cuda.synchronize()
    g.check()
    want = oracle.allreduce_ex(dtype, op, algo, host, group=group or 0, hop=hop)
    for j, o in enumerate(g.host()):
        assert_same(o, want, f"allreduce_ex {dtype} {op} {algo} g={group} hop={hop} W={W} N={N} rank {j}")
    if N % W == 0:
        sh = Guarded(W, N // W, dtype)
        mr.mr_reduce_scatter_ex(xs, sh.views, op=op, algo=algo, group=group, per_hop=hop)
        torch.cuda.synchronize()
        sh.check()
        want_rs = oracle.reduce_scatter_ex(dtype, op, algo, host, group=group or 0, hop=hop)
        for k, o in enumerate(sh.host()):
            assert_same(o, want_rs[k], f"reduce_scatter_ex {dtype} {op} {algo} g={group} hop={hop} shard {k}")


@pytest.mark.parametrize("W,group", [(2, 1), (4, 2), (6, 3), (8, 2), (8, 4), (10, 5), (12, 4), (16, 4), (16, 8), (24, 6),
                                     (64, 8)])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int32"])
def test_hier_parity(mr, W, group, dtype):
    for N in (W * 1024 * 2 + W * 3, 5 * W + 3):
        for op in ("sum", "prod", "max", "avg"):
            check(mr, dtype, op, "hier", group, False, W, N)


@pytest.mark.parametrize("algo,group", [("ring", None), ("tree", None), ("hier", 4)])
@pytest.mark.parametrize("W", [2, 8, 10, 12, 16, 40])
def test_per_hop_bf16_parity(mr, algo, group, W):
    if algo == "hier" and W % 4:
        group = 2
    for N in (W * 4096 + 24, 7 * W):
        for op in ("sum", "avg", "min"):
            check(mr, "bf16", op, algo, group, True, W, N)


@pytest.mark.parametrize("algo,group", [("ring", None), ("tree", None), ("hier", 4)])
@pytest.mark.parametrize("W", [3, 8, 16, 40])
def test_per_hop_bf16_wide_values(mr, algo, group, W):
    """Per-hop bf16 sum and avg on values spread over the whole exponent range,
    subnormals included: every hop's rounding decides the result, so a kernel
    that rounded differently from the oracle's fp32-add-then-round would
    differ somewhere in these buffers."""
    import oracle
    import torch
    if algo == "hier" and W % 4:
        group = 3 if W % 3 == 0 else 2
    for N in (W * 8192 + 40, 9 * W):
        host = synth.bf16_wide(740 + W, W, N)
        xs = [to_device(h, "bf16") for h in host]
        for op in ("sum", "avg"):
            g = Guarded(W, N, "bf16")
            mr.mr_allreduce_ex(xs, g.views, op=op, algo=algo, group=group, per_hop=True)
            torch.cuda.synchronize()
            g.check()
            want = oracle.allreduce_ex("bf16", op, algo, host, group=group or 0, hop=True)
            for j, o in enumerate(g.host()):
                assert_same(o, want, f"per-hop wide {op} {algo} W={W} N={N} rank {j}")
            if N % W == 0:
                sh = Guarded(W, N // W, "bf16")
                mr.mr_reduce_scatter_ex(xs, sh.views, op=op, algo=algo, group=group, per_hop=True)
                torch.cuda.synchronize()
                sh.check()
                want_rs = oracle.reduce_scatter_ex("bf16", op, algo, host, group=group or 0, hop=True)
                for k, o in enumerate(sh.host()):
                    assert_same(o, want_rs[k], f"per-hop wide rs {op} {algo} W={W} shard {k}")


def test_ex_defaults_match_plain(mr):
    """ring / tree through the _ex entry points are the plain calls."""
    import torch
    W, N = 8, 8 * 5000
    host = synth.random_values(710, W, N, "fp32")
    xs = [to_device(h, "fp32") for h in host]
    for algo in ("ring", "tree"):
        a = [torch.empty_like(x) for x in xs]
        b = [torch.empty_like(x) for x in xs]
        mr.mr_allreduce(xs, a, op="sum", algo=algo)
        mr.mr_allreduce_ex(xs, b, op="sum", algo=algo)
        torch.cuda.synchronize()
        assert all(torch.equal(p, q) for p, q in zip(a, b))


def test_hier_errors(mr):
    import torch
    xs = [torch.zeros(64, device="cuda") for _ in range(6)]
    ys = [torch.zeros(64, device="cuda") for _ in range(6)]
    with pytest.raises(mr.MRError) as e:
        mr.mr_allreduce_ex(xs, ys, algo="hier", group=4)       # 4 does not divide 6
    assert e.value.status == 1
    with pytest.raises(mr.MRError) as e:
        mr.mr_allreduce(xs, ys, algo="hier")                   # the plain call has no group
    assert e.value.status == 1


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int32"])
def test_auto_equals_the_planned_order(mr, dtype):
    """MR_AUTO gives exactly the result of the order mr_plan_auto names."""
    import oracle
    import torch
    for W, N in ((2, 4096), (8, 1 << 16), (16, 1 << 14), (33, 3000), (8, 1 << 22)):
        host = synth.random_values(720 + W, W, N, dtype)
        xs = [to_device(h, dtype) for h in host]
        planned, _ = mr.mr_plan_auto(W, N, dtype)
        ys = [torch.empty_like(x) for x in xs]
        mr.mr_allreduce(xs, ys, op="avg", algo="auto")
        torch.cuda.synchronize()
        want = oracle.allreduce(dtype, "avg", planned, host)
        for j, y in enumerate(ys):
            assert_same(y.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else y.cpu().numpy(),
                        want, f"auto ({planned}) {dtype} W={W} N={N} rank {j}")
        if N % W == 0:
            planned_rs, _ = mr.mr_plan_auto(W, N, dtype, reduce_scatter=True)
            sh = [torch.empty(N // W, dtype=xs[0].dtype, device="cuda") for _ in range(W)]
            mr.mr_reduce_scatter(xs, sh, op="sum", algo="auto")
            torch.cuda.synchronize()
            want_rs = oracle.reduce_scatter(dtype, "sum", planned_rs, host)
            for k, t in enumerate(sh):
                got = t.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else t.cpu().numpy()
                assert_same(got, want_rs[k], f"auto rs ({planned_rs}) {dtype} W={W} shard {k}")
