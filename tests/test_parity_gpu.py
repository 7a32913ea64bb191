"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle,
element by element.  Bit-exact everywhere: the kernels follow the same
accumulation order with the same IEEE fp32 operations (no FMA), integer work
is exact, and bf16 is rounded once from the same fp32 value.

Every output buffer sits between canary guard bands that must survive.
"""
import numpy as np
import pytest

import synth
from golden_io import read_blocks
from gpu_util import Guarded, assert_same, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

OPS = ["sum", "prod", "min", "max", "avg"]
ALGOS = ["ring", "tree"]
DTYPES = ["fp32", "bf16", "int32"]


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
    kind = "near_one" if op == "prod" else "normal"
    vals = synth.random_values(seed, W, N, dtype, kind=kind)
    if op in ("min", "max") and dtype != "int32" and N > 4:
        for r in range(W):        # signed zeros must follow -0 < +0
            neg = r % 2 == 1
            if dtype == "bf16":
                vals[r][3::7] = 0x8000 if neg else 0
            else:
                vals[r][3::7] = -0.0 if neg else 0.0
    return vals


def _allreduce_check(mr, host, dtype, op, algo, offset=0, inplace=False):
    import torch
    W, N = len(host), host[0].size
    xs = [to_device(h, dtype) for h in host]
    if inplace:
        mr.mr_allreduce(xs, xs, op=op, algo=algo)
        torch.cuda.synchronize()
        outs = [to_host(x, dtype) for x in xs]
    else:
        g = Guarded(W, N, dtype, offset=offset)
        src = xs
        if offset:
            src = []
            for x in xs:     # element-aligned but not 16-byte aligned inputs
                buf = torch.empty(N + offset, dtype=x.dtype, device=x.device)
                buf[offset:].copy_(x)
                src.append(buf[offset:])
        mr.mr_allreduce(src, g.views, op=op, algo=algo)
        torch.cuda.synchronize()
        g.check()
        outs = g.host()
    want = oracle_allreduce(dtype, op, algo, host)
    for j, o in enumerate(outs):
        assert_same(o, want, f"allreduce {dtype} {op} {algo} W={W} N={N} rank {j}")


def oracle_allreduce(dtype, op, algo, host):
    import oracle
    return oracle.allreduce(dtype, op, algo, host)


# --------------------------------------------------------------------------
# the worked examples
# --------------------------------------------------------------------------

def test_worked_examples_on_gpu(mr):
    import torch
    for algo in ALGOS:
        for b in read_blocks("worked_examples.txt"):
            ins = [np.array([float(v) for v in b[k].split()], np.float32) for k in ("rank0", "rank1")]
            exp = [np.array([float(v) for v in b[k].split()], np.float32) for k in ("expect0", "expect1")]
            xs = [to_device(x, "fp32") for x in ins]
            outs = [torch.empty(len(e), dtype=torch.float32, device="cuda") for e in exp]
            if b["collective"] == "allreduce":
                mr.mr_allreduce(xs, outs, op=b["op"], algo=algo)
            elif b["collective"] == "reduce_scatter":
                mr.mr_reduce_scatter(xs, outs, op=b["op"], algo=algo)
            else:
                mr.mr_all_gather(xs, outs)
            torch.cuda.synchronize()
            for o, e in zip(outs, exp):
                assert_same(o.cpu().numpy(), e, b["case"])


# --------------------------------------------------------------------------
# small and ragged sizes: every dtype, op, algorithm and several W
# --------------------------------------------------------------------------

def _sizes(W):
    lanes = 4
    per = 256 * lanes * (3 if W <= 16 else 1)
    return [1, 7, W * per + 13, W * per * 2]


# W = 9 to 11 run the batched fold with 16 slots for every order, W = 12 the
# plain 16-slot fold for the ring and the batched one for the tree, 13 and 16
# the batched fold, 17 and up the batched fold with 64 slots, except the tree
# up to 32 ranks (32 slots: 4 batch heads)
CASES = [(W, N) for W in (1, 2, 3, 5, 8, 9, 11, 12, 13, 16, 17, 20, 32, 33, 64) for N in _sizes(W)]


@pytest.mark.parametrize("W,N", CASES)
@pytest.mark.parametrize("dtype", DTYPES)
def test_allreduce_parity(mr, W, N, dtype):
    for op in OPS:
        host = _data(1000 + W, W, N, dtype, op)
        for algo in ALGOS:
            _allreduce_check(mr, host, dtype, op, algo)


@pytest.mark.parametrize("W,C", [(1, 4096), (2, 3), (3, 1000), (8, 5), (8, 4096 + 4), (13, 777), (16, 2048),
                                 (17, 100), (64, 64)])
@pytest.mark.parametrize("dtype", DTYPES)
def test_reduce_scatter_and_all_gather_parity(mr, W, C, dtype):
    import oracle
    import torch
    N = W * C
    for op in OPS:
        host = _data(2000 + W, W, N, dtype, op)
        xs = [to_device(h, dtype) for h in host]
        for algo in ALGOS:
            g = Guarded(W, C, dtype)
            mr.mr_reduce_scatter(xs, g.views, op=op, algo=algo)
            torch.cuda.synchronize()
            g.check()
            want = oracle.reduce_scatter(dtype, op, algo, host)
            for k, s in enumerate(g.host()):
                assert_same(s, want[k], f"reduce_scatter {dtype} {op} {algo} W={W} C={C} shard {k}")
            # all-gather of the shards rebuilds the all-reduce, bit for bit
            full = Guarded(W, N, dtype)
            mr.mr_all_gather(g.views, full.views)
            torch.cuda.synchronize()
            full.check()
            ar = oracle.allreduce(dtype, op, algo, host)
            for j, f in enumerate(full.host()):
                assert_same(f, ar, f"reduce_scatter+all_gather {dtype} {op} {algo} W={W} rank {j}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_all_gather_parity(mr, dtype):
    import oracle
    import torch
    for W, C in ((1, 10), (2, 2), (4, 4097), (8, 1 << 16), (16, 3), (64, 100)):
        shards = synth.random_values(3000 + W, W, C, dtype)
        g = Guarded(W, W * C, dtype)
        mr.mr_all_gather([to_device(s, dtype) for s in shards], g.views)
        torch.cuda.synchronize()
        g.check()
        want = oracle.all_gather(dtype, shards)
        for j, o in enumerate(g.host()):
            assert_same(o, want, f"all_gather {dtype} W={W} C={C} rank {j}")


# --------------------------------------------------------------------------
# in place, misaligned pointers, streams, launches
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(mr, dtype):
    import oracle
    import torch
    W, C = 8, 4096 + 12
    N = W * C
    for algo in ALGOS:
        host = _data(4000, W, N, dtype, "avg")
        _allreduce_check(mr, host, dtype, "avg", algo, inplace=True)
        # reduce-scatter in place: recv[r] is slice r of send[r]
        xs = [to_device(h, dtype) for h in host]
        mr.mr_reduce_scatter(xs, [x[r * C:(r + 1) * C] for r, x in enumerate(xs)], op="sum", algo=algo)
        torch.cuda.synchronize()
        want = oracle.reduce_scatter(dtype, "sum", algo, host)
        for r, x in enumerate(xs):
            assert_same(to_host(x[r * C:(r + 1) * C], dtype), want[r], f"in-place reduce_scatter rank {r}")
        # all-gather in place: send[r] is slice r of recv[r]
        mr.mr_all_gather([x[r * C:(r + 1) * C] for r, x in enumerate(xs)], xs)
        torch.cuda.synchronize()
        cat = np.concatenate(want)
        for r, x in enumerate(xs):
            assert_same(to_host(x, dtype), cat, f"in-place all_gather rank {r}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers(mr, dtype, offset):
    for W in (3, 8, 16, 20, 40):
        N = W * 1024 + 5
        for op in ("sum", "avg", "max"):
            host = _data(5000 + offset, W, N, dtype, op)
            for algo in ALGOS:
                _allreduce_check(mr, host, dtype, op, algo, offset=offset)


def test_side_stream_and_launch_count(mr):
    import oracle
    import torch
    W, N = 8, 1 << 16
    host = synth.normal(6000, W, N, 1.0, "fp32")
    xs = [to_device(h, "fp32") for h in host]
    ys = [torch.empty_like(x) for x in xs]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    before = mr.mr_launch_count()
    with torch.cuda.stream(s):
        mr.mr_allreduce(xs, ys, op="sum", algo="ring")
    assert mr.mr_launch_count() == before + 1
    s.synchronize()
    want = oracle.allreduce("fp32", "sum", "ring", host)
    for y in ys:
        assert_same(y.cpu().numpy(), want, "side stream")


def test_launch_floor_runs_between_calls(mr):
    """The empty kernel launches (1 CTA and a full grid), counts as a launch,
    and leaves the calls queued around it on the stream exact."""
    import oracle
    import torch
    W, N = 4, 4096 + 3
    host = synth.normal(6001, W, N, 1.0, "fp32")
    xs = [to_device(h, "fp32") for h in host]
    ys = [torch.empty_like(x) for x in xs]
    before = mr.mr_launch_count()
    mr.mr_launch_floor(1)
    mr.mr_allreduce(xs, ys, op="sum", algo="tree")
    mr.mr_launch_floor(3 * torch.cuda.get_device_properties(0).multi_processor_count)
    torch.cuda.synchronize()
    assert mr.mr_launch_count() == before + 3
    want = oracle.allreduce("fp32", "sum", "tree", host)
    for y in ys:
        assert_same(y.cpu().numpy(), want, "around the empty kernel")


def test_denormals_and_signed_zero(mr):
    """Subnormal inputs add exactly (no flush to zero) on both sides."""
    W, N = 4, 4096
    host = [(np.arange(N, dtype=np.float32) * np.float32(1e-42) * (r + 1)).astype(np.float32) for r in range(W)]
    host[1][::2] *= -1
    for op in ("sum", "avg", "min", "max"):
        for algo in ALGOS:
            _allreduce_check(mr, host, "fp32", op, algo)


def test_gpu_errors_are_reported(mr):
    import torch
    xs = [torch.zeros(16, device="cuda") for _ in range(3)]
    with pytest.raises(mr.MRError) as e:
        mr.mr_reduce_scatter(xs, [torch.zeros(5, device="cuda") for _ in range(3)])
    assert e.value.status == 1
    with pytest.raises(mr.MRError) as e:
        mr.mr_allreduce(xs, [xs[0], xs[0], xs[0]])
    assert e.value.status == 3


# --------------------------------------------------------------------------
# the workloads at full size, in the launch configuration the benchmark times
# --------------------------------------------------------------------------

def test_small_int_fp32_w2_full(mr):
    import oracle
    import torch
    host = synth.workload_inputs("small_int_fp32_w2")
    for op in ("sum", "avg"):
        _allreduce_check(mr, host, "fp32", op, "ring")
    xs = [to_device(h, "fp32") for h in host]
    shards = [torch.empty(2048, device="cuda") for _ in range(2)]
    mr.mr_reduce_scatter(xs, shards, op="avg", algo="ring")
    full = [torch.empty(4096, device="cuda") for _ in range(2)]
    mr.mr_all_gather(shards, full)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter("fp32", "avg", "ring", host)
    for k in range(2):
        assert_same(shards[k].cpu().numpy(), want[k], "rs")
        assert_same(full[k].cpu().numpy(), np.concatenate(want), "ag")


def test_ddp_bucket_fp32_w8_full(mr):
    """W=8, 2^24 fp32 per rank, ring all-reduce avg: every element of every
    rank's output against the oracle."""
    host = synth.workload_inputs("ddp_bucket_fp32_w8")
    _allreduce_check(mr, host, "fp32", "avg", "ring")


def test_fsdp_bf16_w8_full(mr):
    """W=8, 2^26 bf16 per rank: reduce-scatter avg (fp32 accumulate, bf16
    shards), then all-gather of the bf16 parameter shards."""
    import oracle
    import torch
    name = "fsdp_bf16_w8"
    host = synth.workload_inputs(name)
    W, N = len(host), host[0].size
    C = N // W
    xs = [to_device(h, "bf16") for h in host]
    shards = Guarded(W, C, "bf16")
    mr.mr_reduce_scatter(xs, shards.views, op="avg", algo="ring")
    torch.cuda.synchronize()
    shards.check()
    want = oracle.reduce_scatter("bf16", "avg", "ring", host)
    for k, s in enumerate(shards.host()):
        assert_same(s, want[k], f"fsdp reduce_scatter shard {k}")
    del xs
    params = synth.workload_param_shards(name)
    full = Guarded(W, N, "bf16")
    mr.mr_all_gather([to_device(p, "bf16") for p in params], full.views)
    torch.cuda.synchronize()
    full.check()
    cat = np.concatenate(params)
    for j, f in enumerate(full.host()):
        assert_same(f, cat, f"fsdp all_gather rank {j}")


def test_int_counts_w16_full(mr):
    """W=16, 2^22 int32 per rank: sum, min, max, prod (wrapping), avg
    (truncating divide), ring and tree, bit-exact; ring == tree."""
    import torch
    host = synth.workload_inputs("int_counts_w16")
    xs = [to_device(h, "int32") for h in host]
    for op in OPS:
        import oracle
        want = oracle.allreduce("int32", op, "ring", host)
        for algo in ALGOS:
            ys = [torch.empty_like(x) for x in xs]
            mr.mr_allreduce(xs, ys, op=op, algo=algo)
            torch.cuda.synchronize()
            for j, y in enumerate(ys):
                assert_same(y.cpu().numpy(), want, f"int32 {op} {algo} rank {j}")


@pytest.mark.parametrize("W,dtype,algo,N", [(19, "fp32", "ring", (1 << 19) + 5), (24, "bf16", "tree", (1 << 20) + 5),
                                             (57, "int32", "ring", (1 << 19) + 5)])
def test_grid_not_a_multiple_of_the_segments(mr, W, dtype, algo, N):
    """Calls large enough for a full grid where the full grid (456 CTAs on 152
    SMs) is a multiple of the segment count: the host takes a grid one or more
    CTAs smaller; every element still matches the oracle."""
    import torch
    for op in ("sum", "max"):
        host = _data(7000 + W, W, N, dtype, op)
        xs = [to_device(h, dtype) for h in host]
        ys = [torch.empty_like(x) for x in xs]
        mr.mr_allreduce(xs, ys, op=op, algo=algo)
        torch.cuda.synchronize()
        want = oracle_allreduce(dtype, op, algo, host)
        for j, y in enumerate(ys):
            assert_same(to_host(y, dtype), want, f"allreduce {dtype} {op} {algo} W={W} rank {j}")


def test_sweep_fp32_w8_full(mr):
    """W=8 fp32 Normal(0,1) sum at every sweep size: ring bit-exact; tree
    bit-exact to the oracle's tree order and within 2*W*2^-24*sum|y| of ring."""
    import oracle
    import torch
    W = 8
    for N in synth.WORKLOADS["sweep_fp32_w8"]["Ns"]:
        host = synth.workload_inputs("sweep_fp32_w8", N=N)
        xs = [to_device(h, "fp32") for h in host]
        got = {}
        for algo in ALGOS:
            ys = [torch.empty_like(x) for x in xs]
            mr.mr_allreduce(xs, ys, op="sum", algo=algo)
            torch.cuda.synchronize()
            want = oracle.allreduce("fp32", "sum", algo, host)
            for j, y in enumerate(ys):
                assert_same(y.cpu().numpy(), want, f"sweep N={N} {algo} rank {j}")
            got[algo] = want
        mag = np.zeros(N, np.float64)
        for h in host:
            mag += np.abs(h.astype(np.float64))
        diff = np.abs(got["ring"].astype(np.float64) - got["tree"].astype(np.float64))
        assert np.all(diff <= 2 * W * 2.0 ** -24 * mag)
        del xs
