"""Back-to-back dependent calls on one stream, with no synchronisation between
them, against the oracle applied in the same sequence.

Every kernel of the library is launched with programmatic dependent launch:
its launch may overlap the tail of the kernel before it, and it waits for that
kernel (griddepcontrol.wait) before touching memory.  These tests chain calls
whose inputs are the previous call's outputs (read after write), whose outputs
are the previous call's inputs (write after read), in-place forms, torch
kernels in between, and the same chains replayed from a CUDA graph.  Any call
that read or wrote too early would change a result; every comparison is
bit-exact.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from gpu_util import assert_same, to_device, to_host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


# few CTAs (the next launch can sit beside the running one) and several waves
SIZES = [(8, 8 * 1000 + 5), (8, 1 << 20), (16, 16 * 4096 + 3)]


@pytest.mark.parametrize("W,N", SIZES)
@pytest.mark.parametrize("dtype,op", [("int32", "sum"), ("fp32", "avg"), ("bf16", "max")])
def test_allreduce_chain(mr, oracle_mod, W, N, dtype, op):
    """x -> y -> y (in place) -> x -> ..., eight calls, one sync at the end."""
    import torch
    host = synth.random_values(7, W, N, dtype)
    xs = [to_device(h, dtype) for h in host]
    ys = [torch.empty_like(x) for x in xs]
    want = host
    algos = ["ring", "tree"]
    for i in range(8):
        algo = algos[i % 2]
        if i % 3 == 0:
            mr.mr_allreduce(xs, ys, op=op, algo=algo)
            xs, ys = ys, xs
        else:
            mr.mr_allreduce(xs, xs, op=op, algo=algo)
        want = [oracle_mod.allreduce(dtype, op, algo, want)] * W
    torch.cuda.synchronize()
    for r in range(W):
        assert_same(to_host(xs[r], dtype), want[r], f"chain {dtype} {op} W={W} N={N} rank {r}")


@pytest.mark.parametrize("W,N", [(8, 8 * 2048), (8, 8 << 17), (4, 4 * 777)])
def test_write_after_read(mr, oracle_mod, W, N):
    """a -> b; c -> a (overwrites what the first call read); b -> c
    (reads what the first call wrote, overwrites what the second read)."""
    import torch
    ha = synth.random_values(1, W, N, "fp32")
    hc = synth.random_values(2, W, N, "fp32")
    a = [to_device(h, "fp32") for h in ha]
    c = [to_device(h, "fp32") for h in hc]
    b = [torch.empty_like(x) for x in a]
    for _ in range(3):
        mr.mr_allreduce(a, b, op="sum", algo="ring")
        mr.mr_allreduce(c, a, op="sum", algo="ring")
        mr.mr_allreduce(b, c, op="sum", algo="tree")
        want_b = oracle_mod.allreduce("fp32", "sum", "ring", ha)
        want_a = oracle_mod.allreduce("fp32", "sum", "ring", hc)
        want_c = oracle_mod.allreduce("fp32", "sum", "tree", [want_b] * W)
        ha, hc = [want_a] * W, [want_c] * W
    torch.cuda.synchronize()
    for r in range(W):
        assert_same(to_host(a[r], "fp32"), ha[r], f"a rank {r}")
        assert_same(to_host(c[r], "fp32"), hc[r], f"c rank {r}")
        assert_same(to_host(b[r], "fp32"), want_b, f"b rank {r}")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_reduce_scatter_all_gather_allreduce_chain(mr, oracle_mod, dtype):
    """RS -> AG -> AR (in place) -> RS (in place) -> AG (in place), with a
    torch kernel in the middle, one sync at the end."""
    import torch
    W, N = 8, 8 * 65536
    C = N // W
    host = synth.random_values(3, W, N, dtype)
    xs = [to_device(h, dtype) for h in host]
    shards = [torch.empty(C, dtype=xs[0].dtype, device="cuda") for _ in range(W)]
    full = [torch.empty_like(x) for x in xs]
    mr.mr_reduce_scatter(xs, shards, op="avg", algo="ring")
    mr.mr_all_gather(shards, full)
    mr.mr_allreduce(full, full, op="sum", algo="tree")
    for f in full:
        f.neg_()                                     # a plain torch kernel in between
    views = [full[r][r * C:(r + 1) * C] for r in range(W)]
    mr.mr_reduce_scatter(full, views, op="max", algo="ring")       # in place: recv[r] = send[r] + r*C
    mr.mr_all_gather(views, full)                                  # in place: send[r] = recv[r] + r*C
    torch.cuda.synchronize()

    s = oracle_mod.reduce_scatter(dtype, "avg", "ring", host)
    g = np.concatenate(s)
    a = oracle_mod.allreduce(dtype, "sum", "tree", [g] * W)
    neg = a ^ np.uint16(0x8000) if dtype == "bf16" else -a        # negation flips the sign bit
    s2 = oracle_mod.reduce_scatter(dtype, "max", "ring", [neg] * W)
    want = np.concatenate(s2)
    for r in range(W):
        assert_same(to_host(full[r], dtype), want, f"{dtype} rank {r}")


def test_sign_ef_steps_back_to_back(mr, oracle_mod):
    """Three sign-compressed all-reduce steps and an all-reduce of each result,
    queued without a sync: the residual carries from step to step."""
    import torch
    W, N = 8, 8 * 40000
    g = synth.normal(11, W, N, 1e-3, "fp32")
    e = synth.normal(12, W, N, 1e-4, "fp32")
    dg = [torch.from_numpy(x).cuda() for x in g]
    de = [torch.from_numpy(x).cuda() for x in e]
    outs = [[torch.empty(N, device="cuda") for _ in range(W)] for _ in range(3)]
    sums = [[torch.empty(N, device="cuda") for _ in range(W)] for _ in range(3)]
    scales = [torch.empty(W, device="cuda") for _ in range(3)]
    for t in range(3):
        mr.mr_allreduce_sign_ef(dg, de, outs[t], scales=scales[t], op="avg", algo="ring")
        mr.mr_allreduce(outs[t], sums[t], op="sum", algo="ring")
    torch.cuda.synchronize()
    errs = e
    for t in range(3):
        want_scales = oracle_mod.sign_ef_scales(g, errs)
        assert_same(scales[t].cpu().numpy(), want_scales, f"step {t} scales")
        out, errs = oracle_mod.sign_ef_collective("allreduce", "avg", "ring", g, errs, want_scales)
        for r in range(W):
            assert_same(outs[t][r].cpu().numpy(), out, f"step {t} rank {r}")
        want_sum = oracle_mod.allreduce("fp32", "sum", "ring", [out] * W)
        assert_same(sums[t][0].cpu().numpy(), want_sum, f"step {t} sum")
    for r in range(W):
        assert_same(de[r].cpu().numpy(), errs[r], f"final residual {r}")


def test_chain_replayed_from_a_graph(mr, oracle_mod):
    """The same kind of chain captured into a CUDA graph and replayed twice."""
    import torch
    W, N = 8, 8 * 3000 + 7
    host = synth.random_values(5, W, N, "int32")
    xs = [to_device(h, "int32") for h in host]
    ys = [torch.empty_like(x) for x in xs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(4):
                mr.mr_allreduce(xs, ys, op="sum", algo="ring")
                mr.mr_allreduce(ys, xs, op="max", algo="tree")
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = host
    for _ in range(2):
        graph.replay()
        for _ in range(4):
            y = oracle_mod.allreduce("int32", "sum", "ring", want)
            want = [oracle_mod.allreduce("int32", "max", "tree", [y] * W)] * W
    torch.cuda.synchronize()
    for r in range(W):
        assert_same(to_host(xs[r], "int32"), want[r], f"graph replay rank {r}")


def test_pdl_off_gives_the_same_results():
    """MR_PDL=0 launches every kernel in plain stream order; a fresh process
    runs a short chain that way and checks it against the oracle."""
    code = (
        "import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
        "import torch, synth, oracle, collective_reduction_math_gb300 as mr\n"
        "from gpu_util import to_device, to_host\n"
        "mr.load(); oracle.build()\n"
        "W, N = 8, 8 * 5000 + 3\n"
        "h = synth.random_values(9, W, N, 'int32')\n"
        "xs = [to_device(x, 'int32') for x in h]; ys = [torch.empty_like(x) for x in xs]\n"
        "mr.mr_allreduce(xs, ys, op='sum'); mr.mr_allreduce(ys, xs, op='min', algo='tree')\n"
        "torch.cuda.synchronize()\n"
        "w = oracle.allreduce('int32', 'min', 'tree', [oracle.allreduce('int32', 'sum', 'ring', h)] * W)\n"
        "assert all(to_host(x, 'int32').tobytes() == w.tobytes() for x in xs)\n"
        "print('ok')\n" % (ROOT, os.path.join(ROOT, "tests")))
    env = dict(os.environ, MR_PDL="0")
    p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout + p.stderr


@pytest.mark.parametrize("rows", [64, 600])
def test_rmsnorm_replayed_from_a_graph_matches_eager(mr, rows):
    """The fused RMSNorm (a thread-block-cluster launch for few rows) captured
    into a CUDA graph and replayed twice gives exactly the eager call's
    outputs; the eager call is held to the oracle by test_rmsnorm_gpu."""
    import torch
    W, H = 8, 8192
    N = rows * H
    xs = [to_device(h, "bf16") for h in synth.random_values(31, W, N, "bf16")]
    res = to_device(synth.random_values(32, 1, N, "bf16")[0], "bf16")
    wt = to_device(synth.random_values(33, 1, H, "bf16")[0], "bf16")
    eager = [torch.empty_like(x) for x in xs]
    eager_res = torch.empty_like(res)
    mr.mr_allreduce_rmsnorm(xs, eager, wt, residual=res, residual_out=eager_res, eps=1e-6)
    ys = [torch.empty_like(x) for x in xs]
    rout = torch.empty_like(res)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            mr.mr_allreduce_rmsnorm(xs, ys, wt, residual=res, residual_out=rout, eps=1e-6)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for y in ys:
            y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(rout, eager_res)
        for y, e in zip(ys, eager):
            assert torch.equal(y, e)


def test_sign_ef_steps_replayed_from_a_graph_match_eager(mr):
    """Two sign-compressed reduce-scatter steps (two kernels each, the second
    reading the first's partials) replayed from a CUDA graph give exactly two
    eager steps: outputs, scales and the carried residual."""
    import torch
    W, N = 8, 8 * 30000
    g = [torch.from_numpy(x).cuda() for x in synth.normal(41, W, N, 1e-3, "fp32")]
    e0 = synth.normal(42, W, N, 1e-4, "fp32")
    e_eager = [torch.from_numpy(x).cuda() for x in e0]
    e_graph = [torch.from_numpy(x).cuda() for x in e0]
    C = N // W
    out_e = [torch.empty(C, device="cuda") for _ in range(W)]
    out_g = [torch.empty(C, device="cuda") for _ in range(W)]
    s_e, s_g = torch.empty(W, device="cuda"), torch.empty(W, device="cuda")
    ws_e = torch.empty(mr.mr_sign_ef_workspace_bytes(W, N), dtype=torch.uint8, device="cuda")
    ws_g = torch.empty_like(ws_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            mr.mr_reduce_scatter_sign_ef(g, e_graph, out_g, scales=s_g, workspace=ws_g, op="avg", algo="ring")
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for step in range(2):
        mr.mr_reduce_scatter_sign_ef(g, e_eager, out_e, scales=s_e, workspace=ws_e, op="avg", algo="ring")
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(s_e, s_g), f"step {step}: scales"
        for k in range(W):
            assert torch.equal(out_e[k], out_g[k]), f"step {step}: shard {k}"
            assert torch.equal(e_eager[k], e_graph[k]), f"step {step}: residual {k}"
