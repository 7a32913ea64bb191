"""GPU parity of the 1-bit sign compression with error feedback.

The scales are checked against the oracle's fp64 L1 norm to within one fp32
unit (both round a nearly exact fp64 sum once; the orders differ).  Given the
GPU's own scales, the oracle then reproduces the outputs and the new errors
bit for bit.
"""
import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_same, to_device, to_host

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


def _shift(t, offset):
    import torch
    if not offset:
        return t
    buf = torch.empty(t.numel() + offset, dtype=t.dtype, device=t.device)
    buf[offset:].copy_(t)
    return buf[offset:]


def run(mr, mode, op, algo, g, e, offset=0, steps=1):
    import oracle
    import torch
    W, N = len(g), g[0].size
    gd = [_shift(to_device(x, "fp32"), offset) for x in g]
    ed = [_shift(to_device(x, "fp32"), offset) for x in e]
    n_out = N if mode == "allreduce" else N // W
    host_e = [x.copy() for x in e]
    for _ in range(steps):
        outs = Guarded(W, n_out, "fp32", offset=offset)
        scales = torch.empty(W, device="cuda")
        fn = mr.mr_allreduce_sign_ef if mode == "allreduce" else mr.mr_reduce_scatter_sign_ef
        fn(gd, ed, outs.views, scales=scales, op=op, algo=algo)
        torch.cuda.synchronize()
        outs.check()
        s_gpu = scales.cpu().numpy()
        s_ref = oracle.sign_ef_scales(g, host_e)
        assert np.all(np.abs(s_gpu - s_ref) <= np.spacing(s_ref)), (s_gpu, s_ref)
        want, host_e = oracle.sign_ef_collective(mode, op, algo, g, host_e, s_gpu)
        got = outs.host()
        if mode == "allreduce":
            for j in range(W):
                assert_same(got[j], want, f"{mode} {op} {algo} W={W} N={N} rank {j}")
        else:
            for k in range(W):
                assert_same(got[k], want[k], f"{mode} {op} {algo} W={W} N={N} shard {k}")
        for r in range(W):
            assert_same(to_host(ed[r], "fp32"), host_e[r], f"error feedback rank {r}")


@pytest.mark.parametrize("W,N", [(1, 1000), (2, 64), (3, 3 * 4099), (8, 8 * 5000 + 8), (8, 8 * 3), (13, 13 * 333),
                                 (16, 16 * 2048), (17, 17 * 101), (64, 64 * 64)])
@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_parity(mr, W, N, op, algo):
    g = synth.normal(50 + W, W, N, 1e-3, "fp32")
    e = synth.normal(60 + W, W, N, 1e-4, "fp32")
    run(mr, "reduce_scatter", op, algo, g, e)
    run(mr, "allreduce", op, algo, g, e)


@pytest.mark.parametrize("offset", [1, 2])
def test_unaligned_and_repeated(mr, offset):
    """Element-aligned pointers (offset 2 is 8- but not 16-byte aligned: the
    L1 pass must not use 16-byte loads), and three steps in a row carrying the
    error state on the GPU."""
    for W in (8, 16):
        N = W * 1003
        g = synth.normal(70 + W, W, N, 1e-3, "fp32")
        e = [np.zeros(N, np.float32) for _ in range(W)]
        run(mr, "allreduce", "avg", "ring", g, e, offset=offset, steps=3)


def test_workload_full(mr):
    """W=8, 2^24 fp32 per rank, reduce-scatter avg, ring order."""
    g, e = synth.workload_sign_operands("sign_ef_fp32_w8")
    run(mr, "reduce_scatter", "avg", "ring", g, e)


def test_errors(mr):
    import torch
    x = [torch.zeros(64, device="cuda") for _ in range(2)]
    er = [torch.zeros(64, device="cuda") for _ in range(2)]
    y = [torch.zeros(64, device="cuda") for _ in range(2)]
    with pytest.raises(mr.MRError) as ex:
        mr.mr_allreduce_sign_ef(x, er, y, op="max")
    assert ex.value.status == 2
    with pytest.raises(mr.MRError) as ex:
        mr.mr_allreduce_sign_ef(x, [er[0], er[0]], y)        # two ranks share one residual
    assert ex.value.status == 3
    with pytest.raises(mr.MRError) as ex:
        mr.mr_allreduce_sign_ef(x, er, y, workspace=torch.empty(8, dtype=torch.uint8, device="cuda"))
    assert ex.value.status == 1
