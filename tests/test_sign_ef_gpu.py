"""GPU parity of the 1-bit sign compression with error feedback.

The scale is a function of the data alone (the exact mean magnitude rounded
once to fp32), so the GPU's scales must equal the oracle's bit for bit, and
the outputs and the new errors must equal what the oracle computes from its
own scales, bit for bit.
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
        assert_same(s_gpu, s_ref, f"scales {mode} W={W} N={N}")
        want, host_e = oracle.sign_ef_collective(mode, op, algo, g, host_e, s_ref)
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


def _hard_scale_ranks():
    """One rank per hand-worked case of the scale's exact rounding (ties,
    a remainder that decides a tie, subnormal means, the largest
    magnitudes, a mean an fp64 running sum would round the wrong way), each
    padded with zeros to a common N, plus ranks drawn over every binade."""
    two = 2.0
    cases = [[3.0, 3 * two ** -24, 3 * two ** -100], [1.0, 1 + two ** -23], [1 + two ** -23, 1 + two ** -22],
             [two ** -149, 0.0], [3 * two ** -149, 0.0], [2 * two ** -149, 0.0, 0.0],
             [3 * two ** -125, two ** -147, 0.0], [3.4028234663852886e38] * 2, [-2.0, 2.0, -0.0, 0.0]]
    return cases


@pytest.mark.parametrize("N", [3, 8, 4099, 8 * 8192 + 5])
def test_scales_exact_on_hard_cases(mr, N):
    """Scales of hand-worked and every-binade data, bit for bit.  Zero
    padding changes N but not the sum, so each case's mean is its own sum over
    this N.  The values are split as g + e with e = 0, and also with e
    carrying part of the value (the sum p = g + e is formed in fp32 on both
    sides)."""
    import oracle
    import torch
    rng = np.random.default_rng(N)
    ranks = []
    for c in _hard_scale_ranks():
        if len(c) > N:
            continue
        p = np.zeros(N, np.float32)
        p[:len(c)] = np.array(c, np.float32)
        ranks.append(p)
    for _ in range(3):
        bits = rng.integers(0, 0x7F800000, size=N, dtype=np.uint32) | (rng.integers(0, 2, size=N, dtype=np.uint32) << np.uint32(31))
        ranks.append(bits.view(np.float32).copy())
        ranks.append((bits.view(np.float32) * np.float32(2.0 ** -110)).astype(np.float32))
    W = len(ranks)
    for split in (False, True):
        if split:
            e = [(p * np.float32(0.25)).astype(np.float32) for p in ranks]
            g = [(p - x).astype(np.float32) for p, x in zip(ranks, e)]
        else:
            g, e = ranks, [np.zeros(N, np.float32) for _ in ranks]
        gd = [to_device(x, "fp32") for x in g]
        ed = [to_device(x, "fp32") for x in e]
        out = [torch.empty(N, device="cuda") for _ in range(W)]
        scales = torch.empty(W, device="cuda")
        mr.mr_allreduce_sign_ef(gd, ed, out, scales=scales, op="sum", algo="ring")
        torch.cuda.synchronize()
        assert_same(scales.cpu().numpy(), oracle.sign_ef_scales(g, e), f"hard scales N={N} split={split}")


def test_scales_of_non_finite_values(mr):
    """An infinite |p| makes its rank's scale +inf, a NaN makes it NaN (and
    wins over an infinity); the other ranks are unaffected."""
    import oracle
    import torch
    N = 4096
    g = [np.full(N, 0.5, np.float32) for _ in range(4)]
    g[1][17] = np.inf
    g[2][100] = -np.inf
    g[2][200] = np.nan
    e = [np.zeros(N, np.float32) for _ in range(4)]
    gd = [to_device(x, "fp32") for x in g]
    ed = [to_device(x, "fp32") for x in e]
    out = [torch.empty(N, device="cuda") for _ in range(4)]
    scales = torch.empty(4, device="cuda")
    mr.mr_allreduce_sign_ef(gd, ed, out, scales=scales, op="sum", algo="ring")
    torch.cuda.synchronize()
    got = scales.cpu().numpy()
    want = oracle.sign_ef_scales(g, e)
    assert got[0] == want[0] == np.float32(0.5) and got[3] == np.float32(0.5)
    assert np.isposinf(got[1]) and np.isposinf(want[1])
    assert np.isnan(got[2]) and np.isnan(want[2])


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
