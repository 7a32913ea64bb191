"""GPU parity of the fused all-reduce + residual + RMSNorm against the oracle.

residual_out (the sum plus residual) must match bit for bit: it is the
all-reduce's own arithmetic.  The normalised output is held to a tolerance
derived from the kernel's fp32 arithmetic against the oracle's fp64
evaluation (see ``tolerance``).  All W outputs must be identical.
"""
import math

import numpy as np
import pytest

import synth
from gpu_util import Guarded, assert_same, to_device, to_host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


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


def tolerance(hidden):
    """Relative bound of |kernel - exact| before the final rounding.  The
    kernel's row sum of squares is a per-thread sequential fp32 sum of at most
    ceil(hidden / 256) + 8 terms, then an 8-level tree (256 threads), then at
    most 8 slice totals added in order (a row split over a cluster), plus one
    rounding per square: relative error <= (P + 9) u with
    P = ceil(hidden / 256) + 16.  The mean, + eps, sqrt and divide add 1 u
    each (sqrt halves the incoming error), and the two multiplies 1 u each:
    (P + 9)/2 u + 6 u in total."""
    P = math.ceil(hidden / 256) + 16
    return ((P + 9) / 2 + 6) * U


def _f32(dtype, a):
    return (a.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else a.astype(np.float32)


def check_out(dtype, got, want, hidden):
    g = _f32(dtype, got).astype(np.float64)
    w = _f32(dtype, want).astype(np.float64)
    rel = tolerance(hidden)
    bound = rel * np.abs(w) + np.spacing(np.abs(w).astype(np.float32)).astype(np.float64)
    if dtype == "bf16":
        # both sides round to bf16: values within `rel` of each other can land
        # one bf16 unit apart
        bound = np.maximum(bound, np.spacing(np.abs(w).astype(np.float32)).astype(np.float64) * 65536)
    bad = np.nonzero(np.abs(g - w) > bound)[0]
    assert bad.size == 0, f"{bad.size} elements out of tolerance, first {bad[0]}: got {g[bad[0]]} want {w[bad[0]]}"


def run(mr, dtype, algo, W, rows, hidden, residual=True, residual_out=True, inplace=False, offset=0, seed=0):
    import oracle
    import torch
    N = rows * hidden
    ins = synth.normal(seed + 31, W, N, 0.3, dtype)
    res = synth.normal(seed + 32, 1, N, 1.0, dtype)[0] if residual else None
    wt = synth.draw(("normal_mean", 1.0, 0.1), seed + 33, 1, hidden, dtype)[0]
    eps = 1e-5
    want, want_res = oracle.allreduce_rmsnorm(dtype, algo, ins, rows, hidden, wt, residual=res, eps=eps,
                                              want_residual_out=residual_out)
    xs = [to_device(h, dtype) for h in ins]
    if offset:
        shifted = []
        for x in xs:
            buf = torch.empty(N + offset, dtype=x.dtype, device=x.device)
            buf[offset:].copy_(x)
            shifted.append(buf[offset:])
        xs = shifted
    w_d = to_device(wt, dtype)
    r_d = to_device(res, dtype) if residual else None
    ro = Guarded(1, N, dtype) if residual_out else None
    if inplace:
        outs = xs
        mr.mr_allreduce_rmsnorm(xs, xs, w_d, residual=r_d, residual_out=r_d if residual_out and residual else
                                (ro.views[0] if ro else None), eps=eps, algo=algo)
        torch.cuda.synchronize()
        got = [to_host(x, dtype) for x in outs]
        got_res = to_host(r_d, dtype) if (residual_out and residual) else (ro.host()[0] if ro else None)
    else:
        g = Guarded(W, N, dtype, offset=offset)
        mr.mr_allreduce_rmsnorm(xs, g.views, w_d, residual=r_d, residual_out=ro.views[0] if ro else None,
                                eps=eps, algo=algo)
        torch.cuda.synchronize()
        g.check()
        got = g.host()
        got_res = ro.host()[0] if ro else None
    if ro is not None:
        ro.check()
    for j in range(1, W):
        assert_same(got[j], got[0], f"rank {j} differs from rank 0")
    check_out(dtype, got[0], want, hidden)
    if residual_out:
        assert_same(got_res, want_res, "residual_out")


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("W,rows,hidden", [(1, 3, 64), (2, 5, 100), (3, 7, 1000), (8, 33, 4096), (8, 4, 8192),
                                           (13, 3, 2056), (16, 9, 2048), (17, 2, 96), (8, 2, 49152),
                                           # more rows than one wave of CTAs: a CTA takes 2-3 rows, pass 2 of
                                           # one in the same loop as pass 1 of the next (two row buffers)
                                           (8, 1000, 256), (3, 1001, 264), (16, 700, 512)])
def test_parity(mr, dtype, algo, W, rows, hidden):
    run(mr, dtype, algo, W, rows, hidden, seed=W * 100 + rows)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_options(mr, dtype):
    run(mr, dtype, "ring", 8, 6, 512, residual=False, residual_out=False)
    run(mr, dtype, "ring", 8, 6, 512, residual=True, residual_out=False)
    run(mr, dtype, "ring", 8, 6, 512, residual=False, residual_out=True)
    run(mr, dtype, "tree", 8, 6, 512, inplace=True)
    run(mr, dtype, "ring", 5, 6, 512, offset=1)
    # the same on rows enough for two or three per CTA
    run(mr, dtype, "ring", 8, 1000, 128, residual=False, residual_out=True)
    run(mr, dtype, "ring", 8, 1000, 128, residual=True, residual_out=False)
    run(mr, dtype, "tree", 8, 1000, 128, inplace=True)


def test_workloads_full(mr):
    """The decode and prefill workloads (W=8, 64 / 4096 rows of 8192 bf16)."""
    import oracle
    import torch
    for name in ("tp_decode_rmsnorm_bf16_w8", "tp_prefill_rmsnorm_bf16_w8"):
        w = synth.WORKLOADS[name]
        ins, res, wt = synth.workload_norm_operands(name)
        want, want_res = oracle.allreduce_rmsnorm("bf16", "ring", ins, w["rows"], w["hidden"], wt, residual=res,
                                                  eps=1e-6)
        xs = [to_device(h, "bf16") for h in ins]
        ys = [torch.empty_like(x) for x in xs]
        r_d = to_device(res, "bf16")
        ro = torch.empty_like(r_d)
        mr.mr_allreduce_rmsnorm(xs, ys, to_device(wt, "bf16"), residual=r_d, residual_out=ro, eps=1e-6)
        torch.cuda.synchronize()
        assert_same(to_host(ro, "bf16"), want_res, name)
        for y in ys:
            check_out("bf16", to_host(y, "bf16"), want, w["hidden"])


def test_errors(mr):
    import torch
    xs = [torch.zeros(64, dtype=torch.int32, device="cuda") for _ in range(2)]
    with pytest.raises(mr.MRError) as e:
        mr.mr_allreduce_rmsnorm(xs, xs, torch.zeros(64, dtype=torch.int32, device="cuda"))
    assert e.value.status == 2
    xf = [torch.zeros(64, device="cuda") for _ in range(2)]
    with pytest.raises(mr.MRError) as e:     # the weight aliases an output
        mr.mr_allreduce_rmsnorm(xf, xf, xf[1][:16])
    assert e.value.status == 3
