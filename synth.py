"""Seeded synthetic rank buffers: the one module that both the CUDA path's tests
and benchmark and the CPU oracle draw their inputs from.

It holds no reduction arithmetic.  It only draws random numbers and stores them
in the element type under test:

* rank r of a workload with seed s and stream tag t draws from
  ``numpy.random.Generator(PCG64(SeedSequence([s, t, r])))``;
* "uniform in [a, b]" is inclusive of both ends (``Generator.integers``);
* "Normal(0, sigma)" takes sigma as the standard deviation: numpy's float32
  standard normal times float32(sigma), one fp32 multiply;
* bf16 values are the fp32 draws converted by torch (round to nearest even),
  held as uint16 bit patterns.

The workloads mirror the shapes on the pages: a DDP gradient bucket, the
FSDP bf16 gradient and parameter shards, an integer count all-reduce and the
nccl-tests size sweep.
"""
from __future__ import annotations

import numpy as np

TAG_GRAD = 0
TAG_PARAM = 1
TAG_RESIDUAL = 2
TAG_WEIGHT = 3
TAG_ERR = 4


def _rng(seed: int, tag: int, r: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, r])))


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def uniform_int(seed: int, W: int, N: int, lo: int, hi: int, dtype: str = "int32", tag: int = TAG_GRAD):
    """W buffers of N integers uniform in [lo, hi]; dtype 'int32' or 'fp32'
    (small integers stored exactly as floats)."""
    out = []
    for r in range(W):
        v = _rng(seed, tag, r).integers(lo, hi, size=N, endpoint=True, dtype=np.int64)
        out.append(v.astype(np.int32) if dtype == "int32" else v.astype(np.float32))
    return out


def normal(seed: int, W: int, N: int, sigma: float, dtype: str = "fp32", tag: int = TAG_GRAD):
    """W buffers of N draws from Normal(0, sigma) in fp32 or bf16 (uint16 bits)."""
    out = []
    for r in range(W):
        z = _rng(seed, tag, r).standard_normal(N, dtype=np.float32)
        z *= np.float32(sigma)
        out.append(z if dtype == "fp32" else _to_bf16_bits(z))
    return out


def near_one(seed: int, W: int, N: int, dtype: str = "fp32", tag: int = TAG_GRAD):
    """W buffers uniform in [0.5, 1.5) (products of up to 64 stay finite)."""
    out = []
    for r in range(W):
        z = _rng(seed, tag, r).uniform(0.5, 1.5, size=N).astype(np.float32)
        out.append(z if dtype == "fp32" else _to_bf16_bits(z))
    return out


def bf16_wide(seed: int, W: int, N: int, tag: int = TAG_GRAD):
    """W buffers of N bf16 bit patterns spread over the whole exponent range
    below 2^73 (so sums of up to 64 stay finite): random sign and mantissa,
    exponent field uniform in [0, 200], one in eight subnormal (field 0).
    Sums of such values span gaps far wider than fp32's precision and land
    on bf16 ties, the cases where rounding order matters."""
    out = []
    for r in range(W):
        g = _rng(seed, tag, r)
        sign = g.integers(0, 2, size=N, dtype=np.uint16) << 15
        mant = g.integers(0, 128, size=N, dtype=np.uint16)
        expo = g.integers(1, 201, size=N, dtype=np.uint16)
        expo[g.integers(0, 8, size=N) == 0] = 0
        out.append((sign | (expo << 7) | mant).astype(np.uint16))
    return out


def random_values(seed: int, W: int, N: int, dtype: str, kind: str = "normal", tag: int = TAG_GRAD):
    """Generic test data.  int32: uniform in [-1000, 1000].  Floats: 'normal'
    (sigma 1), 'small_int' (integers in [-8, 8]) or 'near_one' ([0.5, 1.5))."""
    if dtype == "int32":
        return uniform_int(seed, W, N, -1000, 1000, "int32", tag)
    if kind == "small_int":
        vals = uniform_int(seed, W, N, -8, 8, "fp32", tag)
        return vals if dtype == "fp32" else [_to_bf16_bits(v) for v in vals]
    if kind == "near_one":
        return near_one(seed, W, N, dtype, tag)
    return normal(seed, W, N, 1.0, dtype, tag)


# The workloads, by what they are.  Every size is per rank.
WORKLOADS = {
    # W=2, 4096 fp32 per rank, integers in [-8, 8]: sums are exact.
    "small_int_fp32_w2": dict(W=2, N=4096, dtype="fp32", dist=("uniform_int", -8, 8)),
    # W=8 DDP gradient bucket: 2^24 fp32 per rank (64 MiB), Normal(0, 1e-3).
    "ddp_bucket_fp32_w8": dict(W=8, N=1 << 24, dtype="fp32", dist=("normal", 1e-3)),
    # W=8 FSDP step: 2^26 bf16 gradient per rank, Normal(0, 1e-2); parameter
    # shards of 2^23 bf16, Normal(0, 0.02).
    "fsdp_bf16_w8": dict(W=8, N=1 << 26, dtype="bf16", dist=("normal", 1e-2),
                         param_dist=("normal", 0.02)),
    # W=16 integer counts: 2^22 int32 per rank, uniform in [-1000, 1000].
    "int_counts_w16": dict(W=16, N=1 << 22, dtype="int32", dist=("uniform_int", -1000, 1000)),
    # W=8 tensor-parallel decode step: 64 tokens x hidden 8192 bf16 partial
    # outputs Normal(0, 1e-2) per rank, a bf16 residual stream Normal(0, 1) and
    # an RMSNorm weight 1 + Normal(0, 0.1).
    "tp_decode_rmsnorm_bf16_w8": dict(W=8, rows=64, hidden=8192, N=64 * 8192, dtype="bf16",
                                      dist=("normal", 1e-2), residual_dist=("normal", 1.0),
                                      weight_dist=("normal_mean", 1.0, 0.1)),
    # The same at prefill size: 4096 tokens x 8192.
    "tp_prefill_rmsnorm_bf16_w8": dict(W=8, rows=4096, hidden=8192, N=4096 * 8192, dtype="bf16",
                                       dist=("normal", 1e-2), residual_dist=("normal", 1.0),
                                       weight_dist=("normal_mean", 1.0, 0.1)),
    # W=8 DDP bucket sent as 1-bit signs with error feedback: 2^24 fp32
    # gradients Normal(0, 1e-3) and a carried residual Normal(0, 1e-4).
    "sign_ef_fp32_w8": dict(W=8, N=1 << 24, dtype="fp32", dist=("normal", 1e-3), err_dist=("normal", 1e-4)),
    # W=16 ranks as 2 nodes x 8 GPUs: 2^24 bf16 gradients per rank,
    # Normal(0, 1e-2), for the two-level (hierarchical) all-reduce order.
    "hier_bf16_w16": dict(W=16, N=1 << 24, dtype="bf16", dist=("normal", 1e-2)),
    # W=8 size sweep: fp32 Normal(0, 1), N = 2^10, 2^12, ..., 2^26.
    "sweep_fp32_w8": dict(W=8, Ns=[1 << p for p in range(10, 27, 2)], dtype="fp32", dist=("normal", 1.0)),
}


def draw(dist, seed: int, W: int, N: int, dtype: str, tag: int = TAG_GRAD):
    kind = dist[0]
    if kind == "uniform_int":
        return uniform_int(seed, W, N, dist[1], dist[2], dtype, tag)
    if kind == "normal":
        return normal(seed, W, N, dist[1], dtype, tag)
    if kind == "normal_mean":
        out = []
        for r in range(W):
            z = _rng(seed, tag, r).standard_normal(N, dtype=np.float32)
            z = z * np.float32(dist[2]) + np.float32(dist[1])
            out.append(z if dtype == "fp32" else _to_bf16_bits(z))
        return out
    raise ValueError(kind)


def workload_inputs(name: str, seed: int = 0, N: int | None = None, W: int | None = None,
                    dtype: str | None = None):
    """The rank buffers of a named workload.  N overrides the size (for sweeps
    and bounded samples); W and dtype override the rank count and the element
    type, keeping the workload's distribution (an integer distribution is
    needed for int32)."""
    w = WORKLOADS[name]
    n = N if N is not None else w["N"]
    dt = dtype or w["dtype"]
    if dt == "int32" and w["dist"][0] != "uniform_int":
        raise ValueError(f"{name} draws floats; int32 needs an integer workload")
    return draw(w["dist"], seed, W or w["W"], n, dt, TAG_GRAD)


def workload_param_shards(name: str, seed: int = 0, N: int | None = None):
    """The parameter shards of the FSDP workload (W shards of N/W elements)."""
    w = WORKLOADS[name]
    n = N if N is not None else w["N"]
    return draw(w["param_dist"], seed, w["W"], n // w["W"], w["dtype"], TAG_PARAM)


def workload_norm_operands(name: str, seed: int = 0, rows: int | None = None):
    """(inputs, residual, weight) of a fused all-reduce + RMSNorm workload."""
    w = WORKLOADS[name]
    r = rows if rows is not None else w["rows"]
    n = r * w["hidden"]
    ins = draw(w["dist"], seed, w["W"], n, w["dtype"], TAG_GRAD)
    res = draw(w["residual_dist"], seed, 1, n, w["dtype"], TAG_RESIDUAL)[0]
    wt = draw(w["weight_dist"], seed, 1, w["hidden"], w["dtype"], TAG_WEIGHT)[0]
    return ins, res, wt


def workload_sign_operands(name: str, seed: int = 0, N: int | None = None):
    """(gradients, residuals) of a sign-compression workload."""
    w = WORKLOADS[name]
    n = N if N is not None else w["N"]
    return (draw(w["dist"], seed, w["W"], n, w["dtype"], TAG_GRAD),
            draw(w["err_dist"], seed, w["W"], n, w["dtype"], TAG_ERR))


def device_normal(seed: int, W: int, N: int, dtype: str, device="cuda", tag: int = TAG_GRAD):
    """W rank buffers of N Normal(0, 1) draws made on the GPU by torch's
    seeded generator (rank r: seed s * 1000 + 100 * tag + r) -- for buffers
    too large to draw and copy from the host.  fp32 or bf16."""
    import torch
    out = []
    for r in range(W):
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + 100 * tag + r)
        x = torch.randn(N, generator=g, device=device, dtype=torch.float32)
        out.append(x if dtype == "fp32" else x.to(torch.bfloat16))
    return out
