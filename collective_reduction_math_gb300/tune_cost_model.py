"""Fit the alpha-beta cost model that MR_AUTO uses to pick an accumulation
order, and write it to csrc/cost_model.inc.

The model is the one the NCCL planner uses ("How NCCL picks: a cost model,
not a threshold", post on NCCL all-reduce): every candidate costs
    time = lat * latCount + bytes / bw,
and a call takes the argmin.  Here the candidates are the ring and tree
orders, and a call is one kernel launch (latCount = 1).  NCCL keeps a (lat, bw)
pair per protocol, each protocol serving its own range of message sizes; here
the ranges are set by where a call's buffers live and what bounds it: calls
whose buffers take at most 4 MiB are bound by latency, calls whose buffers fit
in L2 run from the cache, larger ones stream from HBM.  So lat (alpha, us) and
bw (beta, GB/s) are fitted three times per element type, rank count and order:
on calls with at most 4 MiB of buffers, on calls with more than that and at
most half of L2, and on calls with at least twice L2.  A call uses the pair of
the range its buffers fall in (the HBM pair beyond L2).  The sizes are
per-rank messages from 4 KiB up to 8 GB of buffers in all (every power of
two), the rank buffers carved from one allocation, each call timed back to
back on one stream.  Each fit minimises the squared relative error
of t = alpha + bytes / beta.

Run on the GPU the library will serve (it takes a few minutes):
    python -m collective_reduction_math_gb300.tune_cost_model
then rebuild (``__graft_entry__.build()``).
"""
from __future__ import annotations

import datetime
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "csrc", "cost_model.inc")
WS = (2, 4, 8, 16, 32, 64)
DTYPES = (("fp32", 0, 4), ("bf16", 1, 2), ("int32", 2, 4))
ALGOS = (("ring", 0), ("tree", 1))
BYTES_PER_RANK = [4096 << i for i in range(19)]           # 4 KiB, 8 KiB, ... 1 GiB per rank
MAX_FOOTPRINT = 8 << 30                                    # W inputs + W outputs
LATENCY_BYTES = 4 << 20                                    # calls with at most this much of buffers


def device_us(torch, fn, bytes_, reps=5):
    """Device time of one call: `n` calls queued back to back on one stream
    (the stream first held on the device while the host queues them), one
    event pair around them all, best of `reps` rounds.  This is how the
    benchmark times a call; in CUDA graphs the ring and tree orders compare
    differently by a few percent at large sizes, more than they differ by."""
    n = 200 if bytes_ <= (64 << 20) else 20
    for _ in range(3):
        fn()
    best = float("inf")
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) * 1e3 / n)
    return best


def fit(bytes_, times):
    """alpha (us), beta (GB/s) minimising sum(((alpha + x/beta) - t) / t)^2."""
    x = np.asarray(bytes_, dtype=np.float64)
    t = np.asarray(times, dtype=np.float64)
    A = np.stack([1.0 / t, x / t], axis=1)           # (alpha, 1/beta) weighted by 1/t
    coef, *_ = np.linalg.lstsq(A, np.ones_like(t), rcond=None)
    alpha, inv_beta = max(coef[0], 0.0), max(coef[1], 1e-12)
    return alpha, 1e-3 / inv_beta                    # bytes/us -> GB/s


def rank_buffers(torch, dev, tdt, W, N):
    """W input and W output rank buffers of N elements, side by side in one
    allocation on 256-byte boundaries (the layout of a framework's flat
    buffers, and of the benchmark): where buffers land in HBM moves the
    throughput by a few percent, more than ring and tree differ by at large
    sizes."""
    es = torch.empty((), dtype=tdt).element_size()
    stride = (N * es + 255) // 256 * 256
    slab = torch.empty(2 * W * stride, dtype=torch.uint8, device=dev)
    bufs = [slab[i * stride:i * stride + N * es].view(tdt) for i in range(2 * W)]
    for x in bufs[:W]:
        if tdt == torch.int32:
            x.copy_(torch.randint(-1000, 1000, (N,), dtype=tdt, device=dev))
        else:
            x.copy_(torch.randn(N, device=dev).to(tdt))
    return bufs[:W], bufs[W:], slab


def render(rows, dev_name, date, l2):
    """The C++ text of cost_model.inc: the range bounds and the table."""
    lines = [
        "// cost_model.inc -- the all-reduce kernel's t = alpha + bytes / beta, per element type,",
        "// rank count and order, fitted on three ranges of a call's buffers: at most",
        "// kCostModelLatencyBytes (latency-bound), up to kCostModelL2Bytes (the L2 of the GPU the",
        "// table was fitted on; fitted on calls within half of it) and beyond (fitted on calls",
        "// of at least twice L2).  MR_AUTO takes the argmin with the pair of the call's range.",
        f"// Fitted by collective_reduction_math_gb300/tune_cost_model.py on {dev_name},",
        f"// {date}, from device times of calls launched back to back (4 KiB per rank to 8 GB",
        "// of buffers in all, carved from one allocation).",
        f"constexpr double kCostModelLatencyBytes = {float(LATENCY_BYTES):.1f};",
        f"constexpr double kCostModelL2Bytes = {float(l2):.1f};",
        "// {dtype, W, algo, {alpha_us, beta_gbs} x (latency, L2, HBM)}",
        "const CostRow kCostModel[] = {",
    ]
    for code, W, acode, *ab in rows:
        pairs = ", ".join(f"{{{ab[2 * i]:.3f}, {ab[2 * i + 1]:.1f}}}" for i in range(3))
        lines.append(f"    {{{code}, {W}, {acode}, {{{pairs}}}}},")
    lines.append("};")
    return "\n".join(lines) + "\n"


def main():
    import argparse

    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=OUT, help="where to write the table (default: csrc/cost_model.inc)")
    out = ap.parse_args().out

    import collective_reduction_math_gb300 as mr
    mr.load()
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    rows = []
    for name, code, b in DTYPES:
        tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "int32": torch.int32}[name]
        for W in WS:
            for algo, acode in ALGOS:
                pts = []
                for per_rank in BYTES_PER_RANK:
                    if 2 * W * per_rank > MAX_FOOTPRINT:
                        break
                    N = per_rank // b
                    xs, ys, slab = rank_buffers(torch, dev, tdt, W, N)
                    t = device_us(torch, lambda: mr.mr_allreduce(xs, ys, op="sum", algo=algo), 2 * W * N * b)
                    pts.append((2 * W * N * b, t))
                    del xs, ys, slab
                    torch.cuda.empty_cache()
                small = [p for p in pts if p[0] <= LATENCY_BYTES]
                cache = [p for p in pts if LATENCY_BYTES < p[0] <= l2 // 2]
                hbm = [p for p in pts if p[0] >= 2 * l2]
                assert min(len(small), len(cache), len(hbm)) >= 2, (name, W, algo, pts)
                fits = [fit(*zip(*r)) for r in (small, cache, hbm)]
                rows.append((code, W, acode, *[v for f in fits for v in f]))
                print(f"{name:5s} W={W:2d} {algo:4s} " + "  ".join(
                    f"{tag}: alpha={a:6.2f} us beta={b:6.0f} GB/s" for tag, (a, b) in zip(("lat", "L2", "HBM"), fits)),
                      flush=True)
                for x, t in pts:
                    print(f"    {x:>12d} B  {t:10.3f} us", flush=True)
    dev_name = torch.cuda.get_device_name(dev)
    with open(out, "w") as f:
        f.write(render(rows, dev_name, datetime.date.today().isoformat(), l2))
    print(f"wrote {out}")


if __name__ == "__main__":
    sys.exit(main())
