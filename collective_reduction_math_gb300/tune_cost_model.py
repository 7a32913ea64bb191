"""Fit the alpha-beta cost model that MR_AUTO uses to pick an accumulation
order, and write it to csrc/cost_model.inc.

The model is the one the NCCL planner uses ("How NCCL picks: a cost model,
not a threshold", post on NCCL all-reduce): every candidate costs
    time = lat * latCount + bytes / bw,
and a call takes the argmin.  Here the candidates are the ring and tree
orders, a call is one kernel launch (latCount = 1), and lat (alpha, us) and bw
(beta, GB/s) are fitted per element type and rank count from device times
measured on this GPU: each order, each W in {2, 4, 8, 16, 32, 64}, per-rank
messages of 4 KiB to 64 MiB, every time the mean of a CUDA graph of calls.
The fit minimises the squared relative error of t = alpha + bytes / beta.

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
BYTES_PER_RANK = [4096 << (2 * i) for i in range(8)] + [64 << 20]     # 4 KiB ... 64 MiB


def device_us(torch, fn, calls=20, reps=3):
    """Mean device time of one call: a CUDA graph of `calls` calls, replayed."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) * 1e3 / calls)
    return best


def fit(bytes_, times):
    """alpha (us), beta (GB/s) minimising sum(((alpha + x/beta) - t) / t)^2."""
    x = np.asarray(bytes_, dtype=np.float64)
    t = np.asarray(times, dtype=np.float64)
    A = np.stack([1.0 / t, x / t], axis=1)           # (alpha, 1/beta) weighted by 1/t
    coef, *_ = np.linalg.lstsq(A, np.ones_like(t), rcond=None)
    alpha, inv_beta = max(coef[0], 0.0), max(coef[1], 1e-12)
    return alpha, 1e-3 / inv_beta                    # bytes/us -> GB/s


def main():
    import argparse

    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=OUT, help="where to write the table (default: csrc/cost_model.inc)")
    out = ap.parse_args().out

    import collective_reduction_math_gb300 as mr
    mr.load()
    dev = torch.device("cuda", 0)
    rows = []
    for name, code, b in DTYPES:
        tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "int32": torch.int32}[name]
        for W in WS:
            for algo, acode in ALGOS:
                xs_b, ts = [], []
                for per_rank in BYTES_PER_RANK:
                    N = per_rank // b
                    if name == "int32":
                        xs = [torch.randint(-1000, 1000, (N,), dtype=tdt, device=dev) for _ in range(W)]
                    else:
                        xs = [torch.randn(N, device=dev).to(tdt) for _ in range(W)]
                    ys = [torch.empty_like(x) for x in xs]
                    t = device_us(torch, lambda: mr.mr_allreduce(xs, ys, op="sum", algo=algo))
                    xs_b.append(2 * W * N * b)
                    ts.append(t)
                    del xs, ys
                alpha, beta = fit(xs_b, ts)
                rows.append((code, W, acode, alpha, beta))
                print(f"{name:5s} W={W:2d} {algo:4s} alpha={alpha:7.2f} us  beta={beta:7.0f} GB/s", flush=True)
    dev_name = torch.cuda.get_device_name(dev)
    with open(out, "w") as f:
        f.write("// cost_model.inc -- alpha (us) and beta (GB/s) of t = alpha + bytes / beta for the\n")
        f.write("// all-reduce kernel, per element type, rank count and order; MR_AUTO takes the argmin.\n")
        f.write(f"// Fitted by collective_reduction_math_gb300/tune_cost_model.py on {dev_name},\n")
        f.write(f"// {datetime.date.today().isoformat()}, from device times of CUDA graphs of calls\n")
        f.write("// (4 KiB to 64 MiB per rank).\n")
        f.write("// {dtype, W, algo, alpha_us, beta_gbs}\n")
        for code, W, acode, alpha, beta in rows:
            f.write(f"{{{code}, {W}, {acode}, {alpha:.3f}, {beta:.1f}}},\n")
    print(f"wrote {out}")


if __name__ == "__main__":
    sys.exit(main())
