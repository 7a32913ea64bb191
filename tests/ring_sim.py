"""A literal, step-by-step simulation of the ring all-reduce schedule, used to
pin the oracle's closed-form ring order.

It follows the kernel skeleton printed in "The ring, exactly as the kernel runs
it" (post on NCCL all-reduce): each rank holds its own buffer; messages move
only from rank r to rank r+1; step 0 sends, then W-2 receive-reduce-send
steps, one receive-reduce-copy-send step that completes a chunk and applies the
postOp, W-2 receive-copy-send steps and a final receive.  Arithmetic is numpy
fp32 / wrapping int32 on whole chunks; bf16 rounding goes through torch.
"""
import numpy as np


def _widen(dtype, a):
    if dtype == "bf16" and a.dtype == np.uint16:     # raw bf16 bits; fp32 values pass through
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.copy()


def _post(dtype, op, W, acc):
    if dtype == "bf16":
        import torch
        return torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "int32" and op == "avg":
        wide = acc.astype(np.int64)
        q = np.abs(wide) // W
        return np.where(wide < 0, -q, q).astype(np.int32)
    return acc


def _to_bf16_and_back(x):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float()
    return t.numpy()


def _combine(dtype, op, received, own, hop=False):
    if op in ("sum", "avg"):
        r = received + own             # numpy: fp32 rounded add / int32 wrap
    elif op == "prod":
        r = received * own
    else:
        raise ValueError("the simulator covers the order-dependent ops only")
    if hop and dtype == "bf16":        # the partial crosses the wire as bf16
        r = _to_bf16_and_back(r)
    return r


def simulate(dtype, op, inputs, hop=False, raw=False):
    """hop: round a bf16 running total to bf16 after every add (and the
    pre-scaled contributions of avg).  raw: skip the postOp and return fp32
    running totals (used to chain simulations)."""
    """Returns (per-rank result buffers, number of link transfers, and for
    each chunk the rank on which its total completed)."""
    W, N = len(inputs), inputs[0].size
    with np.errstate(over="ignore"):
        y = [_widen(dtype, a) for a in inputs]
        if op == "avg" and dtype != "int32":
            s = np.float32(1.0 / W)
            y = [v * s for v in y]
            if hop and dtype == "bf16":
                y = [_to_bf16_and_back(v) for v in y]
        bounds = [(k * N) // W for k in range(W + 1)]
        chunk = [slice(bounds[k], bounds[k + 1]) for k in range(W)]
        post = (lambda a: a) if raw else (lambda a: _post(dtype, op, W, a))
        out_dtype = y[0].dtype if raw else inputs[0].dtype
        result = [np.empty(N, out_dtype) for _ in range(W)]
        if W == 1:
            result[0][:] = post(y[0])
            return result, 0, [0]

        transfers = 0
        inbox = [None] * W
        finisher = [None] * W

        def deliver(outgoing):
            nonlocal transfers
            for r in range(W):
                inbox[(r + 1) % W] = outgoing[r]
            transfers += 1

        # step 0: each rank pushes its own part of chunk r-1 to rank r+1
        deliver([((r - 1) % W, y[r][chunk[(r - 1) % W]].copy()) for r in range(W)])
        # W-2 steps: receive a partial sum, add mine, forward
        for _ in range(W - 2):
            outgoing = []
            for r in range(W):
                c, data = inbox[r]
                outgoing.append((c, _combine(dtype, op, data, y[r][chunk[c]], hop)))
            deliver(outgoing)
        # the arriving chunk completes here: postOp, keep, forward
        outgoing = []
        for r in range(W):
            c, data = inbox[r]
            fin = post(_combine(dtype, op, data, y[r][chunk[c]], hop))
            result[r][chunk[c]] = fin
            finisher[c] = r
            outgoing.append((c, fin))
        deliver(outgoing)
        # W-2 steps: receive a finished chunk, keep it, forward it
        for _ in range(W - 2):
            outgoing = []
            for r in range(W):
                c, data = inbox[r]
                result[r][chunk[c]] = data
                outgoing.append((c, data))
            deliver(outgoing)
        # last step: receive the final chunk
        for r in range(W):
            c, data = inbox[r]
            result[r][chunk[c]] = data
    return result, transfers, finisher
