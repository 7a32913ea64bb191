"""Buffers of more than 2^31 elements per rank (byte offsets past 4 GiB),
checked on sampled outputs, each recomputed by the oracle from the W input
values at that position: the first and last elements, both sides of every
chunk and tree boundary, and random positions."""
import numpy as np
import pytest

import synth

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


def _positions(N, W, extra=()):
    rng = np.random.default_rng(5)
    pts = set(range(0, 64)) | set(range(N - 64, N))
    for k in range(W + 1):
        lo = (k * N) // W
        pts |= {p for p in range(lo - 8, lo + 8) if 0 <= p < N}
    for b in extra:
        pts |= {p for p in range(b - 8, b + 8) if 0 <= p < N}
    pts |= set(rng.integers(0, N, size=1500).tolist())
    return np.array(sorted(pts), dtype=np.int64)


def _raw(t, idx, dtype):
    import torch
    v = t[torch.from_numpy(idx).to(t.device)]
    return v.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else v.cpu().numpy()


@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_allreduce_past_2_31_elements(mr, algo):
    import oracle
    import torch
    W, N, dtype = 2, (1 << 31) + 9, "bf16"
    xs = synth.device_normal(11, W, N, dtype)
    ys = [torch.empty_like(x) for x in xs]
    mr.mr_allreduce(xs, ys, op="avg", algo=algo)
    torch.cuda.synchronize()
    idx = _positions(N, W, extra=(N // 2,))
    vals = [_raw(x, idx, dtype) for x in xs]
    outs = [_raw(y, idx, dtype) for y in ys]
    for n, e in enumerate(idx.tolist()):
        want = oracle.reduce_one(dtype, "avg", algo, N, e, np.array([v[n] for v in vals], np.uint16))
        for j in range(W):
            assert outs[j][n] == want, (algo, e, j)
    del xs, ys
    torch.cuda.empty_cache()


def test_reduce_scatter_and_all_gather_past_2_31_elements(mr):
    import oracle
    import torch
    W, C, dtype = 4, (1 << 29) + 3, "fp32"
    N = W * C                                   # 2^31 + 12 elements per rank
    xs = synth.device_normal(12, W, N, dtype)
    shards = [torch.empty(C, device="cuda") for _ in range(W)]
    mr.mr_reduce_scatter(xs, shards, op="sum", algo="ring")
    torch.cuda.synchronize()
    idx = _positions(N, W)
    vals = [_raw(x, idx, dtype) for x in xs]
    for n, e in enumerate(idx.tolist()):
        k = e // C
        got = shards[k][e - k * C].item()
        want = oracle.reduce_one(dtype, "sum", "ring", N, e, np.array([v[n] for v in vals], np.float32))
        assert np.float32(got).tobytes() == np.float32(want).tobytes(), e
    del xs
    torch.cuda.empty_cache()
    full = [torch.empty(N, device="cuda") for _ in range(W)]
    mr.mr_all_gather(shards, full)
    torch.cuda.synchronize()
    for j in range(W):
        got = _raw(full[j], idx, dtype)
        want = np.array([shards[e // C][e - (e // C) * C].item() for e in idx.tolist()], np.float32)
        assert got.tobytes() == want.tobytes(), j
