"""The reduce kernel's grid, as the library reports it with MR_DEBUG=1.

The host sizes the grid (plan_tiles): one CTA per tile up to the resident
slots (3 or 2 per SM); a mid-size grid (more than 1.25 CTAs per SM, fewer
than the slots) reserves shared memory so that at most ceil(G / SMs) CTAs
share an SM;
a full grid that is a multiple of more than 8 segments is cut to the largest
grid that shares no factor with the segment count.  Each call here runs in a
child process with MR_DEBUG=1 and its reported grid is checked against those
rules (the outputs themselves are checked by the parity tests)."""
import json
import math
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import torch
import collective_reduction_math_gb300 as mr
mr.load()
for W, N, algo in json.loads(sys.argv[1]):
    xs = [torch.ones(N, device="cuda") for _ in range(W)]
    ys = [torch.empty_like(x) for x in xs]
    mr.mr_allreduce(xs, ys, op="sum", algo=algo)
    torch.cuda.synchronize()
"""

LINE = re.compile(r"W=(\d+) N=(\d+) segments=(\d+) tiles=(\d+) vector=(\d) grid=(\d+) threads=\d+ "
                  r"spread_smem=(\d+) sms=(\d+)")


def reported(calls):
    env = dict(os.environ, MR_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", CHILD, json.dumps(calls)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = [tuple(int(g) for g in m.groups()) for m in LINE.finditer(r.stderr)]
    assert len(out) == len(calls), r.stderr[-2000:]
    return out


def test_small_calls_keep_one_cta_per_tile():
    """Fewer tiles than SMs: one CTA per tile, nothing reserved (a 16-segment
    call of 16 tiles once lost a CTA to the segment rule and doubled its
    latency)."""
    calls = [(16, 16 * 1024, "ring"), (64, 64 * 1024, "ring"), (24, 24 * 1024, "tree"), (8, 8 * 1024, "ring")]
    for W, N, nseg, tiles, vec, grid, spread, sms in reported(calls):
        assert vec == 1
        assert tiles <= sms
        assert grid == tiles, (W, tiles, grid)
        assert spread == 0


def test_mid_size_grids_spread_over_the_sms():
    """More than 1.25 tiles per SM but fewer than the slots: one CTA per tile,
    with enough shared memory reserved that at most ceil(G / SMs) share an
    SM; at 1.05 tiles per SM (160 tiles) nothing is reserved."""
    calls = [(8, 1 << 18, "ring"), (32, 1 << 18, "ring"), (16, 1 << 18, "tree"), (8, 160 * 1024, "ring")]
    for W, N, nseg, tiles, vec, grid, spread, sms in reported(calls):
        assert sms < tiles < 3 * sms, (W, tiles, sms)
        assert grid == tiles
        if 4 * grid <= 5 * sms:
            assert spread == 0, (W, grid, spread)
            continue
        cap = -(-grid // sms)
        assert spread > 0
        assert (cap + 1) * (spread + 1024) > 228 * 1024 >= cap * (spread + 1024), (W, cap, spread)


def test_full_grid_not_a_multiple_of_many_segments():
    """A full grid: 3 CTAs per SM; above 8 segments never a multiple of the
    segment count (the largest smaller grid coprime to it); up to 8 segments
    left as it is."""
    calls = [(8, 1 << 24, "ring"), (19, 19 << 18, "ring"), (24, 24 << 18, "ring"), (57, 57 << 16, "ring"),
             (20, 20 << 18, "ring")]
    for W, N, nseg, tiles, vec, grid, spread, sms in reported(calls):
        full = 3 * sms
        assert tiles >= full, (W, tiles)
        assert spread == 0
        if nseg <= 8 or full % nseg != 0:
            assert grid == full, (W, nseg, grid)
        else:
            assert grid < full and math.gcd(grid, nseg) == 1, (W, nseg, grid)
            assert all(math.gcd(g, nseg) != 1 for g in range(grid + 1, full + 1))
