"""The C-ABI boundary on the host: the library loads, exports every symbol
include/mr.h declares, exposes the planner's orders, and rejects bad
arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from golden_io import read_tree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible():
    import torch
    return torch.cuda.is_available() or os.path.exists("/dev/nvidia0")


# These tests hand the library fake device addresses that must never be
# dereferenced; they run only where no GPU exists, so a regression in argument
# checking can never turn into a launch on bogus memory.
pytestmark = pytest.mark.skipif(_gpu_visible(), reason="host-only checks with fake device addresses")


@pytest.fixture(scope="module")
def mr():
    import __graft_entry__
    __graft_entry__.build()
    import collective_reduction_math_gb300 as m
    m.load()
    return m


def _declared_functions():
    names = set()
    include = os.path.join(ROOT, "include")
    for fn in os.listdir(include):
        if fn.endswith(".h"):
            text = open(os.path.join(include, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(mr_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(mr):
    names = _declared_functions()
    assert {"mr_allreduce", "mr_reduce_scatter", "mr_all_gather", "mr_status_string", "mr_last_error"} <= set(names)
    lib = ctypes.CDLL(mr.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(mr):
    assert mr.mr_status_string(0) == "MR_OK"
    assert mr.mr_status_string(3) == "MR_ERR_ALIAS"
    assert mr.mr_status_string(4) == "MR_ERR_CUDA"


def test_ring_order(mr, oracle_mod):
    for W in (1, 2, 3, 8, 16, 64):
        for k in range(W):
            assert mr.mr_plan_ring_order(W, k) == oracle_mod.ring_order(W, k)
    assert mr.mr_plan_ring_order(4, 0) == [1, 2, 3, 0]


def test_tree_matches_diagram_and_oracle(mr, oracle_mod):
    parent, kids = read_tree("tree14.txt")
    root, p, c = mr.mr_plan_tree(14, 1)
    assert (root, p, c) == (0, parent, kids)
    for W in range(1, 65):
        for which in (1, 2):
            assert mr.mr_plan_tree(W, which) == oracle_mod.tree(W, which), (W, which)


def test_chunk_lo(mr):
    for W in (1, 3, 8, 64):
        for N in (0, 5, 4096, 2**40 + 7):
            assert [mr.mr_chunk_lo(W, N, k) for k in range(W + 1)] == [(k * N) // W for k in range(W + 1)]


def _arr(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def _call_ar(lib, send, recv, W, N, dtype=0, op=0, algo=0):
    return lib.mr_allreduce(_arr(send), _arr(recv), W, N, dtype, op, algo, None)


def test_argument_errors(mr):
    lib = mr.load()
    base = 1 << 40                      # never dereferenced: every call below fails validation
    send = [base + r * (1 << 20) for r in range(4)]
    recv = [base + (1 << 30) + r * (1 << 20) for r in range(4)]
    assert _call_ar(lib, send, recv, 0, 16) == 1
    assert _call_ar(lib, send, recv, 65, 16) == 1
    assert _call_ar(lib, send, recv, 4, 16, dtype=3) == 1
    assert _call_ar(lib, send, recv, 4, 16, op=5) == 1
    assert _call_ar(lib, send, recv, 4, 16, algo=4) == 1
    assert "algo" in mr.mr_last_error()
    assert _call_ar(lib, send, recv, 4, 16, algo=2) == 1          # MR_HIER needs the _ex call
    assert "group" in mr.mr_last_error()
    assert _call_ar(lib, send[:3] + [0], recv, 4, 16) == 1
    assert "send[3]" in mr.mr_last_error()
    assert _call_ar(lib, send, recv[:2] + [recv[2] + 2] + recv[3:], 4, 16) == 1     # misaligned fp32
    assert _call_ar(lib, send, recv[:2] + [recv[2] + 1] + recv[3:], 4, 16, dtype=1) == 1  # misaligned bf16
    assert lib.mr_allreduce(None, _arr(recv), 4, 16, 0, 0, 0, None) == 1
    # N == 0 is a no-op that needs no GPU
    assert _call_ar(lib, send, recv, 4, 0) == 0
    # reduce-scatter / all-gather need N % W == 0
    assert lib.mr_reduce_scatter(_arr(send), _arr(recv), 4, 18, 0, 0, 0, None) == 1
    assert lib.mr_all_gather(_arr(send), _arr(recv), 4, 18, 0, None) == 1
    assert "divisible" in mr.mr_last_error()


def test_alias_rules(mr):
    lib = mr.load()
    W, N, b = 4, 1024, 4
    base = 1 << 40
    send = [base + r * N * b for r in range(W)]           # contiguous, disjoint
    other = [base + (1 << 30) + r * N * b for r in range(W)]
    # all-reduce: recv[r] == send[r] is allowed (it then needs a GPU: not run here)
    # any other overlap is refused
    shifted = [s + 64 for s in send]
    assert _call_ar(lib, send, shifted, W, N) == 3
    assert _call_ar(lib, send, [other[0]] * W, W, N) == 3              # outputs overlap each other
    assert _call_ar(lib, send, [other[0], send[0]] + other[2:], W, N) == 3   # rank 1 writes rank 0's input
    assert _call_ar(lib, [send[0], send[0]] + send[2:], other, W, N) == 3  # inputs overlap
    # reduce-scatter: recv[r] == send[r] + r*C is the in-place form; recv[r] == send[r] is not
    C = N // W
    assert lib.mr_reduce_scatter(_arr(send), _arr(send), W, N, 0, 0, 0, None) == 3
    # all-gather: send[r] == recv[r] + r*C is the in-place form; send[r] == recv[r] for r > 0 is not
    assert lib.mr_all_gather(_arr(send), _arr(send), W, N, 0, None) == 3
    assert "overlaps" in mr.mr_last_error()
    _ = C


def test_valid_call_without_gpu_reports_cuda_error(mr):
    """With no usable GPU the launch itself fails: the call returns MR_ERR_CUDA
    with the runtime's message instead of falling back to anything."""
    lib = mr.load()
    base = 1 << 40
    send = [base + r * 4096 for r in range(2)]
    recv = [base + (1 << 30) + r * 4096 for r in range(2)]
    assert _call_ar(lib, send, recv, 2, 1024) == 4
    assert "launch failed" in mr.mr_last_error()


def _sign_rs(lib, name, grad, err, recv, W, N, op=4, algo=0, workspace=None, ws_bytes=0):
    args = [_arr(grad) if grad else None, _arr(err) if err else None, _arr(recv) if recv else None, None, W, N, op, algo]
    if name == "mr_reduce_scatter_sign_ef":
        args += [workspace, ws_bytes]
    return getattr(lib, name)(*args, None)


def test_sign_workspace_is_bounded(mr):
    """At most 2048 partials of 11 words per call, whatever W and N: 90112
    bytes, which the allocation-free entry point's 96 KiB array holds."""
    lib = mr.load()
    lib.mr_sign_ef_workspace_bytes.restype = ctypes.c_size_t
    lib.mr_sign_ef_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_size_t]
    worst = 0
    for W in range(1, 65):
        for N in (1, 8191, 8192, 8193, 1 << 20, 1 << 24, 1 << 36):
            b = lib.mr_sign_ef_workspace_bytes(W, N)
            assert b % 44 == 0 and b >= 44 * W
            worst = max(worst, b)
    assert worst == 2048 * 44 <= 96 * 1024
    assert lib.mr_sign_ef_workspace_bytes(0, 100) == 0


def test_sign_entry_points_check_arguments_alike(mr):
    """The allocation-free entry point checks its arguments exactly as the
    workspace one does, before anything touches the GPU: the same status for
    every bad call (a NULL array or pointer, an unsupported op, N not divisible
    by W, W out of range, N past 2^37), and nothing to do for N == 0."""
    lib = mr.load()
    base = 1 << 40
    W, N = 4, 4096
    g = [base + r * (1 << 20) for r in range(W)]
    e = [base + (1 << 30) + r * (1 << 20) for r in range(W)]
    o = [base + (1 << 31) + r * (1 << 20) for r in range(W)]
    ws = base + (1 << 32)
    cases = [
        dict(grad=None, err=e, recv=o, W=W, N=N),
        dict(grad=g, err=None, recv=o, W=W, N=N),
        dict(grad=g, err=e[:3] + [0], recv=o, W=W, N=N),
        dict(grad=g, err=e, recv=o, W=W, N=N, op=3),
        dict(grad=g, err=e, recv=o, W=W, N=N, algo=7),
        dict(grad=g, err=e, recv=o, W=W, N=N + 2),
        dict(grad=g, err=e, recv=o, W=0, N=N),
        dict(grad=g, err=e, recv=o, W=W, N=1 << 37),
        dict(grad=g, err=[g[0]] + e[1:], recv=o, W=W, N=N),
    ]
    for c in cases:
        a = _sign_rs(lib, "mr_reduce_scatter_sign_ef", workspace=ws, ws_bytes=1 << 20, **c)
        b = _sign_rs(lib, "mr_reduce_scatter_sign_ef_noalloc", **c)
        assert a == b != 0, c
    assert _sign_rs(lib, "mr_reduce_scatter_sign_ef_noalloc", g, e, o, W, 0) == 0
    # a valid call reaches the scratch lookup, which needs a GPU
    assert _sign_rs(lib, "mr_reduce_scatter_sign_ef_noalloc", g, e, o, W, N) == 4
    assert "static scratch" in mr.mr_last_error()


def test_launch_floor_arguments(mr):
    lib = mr.load()
    assert lib.mr_launch_floor(0, None) == 1
    assert lib.mr_launch_floor(65536, None) == 1
    assert "ctas" in mr.mr_last_error()
    assert lib.mr_launch_floor(1, None) == 4        # no GPU here: the launch itself fails
    assert "launch failed" in mr.mr_last_error()


def _cost_table():
    """(latency bound, L2 bytes, rows) of the table the library is built with;
    a row is (dtype, W, algo, [(alpha, beta) x 3])."""
    rows, bounds = [], {}
    path = os.path.join(ROOT, "collective_reduction_math_gb300", "csrc", "cost_model.inc")
    for line in open(path):
        line = line.strip()
        if line.startswith("constexpr double"):
            name, val = line[len("constexpr double"):].split("=")
            bounds[name.strip()] = float(val.strip(" ;"))
        if line.startswith("{") and not line.startswith("{dtype"):
            nums = [float(x) for x in re.findall(r"-?\d+(?:\.\d+)?", line)]
            rows.append((int(nums[0]), int(nums[1]), int(nums[2]),
                         [(nums[3 + 2 * i], nums[4 + 2 * i]) for i in range(3)]))
    return bounds["kCostModelLatencyBytes"], bounds["kCostModelL2Bytes"], rows


def test_auto_is_the_cost_model_argmin(mr):
    """MR_AUTO picks, per call, the order with the smaller alpha + bytes/beta
    of the table the library was built with, taking the (alpha, beta) of the
    range the call's buffers fall in: latency-bound, within L2, beyond L2
    (recomputed here from the table)."""
    lat, l2, rows = _cost_table()
    assert 0 < lat < l2
    assert len(rows) == 3 * 6 * 2
    codes = {"fp32": 0, "bf16": 1, "int32": 2}
    sizes = {"fp32": 4, "bf16": 2, "int32": 4}
    for dtype in codes:
        for W in (1, 2, 3, 8, 13, 16, 33, 64):
            for N in (1 << 10, 1 << 14, 1 << 16, 1 << 20, 1 << 22, 1 << 24, 1 << 27):
                for rs in (False, True):
                    b = sizes[dtype] * N * ((W + 1) if rs else 2 * W)
                    t = {}
                    for a in (0, 1):
                        cand = [r for r in rows if r[0] == codes[dtype] and r[2] == a]
                        cover = [r for r in cand if r[1] >= W]
                        row = min(cover, key=lambda r: r[1]) if cover else max(cand, key=lambda r: r[1])
                        alpha, beta = row[3][0 if b <= lat else 1 if b <= l2 else 2]
                        t[a] = alpha + b / (beta * 1e3)
                    want = "tree" if t[1] < t[0] else "ring"
                    algo, pred = mr.mr_plan_auto(W, N, dtype, rs)
                    assert algo == want, (dtype, W, N, rs)
                    assert abs(pred - min(t.values())) <= 1e-9 * max(1.0, pred)
