"""bench.py's host logic on the CPU: the one-allocation buffer layout, the
uploads, the per-workload buffer sets and their algorithmic byte counts."""
import argparse
import sys

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = argv
    return b


class FakeLibrary:
    """Stands in for the binding where Step only binds calls."""

    def mr_sign_ef_workspace_bytes(self, W, N):
        return 8 * W * 256

    def __getattr__(self, name):
        return lambda *a, **k: None


def test_carve_one_allocation_aligned(bench):
    import torch
    specs = [(3, torch.float32), (5, torch.bfloat16), (7, torch.int32), (1, torch.float32)]
    bufs = bench.carve(torch, torch.device("cpu"), specs)
    base = bufs[0].untyped_storage().data_ptr()
    for t, (n, dt) in zip(bufs, specs):
        assert t.untyped_storage().data_ptr() == base            # one allocation
        assert t.numel() == n and t.dtype == dt and t.is_contiguous()
        assert (t.data_ptr() - base) % 256 == 0                  # each on a 256-byte boundary
    ends = sorted((t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()) for t in bufs)
    assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:]))     # disjoint


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int32"])
def test_upload_copies_the_bits(bench, dtype):
    import torch
    host = synth.random_values(3, 4, 1000, dtype)
    ins, extra = bench.upload(torch, torch.device("cpu"), host, dtype, [17, 5])
    for t, h in zip(ins, host):
        got = t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()
        assert got.tobytes() == np.ascontiguousarray(h).tobytes()
    assert [t.numel() for t in extra] == [17, 5]


CASES = [("small_int_fp32_w2", None, None, lambda W, N, b: 2 * W * N * b),
         ("fsdp_bf16_w8", None, 8 * 1024, lambda W, N, b: (W + 1) * N * b),
         ("fsdp_bf16_w8", "all_gather", 8 * 1024, lambda W, N, b: (1 + W) * N * b),
         ("int_counts_w16", None, 16 * 64, lambda W, N, b: 2 * W * N * b),
         ("sign_ef_fp32_w8", None, 8 * 1000, lambda W, N, b: 5 * W * N * b + N * b),
         ("sign_ef_fp32_w8", "allreduce_sign_ef", 8 * 1000, lambda W, N, b: 5 * W * N * b + W * N * b),
         ("tp_decode_rmsnorm_bf16_w8", None, None, lambda W, N, b: (2 * W + 2) * N * b + 8192 * b),
         ("tp_decode_rmsnorm_bf16_w8", "allreduce_then_rmsnorm", None,
          lambda W, N, b: (2 * W + 2) * N * b + 8192 * b)]


@pytest.mark.parametrize("workload,collective,n,bytes_of", CASES)
def test_step_buffers_and_bytes(bench, workload, collective, n, bytes_of):
    import torch
    args = argparse.Namespace(workload=workload, collective=collective, op=None, algo="ring", group=None,
                              per_hop=False, n=n)
    S = bench.Step(args, FakeLibrary(), torch, torch.device("cpu"))
    b = 2 if S.dtype == "bf16" else 4
    assert S.bytes == bytes_of(S.W, S.N, b)
    # every buffer of a step sits in one allocation
    stores = {t.untyped_storage().data_ptr() for t in S.e2e_in + S.e2e_out}
    assert len(stores) == 1
    # the second buffer set for pipelined e2e steps: fresh memory, same aliasing
    ins, outs, _ = S.make_set(torch)
    alias_a = [[o is i for i in S.e2e_in] for o in S.e2e_out]
    alias_b = [[o is i for i in ins] for o in outs]
    assert alias_a == alias_b
    old = {t.data_ptr() for t in S.e2e_in + S.e2e_out}
    assert not any(t.data_ptr() in old for t in ins + outs)
    assert [t.numel() for t in ins] == [t.numel() for t in S.e2e_in]
    assert [t.numel() for t in outs] == [t.numel() for t in S.e2e_out]


@pytest.mark.parametrize("ranks,dtype", [(10, None), (12, "bf16"), (3, "fp32")])
def test_rank_and_dtype_overrides(bench, ranks, dtype):
    import torch
    args = argparse.Namespace(workload="sweep_fp32_w8", collective=None, op=None, algo="tree", group=None,
                              per_hop=False, n=4096, ranks=ranks, dtype=dtype)
    S = bench.Step(args, FakeLibrary(), torch, torch.device("cpu"))
    assert S.W == ranks and len(S.xs) == ranks and S.dtype == (dtype or "fp32")
    assert S.bytes == 2 * ranks * 4096 * (2 if dtype == "bf16" else 4)
    cfg = S.config("one call per step")
    assert cfg["W"] == ranks and cfg["algo"] == "tree"
    with pytest.raises(ValueError):
        synth.workload_inputs("sweep_fp32_w8", N=16, dtype="int32")     # a float workload has no int32 form


def test_both_arms_report_the_same_config(bench):
    """The reference arm's config is the GPU arm's for the headline workload,
    key for key (N_timed tells a sampled run apart)."""
    import torch
    args = argparse.Namespace(workload=bench.WORKLOAD, collective=None, op=None, algo="ring", group=None,
                              per_hop=False, n=8 * 1024)
    S = bench.Step(args, FakeLibrary(), torch, torch.device("cpu"))
    gpu = S.config("one call per step")
    W, N = S.W, S.N
    ref = bench.config_dict(bench.WORKLOAD, "allreduce", W, N, "fp32", "avg", "ring", None, False, 2 * W * N * 4,
                            gpu["l2"], N, "one call per step")
    assert gpu == ref
