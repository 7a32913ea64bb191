"""The allocation-free reduce-scatter with sign compression.

mr_reduce_scatter_sign_ef_noalloc serves callers that cannot allocate device
memory (a plugin given only its tensors, a runtime whose memory belongs to
another allocator, a loop that cannot pay for cudaMalloc's synchronisation):
it keeps its scratch in a fixed array inside the library instead of asking for
a workspace.  Here it is called through the C ABI and must give exactly what
the workspace entry point gives, on two calls in a row (the second continuing
from the error state the first left).  This file is collected last.
"""
import ctypes

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


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


# The last case needs the most partials any call can have (64 ranks x 32
# blocks), which the library's array must hold.
@pytest.mark.parametrize("W,N,op,algo", [(8, 8 * 50000, "avg", "ring"), (5, 5 * 1001, "sum", "tree"),
                                         (64, 1 << 18, "avg", "ring")])
def test_noalloc_matches_workspace_entry_point(mr, W, N, op, algo):
    import torch
    lib = mr.load()
    g = [torch.from_numpy(x).cuda() for x in synth.normal(90 + W, W, N, 1e-3, "fp32")]
    e0 = synth.normal(91 + W, W, N, 1e-4, "fp32")
    err_a = [torch.from_numpy(x).cuda() for x in e0]
    err_b = [torch.from_numpy(x).cuda() for x in e0]
    C = N // W
    out_a = [torch.empty(C, device="cuda") for _ in range(W)]
    out_b = [torch.empty(C, device="cuda") for _ in range(W)]
    s_a = torch.empty(W, device="cuda")
    s_b = torch.empty(W, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        mr.mr_reduce_scatter_sign_ef(g, err_a, out_a, scales=s_a, op=op, algo=algo)
        st = lib.mr_reduce_scatter_sign_ef_noalloc(_ptrs(g), _ptrs(err_b), _ptrs(out_b), s_b.data_ptr(), W, N,
                                                   mr.OPS[op], mr.ALGOS[algo], stream)
        assert st == 0, mr.mr_last_error()
        torch.cuda.synchronize()
        assert torch.equal(s_a, s_b), f"call {call}: scales differ"
        for k in range(W):
            assert torch.equal(out_a[k], out_b[k]), f"call {call}: shard {k} differs"
            assert torch.equal(err_a[k], err_b[k]), f"call {call}: residual {k} differs"
    # the second call really continued from the first one's residuals
    assert not np.array_equal(err_b[0].cpu().numpy(), e0[0])
