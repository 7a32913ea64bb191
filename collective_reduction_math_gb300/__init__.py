"""Python binding of libmr.so, the C-ABI library of collective reduction math
on one GPU (see include/mr.h for the contract).

Argument marshalling only: every step of every collective runs in the CUDA
kernels of libmr.so.  PyTorch supplies the device memory and the stream.  If
the library has not been built, every call raises instead of computing
anything elsewhere.

    import torch, collective_reduction_math_gb300 as mr
    xs = [torch.randn(1 << 20, device="cuda") for _ in range(8)]
    ys = [torch.empty_like(x) for x in xs]
    mr.mr_allreduce(xs, ys, op="avg", algo="ring")
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "mr_allreduce", "mr_reduce_scatter", "mr_all_gather", "mr_allreduce_ex", "mr_reduce_scatter_ex", "mr_allreduce_rmsnorm", "mr_allreduce_sign_ef",
    "mr_reduce_scatter_sign_ef", "mr_reduce_scatter_sign_ef_noalloc", "mr_sign_ef_workspace_bytes",
    "mr_status_string", "mr_last_error",
    "mr_allreduce_ptrs", "mr_plan_auto", "mr_plan_ring_order", "mr_plan_tree", "mr_chunk_lo", "mr_launch_count", "mr_launch_floor", "MRError",
    "load", "LIB_PATH",
    "DTYPES", "OPS", "ALGOS", "MAX_RANKS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmr.so")
MAX_RANKS = 64
DTYPES = {"fp32": 0, "bf16": 1, "int32": 2}
OPS = {"sum": 0, "prod": 1, "min": 2, "max": 3, "avg": 4}
ALGOS = {"ring": 0, "tree": 1, "hier": 2, "auto": 3}
STATUS = {0: "MR_OK", 1: "MR_ERR_INVALID_ARGUMENT", 2: "MR_ERR_UNSUPPORTED", 3: "MR_ERR_ALIAS", 4: "MR_ERR_CUDA"}

_lib = None


class Order(ctypes.Structure):
    """mr_order_t: accumulation order for mr_allreduce_ex / mr_reduce_scatter_ex."""
    _fields_ = [("algo", ctypes.c_int), ("group", ctypes.c_int), ("per_hop_rounding", ctypes.c_int)]


class MRError(RuntimeError):
    """A non-OK status from the library; ``status`` holds the code."""

    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status


def load():
    """Load libmr.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first "
                           "(there is no fallback: the collectives run only in its CUDA kernels)")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.mr_allreduce.argtypes = [vp, vp, i, sz, i, i, i, vp]
    L.mr_allreduce.restype = i
    L.mr_reduce_scatter.argtypes = [vp, vp, i, sz, i, i, i, vp]
    L.mr_reduce_scatter.restype = i
    L.mr_all_gather.argtypes = [vp, vp, i, sz, i, vp]
    L.mr_all_gather.restype = i
    L.mr_allreduce_rmsnorm.argtypes = [vp, vp, i, sz, sz, vp, vp, vp, ctypes.c_float, i, i, vp]
    L.mr_allreduce_rmsnorm.restype = i
    L.mr_sign_ef_workspace_bytes.argtypes = [i, sz]
    L.mr_sign_ef_workspace_bytes.restype = sz
    for f in (L.mr_allreduce_sign_ef, L.mr_reduce_scatter_sign_ef):
        f.argtypes = [vp, vp, vp, vp, i, sz, i, i, vp, sz, vp]
        f.restype = i
    L.mr_reduce_scatter_sign_ef_noalloc.argtypes = [vp, vp, vp, vp, i, sz, i, i, vp]
    L.mr_reduce_scatter_sign_ef_noalloc.restype = i
    for f in (L.mr_allreduce_ex, L.mr_reduce_scatter_ex):
        f.argtypes = [vp, vp, i, sz, i, i, ctypes.POINTER(Order), vp]
        f.restype = i
    L.mr_status_string.argtypes = [i]
    L.mr_status_string.restype = ctypes.c_char_p
    L.mr_last_error.argtypes = []
    L.mr_last_error.restype = ctypes.c_char_p
    L.mr_plan_ring_order.argtypes = [i, i, vp]
    L.mr_plan_ring_order.restype = i
    L.mr_plan_tree.argtypes = [i, i, vp, vp, vp]
    L.mr_plan_tree.restype = i
    L.mr_chunk_lo.argtypes = [i, sz, i]
    L.mr_chunk_lo.restype = sz
    L.mr_plan_auto.argtypes = [i, sz, i, i, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
    L.mr_plan_auto.restype = i
    L.mr_launch_count.argtypes = []
    L.mr_launch_count.restype = ctypes.c_ulonglong
    L.mr_launch_floor.argtypes = [ctypes.c_uint, vp]
    L.mr_launch_floor.restype = i
    _lib = L
    return L


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: 0, torch.bfloat16: 1, torch.int32: 2}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}: fp32, bf16 or int32")
    return codes[t.dtype]


def _pointers(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(tensors, name):
    if not tensors:
        raise ValueError(f"{name}: empty list of rank buffers")
    d = tensors[0].dtype
    for t in tensors:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != d:
            raise ValueError(f"{name}: rank buffers must be contiguous CUDA tensors of one dtype")


def _raise(status: int):
    L = load()
    raise MRError(status, L.mr_last_error().decode())


def _code(table, key, what):
    if isinstance(key, int):
        return key
    if key not in table:
        raise ValueError(f"unknown {what} {key!r}")
    return table[key]


# --------------------------------------------------------------------------
# the collectives (same names as the C ABI)
# --------------------------------------------------------------------------

def mr_allreduce(send, recv, op="sum", algo="ring", stream=None):
    """All-reduce: every recv[j] receives the reduction of send[0..W-1].
    send, recv: lists of W CUDA tensors of N elements (recv may be send)."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    st = L.mr_allreduce(_pointers(send), _pointers(recv), len(send), send[0].numel(), _dtype_code(send[0]),
                        _code(OPS, op, "op"), _code(ALGOS, algo, "algo"), _stream(stream))
    if st:
        _raise(st)


def mr_reduce_scatter(send, recv, op="sum", algo="ring", stream=None):
    """Reduce-scatter: recv[k] (N/W elements) receives chunk k of the reduction
    of send[0..W-1] (N elements each)."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    st = L.mr_reduce_scatter(_pointers(send), _pointers(recv), len(send), send[0].numel(), _dtype_code(send[0]),
                             _code(OPS, op, "op"), _code(ALGOS, algo, "algo"), _stream(stream))
    if st:
        _raise(st)


def mr_all_gather(send, recv, stream=None):
    """All-gather: every recv[j] (N elements) receives the concatenation of the
    shards send[0..W-1] (N/W elements each)."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    st = L.mr_all_gather(_pointers(send), _pointers(recv), len(send), recv[0].numel(), _dtype_code(recv[0]),
                         _stream(stream))
    if st:
        _raise(st)


def _order(algo, group, per_hop):
    return Order(_code(ALGOS, algo, "algo"), int(group or 0), 1 if per_hop else 0)


def mr_allreduce_ex(send, recv, op="sum", algo="ring", group=None, per_hop=False, stream=None):
    """All-reduce with a choice of order: algo 'hier' folds groups of
    ``group`` consecutive ranks first, then the group totals; ``per_hop``
    rounds a bf16 running total to bf16 after every combine."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    o = _order(algo, group, per_hop)
    st = L.mr_allreduce_ex(_pointers(send), _pointers(recv), len(send), send[0].numel(), _dtype_code(send[0]),
                           _code(OPS, op, "op"), ctypes.byref(o), _stream(stream))
    if st:
        _raise(st)


def mr_reduce_scatter_ex(send, recv, op="sum", algo="ring", group=None, per_hop=False, stream=None):
    """Reduce-scatter with a choice of order (see mr_allreduce_ex)."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    o = _order(algo, group, per_hop)
    st = L.mr_reduce_scatter_ex(_pointers(send), _pointers(recv), len(send), send[0].numel(), _dtype_code(send[0]),
                                _code(OPS, op, "op"), ctypes.byref(o), _stream(stream))
    if st:
        _raise(st)


def mr_allreduce_rmsnorm(send, recv, weight, residual=None, residual_out=None, eps=1e-6, algo="ring",
                         stream=None):
    """All-reduce (sum) of send[0..W-1], residual add, then RMSNorm of every
    row of ``weight.numel()`` elements scaled by ``weight``; every recv[j]
    receives the normalised rows and residual_out (if given) the pre-norm sum
    plus residual."""
    _check(send, "send")
    _check(recv, "recv")
    L = load()
    hidden = weight.numel()
    n = send[0].numel()
    if hidden == 0 or n % hidden:
        raise ValueError("the buffers must hold whole rows of weight.numel() elements")
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    st = L.mr_allreduce_rmsnorm(_pointers(send), _pointers(recv), len(send), n // hidden, hidden, ptr(residual),
                                ptr(residual_out), weight.data_ptr(), float(eps), _dtype_code(send[0]),
                                _code(ALGOS, algo, "algo"), _stream(stream))
    if st:
        _raise(st)


def mr_sign_ef_workspace_bytes(W: int, N: int) -> int:
    return int(load().mr_sign_ef_workspace_bytes(W, N))


def _sign_ef(fn, grad, err, recv, scales, workspace, op, algo, stream):
    import torch
    _check(grad, "grad")
    _check(err, "err")
    _check(recv, "recv")
    for t in grad + err + recv:
        if t.dtype != torch.float32:
            raise TypeError("sign compression takes fp32 buffers")
    W, N = len(grad), grad[0].numel()
    need = mr_sign_ef_workspace_bytes(W, N)
    if workspace is None:        # plumbing: torch provides the device memory
        workspace = torch.empty(need, dtype=torch.uint8, device=grad[0].device)
    st = fn(_pointers(grad), _pointers(err), _pointers(recv), None if scales is None else scales.data_ptr(), W, N,
            _code(OPS, op, "op"), _code(ALGOS, algo, "algo"), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if st:
        _raise(st)


def mr_allreduce_sign_ef(grad, err, recv, scales=None, workspace=None, op="avg", algo="ring", stream=None):
    """1-bit sign compression with error feedback, then all-reduce: every
    recv[j] gets the reduction of sign(grad[r] + err[r]) * s_r; err[r] is
    updated in place; scales (W fp32, optional) receives s_r."""
    _sign_ef(load().mr_allreduce_sign_ef, grad, err, recv, scales, workspace, op, algo, stream)


def mr_reduce_scatter_sign_ef(grad, err, recv, scales=None, workspace=None, op="avg", algo="ring", stream=None):
    """As mr_allreduce_sign_ef, but recv[k] (N/W elements) gets chunk k."""
    _sign_ef(load().mr_reduce_scatter_sign_ef, grad, err, recv, scales, workspace, op, algo, stream)


def mr_reduce_scatter_sign_ef_noalloc(grad, err, recv, scales=None, op="avg", algo="ring", stream=None):
    """mr_reduce_scatter_sign_ef without a workspace argument: the library
    uses its own fixed 64 KiB scratch, for callers that cannot allocate device
    memory.  Concurrent calls race on that scratch."""
    _check(grad, "grad")
    _check(err, "err")
    _check(recv, "recv")
    st = load().mr_reduce_scatter_sign_ef_noalloc(
        _pointers(grad), _pointers(err), _pointers(recv), None if scales is None else scales.data_ptr(), len(grad),
        grad[0].numel(), _code(OPS, op, "op"), _code(ALGOS, algo, "algo"), _stream(stream))
    if st:
        _raise(st)


def mr_allreduce_ptrs(send_ptrs, recv_ptrs, N, dtype, op, algo, stream):
    """The raw form: integer device pointers, as the C ABI takes them.
    Returns the status code instead of raising."""
    L = load()
    s = (ctypes.c_void_p * len(send_ptrs))(*send_ptrs)
    r = (ctypes.c_void_p * len(recv_ptrs))(*recv_ptrs)
    return L.mr_allreduce(s, r, len(send_ptrs), N, _code(DTYPES, dtype, "dtype"), _code(OPS, op, "op"),
                          _code(ALGOS, algo, "algo"), stream)


def mr_status_string(status: int) -> str:
    return load().mr_status_string(status).decode()


def mr_last_error() -> str:
    return load().mr_last_error().decode()


def mr_plan_ring_order(W: int, k: int):
    out = (ctypes.c_int * W)()
    st = load().mr_plan_ring_order(W, k, out)
    if st:
        _raise(st)
    return list(out)


def mr_plan_tree(W: int, which: int):
    """Returns (root, parent[W], children[W])."""
    parent = (ctypes.c_int * W)()
    child = (ctypes.c_int * (2 * W))()
    root = ctypes.c_int()
    st = load().mr_plan_tree(W, which, parent, child, ctypes.byref(root))
    if st:
        _raise(st)
    kids = [[c for c in child[2 * r:2 * r + 2] if c >= 0] for r in range(W)]
    return root.value, list(parent), kids


def mr_plan_auto(W: int, N: int, dtype: str, reduce_scatter: bool = False):
    """The order MR_AUTO picks for a call, and the cost model's time (us)."""
    a = ctypes.c_int()
    t = ctypes.c_double()
    st = load().mr_plan_auto(W, N, _code(DTYPES, dtype, "dtype"), int(reduce_scatter), ctypes.byref(a), ctypes.byref(t))
    if st:
        _raise(st)
    return {0: "ring", 1: "tree"}[a.value], t.value


def mr_chunk_lo(W: int, N: int, k: int) -> int:
    return int(load().mr_chunk_lo(W, N, k))


def mr_launch_count() -> int:
    return int(load().mr_launch_count())


def mr_launch_floor(ctas: int = 1, stream=None):
    """One empty kernel of ``ctas`` CTAs on the stream (the launch floor)."""
    st = load().mr_launch_floor(ctas, _stream(stream))
    if st:
        _raise(st)
