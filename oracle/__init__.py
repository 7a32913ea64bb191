"""CPU oracle for the collective reduction math.  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it, and
the two share no code: the oracle is plain single-threaded C (``oracle.c``)
compiled with gcc and reached through ctypes.

Buffers are numpy arrays: fp32 as ``float32``, bf16 as ``uint16`` bit
patterns, int32 as ``int32``.

What each routine follows (page title and section):
  * ``allreduce`` / ``reduce_scatter`` / ``all_gather``: "What all-reduce
    promises" and "The ring, exactly as the kernel runs it" (post on NCCL
    all-reduce); "All-gather: everyone shows their piece" and "Why backward
    needs a different collective" (FSDP collectives 101).
  * ``ring_order``: "The ring, exactly as the kernel runs it".
  * ``tree``: "The double binary tree".
  * ``chunk_lo``: Eq. (2), "Local shard bounds" (NCCL M2N).
  * ``bf16_rne``: the single bf16 rounding of an fp32 accumulator.
  * ``sign_ef_scales`` / ``sign_ef_collective``: "Communication Optimization:
    Gradient Compression, NCCL ..." -- 1-bit SGD (sign times ||g||_1 / d) with
    the error feedback of its top-K section.
  * ``allreduce_rmsnorm``: "How this survives ten thousand GPUs" (post on NCCL
    all-reduce): in decoding, the merge (residual add) and the RMSNorm that
    follow the all-reduce are fused into it.

Parity unpinned: NaN and infinity payloads through min/max and bf16 rounding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

DTYPES = {"fp32": 0, "bf16": 1, "int32": 2}
OPS = {"sum": 0, "prod": 1, "min": 2, "max": 3, "avg": 4}
ALGOS = {"ring": 0, "tree": 1, "hier": 2}
NP_DTYPE = {"fp32": np.float32, "bf16": np.uint16, "int32": np.int32}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.or_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        L.or_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.or_f32_to_bf16_rne_array.argtypes = [vp, vp, sz]
        L.or_f32_to_bf16_rne_array.restype = None
        L.or_chunk_lo.argtypes = [i, sz, i]
        L.or_chunk_lo.restype = sz
        L.or_ring_order.argtypes = [i, i, vp]
        L.or_ring_order.restype = None
        L.or_tree_build.argtypes = [i, i, vp, vp]
        L.or_tree_build.restype = i
        L.or_allreduce.argtypes = [i, i, i, i, sz, vp, vp]
        L.or_allreduce.restype = i
        L.or_reduce_scatter.argtypes = [i, i, i, i, sz, vp, vp]
        L.or_reduce_scatter.restype = i
        L.or_all_gather.argtypes = [i, i, sz, vp, vp]
        L.or_all_gather.restype = i
        L.or_reduce_one.argtypes = [i, i, i, i, sz, sz, vp, vp]
        L.or_reduce_one.restype = i
        _lib = L
    return _lib


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return arr


def _check_inputs(dtype, arrays, n):
    want = NP_DTYPE[dtype]
    for a in arrays:
        if a.dtype != want or not a.flags.c_contiguous or a.size != n:
            raise ValueError(f"oracle input must be contiguous {want.__name__}[{n}]")


def allreduce(dtype: str, op: str, algo: str, inputs, all_ranks: bool = False):
    """All-reduce of W rank buffers.  Returns one copy of the (identical)
    result, or with ``all_ranks`` the list of every rank's output buffer."""
    W, N = len(inputs), inputs[0].size
    _check_inputs(dtype, inputs, N)
    copies = W if all_ranks else 1
    outs = [np.empty(N, NP_DTYPE[dtype]) for _ in range(copies)]
    out_ptrs = [outs[j % copies] for j in range(W)]
    rc = lib().or_allreduce(DTYPES[dtype], OPS[op], ALGOS[algo], W, N, _ptrs(inputs), _ptrs(out_ptrs))
    if rc != 0:
        raise ValueError("oracle allreduce rejected its arguments")
    return outs if all_ranks else outs[0]


def reduce_scatter(dtype: str, op: str, algo: str, inputs):
    """Reduce-scatter: returns W shards; shard k is chunk k of the result."""
    W, N = len(inputs), inputs[0].size
    _check_inputs(dtype, inputs, N)
    if N % W:
        raise ValueError("reduce-scatter needs N divisible by W")
    outs = [np.empty(N // W, NP_DTYPE[dtype]) for _ in range(W)]
    rc = lib().or_reduce_scatter(DTYPES[dtype], OPS[op], ALGOS[algo], W, N, _ptrs(inputs), _ptrs(outs))
    if rc != 0:
        raise ValueError("oracle reduce_scatter rejected its arguments")
    return outs


def all_gather(dtype: str, shards, all_ranks: bool = False):
    """All-gather of W shards: one copy of the full buffer, or every rank's."""
    W, C = len(shards), shards[0].size
    _check_inputs(dtype, shards, C)
    copies = W if all_ranks else 1
    outs = [np.empty(C * W, NP_DTYPE[dtype]) for _ in range(copies)]
    out_ptrs = [outs[j % copies] for j in range(W)]
    rc = lib().or_all_gather(DTYPES[dtype], W, C * W, _ptrs(shards), _ptrs(out_ptrs))
    if rc != 0:
        raise ValueError("oracle all_gather rejected its arguments")
    return outs if all_ranks else outs[0]


def reduce_one(dtype: str, op: str, algo: str, N: int, e: int, y):
    """Result at element e of an N-element all-reduce, from the W values y[r]."""
    y = np.ascontiguousarray(y, dtype=NP_DTYPE[dtype])
    res = np.empty(1, NP_DTYPE[dtype])
    rc = lib().or_reduce_one(DTYPES[dtype], OPS[op], ALGOS[algo], y.size, N, e,
                             y.ctypes.data, res.ctypes.data)
    if rc != 0:
        raise ValueError("oracle reduce_one rejected its arguments")
    return res[0]


def ring_order(W: int, k: int):
    out = np.empty(W, np.int32)
    lib().or_ring_order(W, k, out.ctypes.data)
    return out.tolist()


def tree(W: int, which: int):
    """Returns (root, parent[W], children[W] as lists)."""
    parent = np.empty(W, np.int32)
    child = np.empty(2 * W, np.int32)
    root = lib().or_tree_build(W, which, parent.ctypes.data, child.ctypes.data)
    if root < 0:
        raise ValueError("bad W")
    kids = [[c for c in child[2 * r:2 * r + 2].tolist() if c >= 0] for r in range(W)]
    return root, parent.tolist(), kids


def chunk_lo(W: int, N: int, k: int) -> int:
    return int(lib().or_chunk_lo(W, N, k))


def bf16_rne(bits_u32) -> np.ndarray:
    """Round fp32 bit patterns (uint32 array) to bf16 patterns (uint16)."""
    a = np.ascontiguousarray(bits_u32, dtype=np.uint32)
    out = np.empty(a.size, np.uint16)
    lib().or_f32_to_bf16_rne_array(a.ctypes.data, out.ctypes.data, a.size)
    return out


def allreduce_rmsnorm(dtype: str, algo: str, inputs, rows: int, hidden: int, weight, residual=None,
                      eps: float = 1e-6, want_residual_out: bool = True):
    """All-reduce sum of W buffers of rows*hidden elements, residual add, then
    RMSNorm of every row scaled by ``weight``.  Returns (out, residual_out or
    None); every rank's output is the same, so one copy is returned."""
    W, N = len(inputs), inputs[0].size
    if N != rows * hidden:
        raise ValueError("inputs must hold rows*hidden elements")
    _check_inputs(dtype, inputs, N)
    L = lib()
    if not hasattr(L, "_rms_typed"):
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.or_allreduce_rmsnorm.argtypes = [i, i, i, sz, sz, vp, vp, vp, ctypes.c_double, vp, vp]
        L.or_allreduce_rmsnorm.restype = i
        L._rms_typed = True
    out = np.empty(N, NP_DTYPE[dtype])
    res_out = np.empty(N, NP_DTYPE[dtype]) if want_residual_out else None
    w = np.ascontiguousarray(weight, dtype=NP_DTYPE[dtype])
    r = None if residual is None else np.ascontiguousarray(residual, dtype=NP_DTYPE[dtype])
    rc = L.or_allreduce_rmsnorm(DTYPES[dtype], ALGOS[algo], W, rows, hidden, _ptrs(inputs),
                                None if r is None else r.ctypes.data, w.ctypes.data, eps,
                                _ptrs([out] * W), None if res_out is None else res_out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle allreduce_rmsnorm rejected its arguments")
    return out, res_out


def sign_ef_scales(grads, errs):
    """s_r = ||g_r + e_r||_1 / N for every rank: the exact sum of the fp32
    magnitudes over the exact N, rounded once to the nearest fp32."""
    W, N = len(grads), grads[0].size
    _check_inputs("fp32", grads, N)
    _check_inputs("fp32", errs, N)
    L = lib()
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.or_sign_ef_scales.argtypes = [i, sz, vp, vp, vp]
    L.or_sign_ef_scales.restype = i
    out = np.empty(W, np.float32)
    if L.or_sign_ef_scales(W, N, _ptrs(grads), _ptrs(errs), out.ctypes.data) != 0:
        raise ValueError("oracle sign_ef_scales rejected its arguments")
    return out


def sign_ef_collective(mode: str, op: str, algo: str, grads, errs, scales):
    """Decode sign(g + e) * s_r, reduce (sum / avg), update the errors.
    mode 'allreduce' or 'reduce_scatter'.  Returns (outputs, new errors); the
    inputs are not modified."""
    W, N = len(grads), grads[0].size
    _check_inputs("fp32", grads, N)
    errs = [np.array(e, dtype=np.float32, copy=True) for e in errs]
    L = lib()
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.or_sign_ef_collective.argtypes = [i, i, i, i, sz, vp, vp, vp, vp]
    L.or_sign_ef_collective.restype = i
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    if mode == "allreduce":
        out = np.empty(N, np.float32)
        outs, m = [out] * W, 0
    else:
        outs, m = [np.empty(N // W, np.float32) for _ in range(W)], 1
    rc = L.or_sign_ef_collective(m, OPS[op], ALGOS[algo], W, N, _ptrs(grads), _ptrs(errs), sc.ctypes.data,
                                 _ptrs(outs))
    if rc != 0:
        raise ValueError("oracle sign_ef_collective rejected its arguments")
    return (outs[0] if m == 0 else outs), errs


def allreduce_ex(dtype: str, op: str, algo: str, inputs, group: int = 0, hop: bool = False,
                 all_ranks: bool = False):
    """All-reduce with a choice of order: algo 'hier' needs ``group`` (ranks
    per group, dividing W); ``hop`` rounds a bf16 running total to bf16 after
    every combine."""
    W, N = len(inputs), inputs[0].size
    _check_inputs(dtype, inputs, N)
    L = lib()
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.or_allreduce_ex.argtypes = [i, i, i, i, i, i, sz, vp, vp]
    L.or_allreduce_ex.restype = i
    copies = W if all_ranks else 1
    outs = [np.empty(N, NP_DTYPE[dtype]) for _ in range(copies)]
    rc = L.or_allreduce_ex(DTYPES[dtype], OPS[op], ALGOS[algo], group, int(hop), W, N, _ptrs(inputs),
                           _ptrs([outs[j % copies] for j in range(W)]))
    if rc != 0:
        raise ValueError("oracle allreduce_ex rejected its arguments")
    return outs if all_ranks else outs[0]


def reduce_scatter_ex(dtype: str, op: str, algo: str, inputs, group: int = 0, hop: bool = False):
    W, N = len(inputs), inputs[0].size
    _check_inputs(dtype, inputs, N)
    L = lib()
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.or_reduce_scatter_ex.argtypes = [i, i, i, i, i, i, sz, vp, vp]
    L.or_reduce_scatter_ex.restype = i
    outs = [np.empty(N // W, NP_DTYPE[dtype]) for _ in range(W)]
    rc = L.or_reduce_scatter_ex(DTYPES[dtype], OPS[op], ALGOS[algo], group, int(hop), W, N, _ptrs(inputs),
                                _ptrs(outs))
    if rc != 0:
        raise ValueError("oracle reduce_scatter_ex rejected its arguments")
    return outs
