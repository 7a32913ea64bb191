"""Helpers for the GPU parity tests: host <-> device copies of raw rank
buffers, and output buffers fenced by canary guard bands."""
import numpy as np

TORCH_DT = {"fp32": "float32", "bf16": "bfloat16", "int32": "int32"}
GUARD = 64              # elements of canary before and after every output
CANARY = {"fp32": np.uint32(0x7FBADBAD), "bf16": np.uint16(0x7FBD), "int32": np.uint32(0xDEADBEEF)}


def torch_dtype(dtype):
    import torch
    return getattr(torch, TORCH_DT[dtype])


def to_device(host, dtype, dev="cuda"):
    """numpy raw buffer (float32 / uint16 bf16 bits / int32) -> CUDA tensor."""
    import torch
    if dtype == "bf16":
        return torch.from_numpy(host.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(host).to(dev)


def to_host(t, dtype):
    """CUDA tensor -> numpy raw buffer in the oracle's representation."""
    import torch
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class Guarded:
    """W output buffers of n elements, each inside a larger allocation whose
    guard bands hold a canary pattern; ``check()`` verifies they are intact."""

    def __init__(self, W, n, dtype, dev="cuda", offset=0):
        import torch
        self.dtype, self.n, self.offset = dtype, n, offset
        bits = torch.int16 if dtype == "bf16" else torch.int32
        can = CANARY[dtype].astype(np.int16 if dtype == "bf16" else np.int32)
        self.raw = [torch.full((n + 2 * GUARD + offset,), int(can), dtype=bits, device=dev) for _ in range(W)]
        tdt = torch_dtype(dtype)
        self.views = [r[GUARD + offset:GUARD + offset + n].view(tdt) for r in self.raw]
        self._can = int(can)

    def check(self):
        for r in self.raw:
            head = r[:GUARD + self.offset]
            tail = r[GUARD + self.offset + self.n:]
            assert bool((head == self._can).all()) and bool((tail == self._can).all()), "guard band overwritten"

    def host(self):
        return [to_host(v, self.dtype) for v in self.views]


def first_mismatch(got, want):
    g = np.frombuffer(got.tobytes(), np.uint8)
    w = np.frombuffer(want.tobytes(), np.uint8)
    if g.size != w.size:
        return f"size {g.size} != {w.size}"
    idx = np.nonzero(g != w)[0]
    if idx.size == 0:
        return None
    e = idx[0] // got.itemsize
    return f"first mismatch at element {e}: got {got[e]!r} want {want[e]!r} ({idx.size} bytes differ)"


def assert_same(got, want, what=""):
    m = first_mismatch(got, want)
    assert m is None, f"{what}: {m}"
