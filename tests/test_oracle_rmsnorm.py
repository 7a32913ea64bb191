"""Pins of the oracle's all-reduce + residual + RMSNorm: the sum is the pinned
all-reduce, the residual add is one fp32 add, and the norm agrees with torch's
own rms_norm evaluated in fp64 (an independent library), with closed forms."""
import numpy as np
import pytest

import synth


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _widen(dtype, a):
    return _f32(a) if dtype == "bf16" else a.astype(np.float32)


def _round(dtype, x64):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64)).float()
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("W,rows,hidden", [(1, 3, 64), (2, 4, 100), (8, 5, 256), (3, 2, 1000)])
def test_against_torch_rms_norm(oracle_mod, dtype, algo, W, rows, hidden):
    import torch
    N = rows * hidden
    x = synth.normal(21, W, N, 0.5, dtype)
    res = synth.normal(22, 1, N, 1.0, dtype)[0]
    w = synth.normal(23, 1, hidden, 1.0, dtype)[0]
    eps = 1e-5
    out, rout = oracle_mod.allreduce_rmsnorm(dtype, algo, x, rows, hidden, w, residual=res, eps=eps)
    # the sum is the (pinned) all-reduce in fp32, before its final rounding
    s = oracle_mod.allreduce("fp32", "sum", algo, [_widen(dtype, a) for a in x])
    h = (s + _widen(dtype, res)).astype(np.float32)
    assert rout.tobytes() == _round(dtype, h.astype(np.float64)).tobytes()
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h.astype(np.float64)).view(rows, hidden), (hidden,),
                                       weight=torch.from_numpy(_widen(dtype, w).astype(np.float64)), eps=eps)
    want = _round(dtype, ref.reshape(-1).numpy())
    got_f, want_f = _widen(dtype, out), _widen(dtype, want)
    # fp64 evaluation on both sides: equal after rounding, except a value
    # within an fp64 rounding of a tie, which may land one unit apart
    ulp = np.spacing(np.abs(want_f).astype(np.float32))
    if dtype == "bf16":
        ulp = ulp * 65536
    assert np.all(np.abs(got_f - want_f) <= ulp)
    assert np.mean(got_f == want_f) > 0.999


def test_closed_form_constant_rows(oracle_mod):
    """A row of constant c normalises to c / sqrt(c^2 + eps) * w."""
    W, rows, hidden, eps = 1, 2, 16, 1e-3
    x = [np.concatenate([np.full(hidden, 3.0, np.float32), np.full(hidden, -0.5, np.float32)])]
    w = np.linspace(0.5, 2.0, hidden).astype(np.float32)
    out, rout = oracle_mod.allreduce_rmsnorm("fp32", "ring", x, rows, hidden, w, eps=eps)
    for r, c in enumerate((3.0, -0.5)):
        want = (c / np.sqrt(c * c + eps) * w.astype(np.float64)).astype(np.float32)
        assert np.array_equal(out[r * hidden:(r + 1) * hidden], want)
    assert np.array_equal(rout, x[0])


def test_sum_then_norm_matches_parts(oracle_mod):
    """Without residual the output is the RMSNorm of the all-reduce sum, and
    scaling every input by a power of two leaves it unchanged (eps = 0)."""
    W, rows, hidden = 4, 3, 128
    x = synth.normal(24, W, rows * hidden, 1.0, "fp32")
    w = np.ones(hidden, np.float32)
    a, _ = oracle_mod.allreduce_rmsnorm("fp32", "ring", x, rows, hidden, w, eps=0.0, want_residual_out=False)
    b, _ = oracle_mod.allreduce_rmsnorm("fp32", "ring", [v * np.float32(8) for v in x], rows, hidden, w, eps=0.0,
                                        want_residual_out=False)
    assert np.array_equal(a, b)
    rms = np.sqrt(np.mean(a.reshape(rows, hidden).astype(np.float64) ** 2, axis=1))
    assert np.allclose(rms, 1.0, rtol=1e-6)


def test_rejects_int32(oracle_mod):
    x = [np.zeros(8, np.int32)] * 2
    with pytest.raises(ValueError):
        oracle_mod.allreduce_rmsnorm("int32", "ring", x, 2, 4, np.ones(4, np.int32))
