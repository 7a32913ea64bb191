"""Pins of the oracle's 1-bit sign compression with error feedback: the scale
against an exact sum (math.fsum), closed forms, the sign rule, the
error-feedback telescoping identity, and the reduction against the pinned
all-reduce applied to the decoded values."""
import math

import numpy as np
import pytest

import synth


def _data(seed, W, N):
    g = synth.normal(seed, W, N, 1e-3, "fp32")
    e = synth.normal(seed + 1, W, N, 1e-4, "fp32")
    return g, e


def test_scale_is_l1_over_n(oracle_mod):
    W, N = 3, 100003
    g, e = _data(41, W, N)
    s = oracle_mod.sign_ef_scales(g, e)
    for r in range(W):
        p = (g[r] + e[r]).astype(np.float32)
        exact = math.fsum(abs(float(x)) for x in p) / N
        want = np.float32(exact)
        assert abs(float(s[r]) - float(want)) <= float(np.spacing(want))


def test_closed_forms_and_sign_rule(oracle_mod):
    N = 8
    g = [np.array([0.5, 0.5, 0.0, -0.0, 0.5, 0.5, 0.5, 0.5], np.float32)]
    e = [np.zeros(N, np.float32)]
    s = oracle_mod.sign_ef_scales(g, e)
    assert s[0] == np.float32(3.0 / 8)
    out, e2 = oracle_mod.sign_ef_collective("allreduce", "sum", "ring", g, e, s)
    # zero and negative zero take the + sign
    assert out.tolist() == [0.375] * 8
    assert np.array_equal(e2[0], (g[0] - np.float32(0.375)).astype(np.float32))
    # a constant positive buffer is sent exactly: no residual
    c = [np.full(16, 0.25, np.float32)]
    z = [np.zeros(16, np.float32)]
    s = oracle_mod.sign_ef_scales(c, z)
    out, e2 = oracle_mod.sign_ef_collective("allreduce", "sum", "ring", c, z, s)
    assert s[0] == np.float32(0.25) and np.all(out == np.float32(0.25)) and np.all(e2[0] == 0)


@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("W,N", [(2, 64), (5, 1003), (8, 4096)])
def test_reduction_of_decoded_values(oracle_mod, op, algo, W, N):
    """The output is the all-reduce of the decoded values q_r = sign(p_r) s_r,
    and each rank's new error is p_r - q_r."""
    g, e = _data(42 + W, W, N)
    s = oracle_mod.sign_ef_scales(g, e)
    out, e2 = oracle_mod.sign_ef_collective("allreduce", op, algo, g, e, s)
    q = []
    for r in range(W):
        p = (g[r] + e[r]).astype(np.float32)
        qr = np.where(p >= 0, s[r], -s[r]).astype(np.float32)
        q.append(qr)
        assert np.array_equal(e2[r], (p - qr).astype(np.float32))
    want = oracle_mod.allreduce("fp32", op, algo, q)
    assert out.tobytes() == want.tobytes()
    if N % W == 0:
        shards, _ = oracle_mod.sign_ef_collective("reduce_scatter", op, algo, g, e, s)
        assert np.concatenate(shards).tobytes() == want.tobytes()


def test_error_feedback_telescopes(oracle_mod):
    """Over T steps with one rank, what was transmitted plus what is still owed
    equals what the gradients added: sum_t q_t + e_T = T g + e_0 (up to the
    rounding of the fp32 updates)."""
    N, T = 2000, 6
    g = synth.normal(43, 1, N, 1e-3, "fp32")
    e = [np.zeros(N, np.float32)]
    sent = np.zeros(N, np.float64)
    for _ in range(T):
        s = oracle_mod.sign_ef_scales(g, e)
        q, e = oracle_mod.sign_ef_collective("allreduce", "sum", "ring", g, e, s)
        sent += q.astype(np.float64)
    lhs = sent + e[0].astype(np.float64)
    rhs = T * g[0].astype(np.float64)
    assert np.all(np.abs(lhs - rhs) <= 4 * T * np.spacing(np.float32(2e-2)))


def test_ranks_are_independent(oracle_mod):
    """Each rank's error update depends on that rank alone."""
    W, N = 4, 777
    g, e = _data(44, W, N)
    s = oracle_mod.sign_ef_scales(g, e)
    _, e2 = oracle_mod.sign_ef_collective("allreduce", "avg", "tree", g, e, s)
    for r in range(W):
        s1 = oracle_mod.sign_ef_scales([g[r]], [e[r]])
        assert s1[0] == s[r]
        _, e1 = oracle_mod.sign_ef_collective("allreduce", "sum", "ring", [g[r]], [e[r]], s1)
        assert np.array_equal(e1[0], e2[r])
