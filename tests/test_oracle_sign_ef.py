"""Pins of the oracle's 1-bit sign compression with error feedback: the scale
against an independent exact computation (Python integers and fractions) on
gradient-like data, on hand-worked ties, subnormals and extremes, and over
every binade; closed forms, the sign rule, the
error-feedback telescoping identity, and the reduction against the pinned
all-reduce applied to the decoded values."""
import math
from fractions import Fraction

import numpy as np
import pytest

import synth


def _data(seed, W, N):
    g = synth.normal(seed, W, N, 1e-3, "fp32")
    e = synth.normal(seed + 1, W, N, 1e-4, "fp32")
    return g, e


def exact_l1_mean_f32(p):
    """The nearest fp32 to sum(|p|) / N, ties to even, written independently of
    the oracle: the magnitudes are grouped by binary exponent and summed as
    Python integers, the mean is an exact fraction, and the answer is the
    closest of the fp32 neighbours around its double approximation."""
    a = np.abs(np.asarray(p, np.float32).astype(np.float64))
    if np.isnan(a).any():
        return np.float32(np.nan)
    if np.isinf(a).any():
        return np.float32(np.inf)
    m, ex = np.frexp(a)                       # a = m * 2^ex, 0.5 <= m < 1 (or 0)
    ints = np.ldexp(m, 24).astype(np.int64)   # an fp32 magnitude has at most 24 significant bits
    ex = ex - 24
    total = Fraction(0)
    for k in np.unique(ex):
        total += Fraction(int(ints[ex == k].sum())) * Fraction(2) ** int(k)
    t = total / a.size
    c = np.float32(float(t))
    best = None
    with np.errstate(over="ignore"):
        cands = (np.nextafter(c, np.float32(0)), c, np.nextafter(c, np.float32(np.inf)))
    for cand in cands:
        if not np.isfinite(cand):
            continue
        key = (abs(Fraction(float(cand)) - t), int(np.array(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def _scale_of(oracle_mod, p):
    p = np.asarray(p, np.float32)
    return oracle_mod.sign_ef_scales([p], [np.zeros_like(p)])[0]


def test_scale_is_l1_over_n(oracle_mod):
    """Gradient-like data: the scale equals the exact mean magnitude rounded
    once, and (the sum being nearly exact either way) the fsum-based value."""
    W, N = 3, 100003
    g, e = _data(41, W, N)
    s = oracle_mod.sign_ef_scales(g, e)
    for r in range(W):
        p = (g[r] + e[r]).astype(np.float32)
        assert s[r].tobytes() == exact_l1_mean_f32(p).tobytes()
        want = np.float32(math.fsum(abs(float(x)) for x in p) / N)
        assert abs(float(s[r]) - float(want)) <= float(np.spacing(want))


F = np.float32
TWO = 2.0


@pytest.mark.parametrize("p,want", [
    # exact sum 3(1 + 2^-24 + 2^-100): the mean lies just above the tie
    # between 1 and 1 + 2^-23, so it rounds up; an fp64 running sum drops the
    # 2^-100 term and lands on the tie (then to even: 1.0)
    ([3.0, 3 * TWO ** -24, 3 * TWO ** -100], 1 + TWO ** -23),
    # exact ties go to the even neighbour
    ([1.0, 1 + TWO ** -23], 1.0),
    ([1 + TWO ** -23, 1 + TWO ** -22], 1 + TWO ** -22),
    # subnormal means: multiples of 2^-149, the same tie rule
    ([TWO ** -149, 0.0], 0.0),
    ([3 * TWO ** -149, 0.0], 2 * TWO ** -149),
    ([TWO ** -149, 0.0, 0.0], 0.0),
    ([2 * TWO ** -149, 0.0, 0.0], TWO ** -149),
    ([TWO ** -126, TWO ** -149], TWO ** -127),         # (2^23 + 1) / 2 units: tie, to even
    # (3 * 2^24 + 4) / 3 units = 2^24 + 1 + 1/3: the quotient's dropped bit is
    # exactly one half, and only the remainder 1/3 lifts it past the tie
    ([3 * TWO ** -125, TWO ** -147, 0.0], TWO ** -125 + TWO ** -148),
    # the largest magnitudes do not overflow the sum
    ([3.4028234663852886e38] * 2, 3.4028234663852886e38),
    ([3.4028234663852886e38, 0.0], 1.7014117331926443e38),
    # signs do not matter, -0 adds nothing
    ([-2.0, 2.0, -0.0, 0.0], 1.0),
])
def test_scale_rounds_the_exact_mean_once(oracle_mod, p, want):
    got = _scale_of(oracle_mod, p)
    assert got.tobytes() == F(want).tobytes(), (got, want)
    assert got.tobytes() == exact_l1_mean_f32(p).tobytes()


def test_scale_of_non_finite(oracle_mod):
    assert np.isposinf(_scale_of(oracle_mod, [1.0, np.inf, -2.0]))
    assert np.isnan(_scale_of(oracle_mod, [1.0, np.inf, np.nan]))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_scale_over_every_binade(oracle_mod, seed):
    """Magnitudes drawn over the whole fp32 range, subnormals included, with
    random signs: the oracle's big-integer sum against the exponent-grouped
    one, for several N (the division's remainders differ)."""
    rng = np.random.default_rng(seed)
    for N in (1, 2, 3, 7, 1000, 10007):
        bits = rng.integers(0, 0x7F800000, size=N, dtype=np.uint32)
        bits |= rng.integers(0, 2, size=N, dtype=np.uint32) << np.uint32(31)
        p = bits.view(np.float32)
        assert _scale_of(oracle_mod, p).tobytes() == exact_l1_mean_f32(p).tobytes(), N
        q = (p * F(2.0 ** -100)).astype(np.float32)        # mostly subnormal and zero
        assert _scale_of(oracle_mod, q).tobytes() == exact_l1_mean_f32(q).tobytes(), N


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
