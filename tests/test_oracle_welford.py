"""Pins of the Welford / Chan oracle against what the mathematics fixes:
exact rational arithmetic on small integer samples, the library variance,
every bracketing and chunking of the merge, the identity law, the twist to
plain sums, a sample where the one-pass sum-of-squares formula fails, and
planted mistakes that the pins must catch."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import welford as wf


def _exact(xs):
    """Mean and M2 in exact rational arithmetic."""
    n = len(xs)
    mu = Fraction(sum(xs), n)
    return n, mu, sum((Fraction(x) - mu) ** 2 for x in xs)


def test_worked_example_exact():
    xs = [2, 4, 4, 4, 5, 5, 7, 9]  # mean 5, population variance 4
    n, mu, m2 = wf.two_pass(xs)
    assert (n, mu, m2) == (8.0, 5.0, 32.0)
    st = wf.IDENTITY
    for x in xs:
        st = wf.update(st, x)
    assert st == (8.0, 5.0, 32.0)
    assert wf.finalize(st) == (5.0, 4.0)
    assert wf.finalize(st, ddof=1) == (5.0, 32.0 / 7.0)


@pytest.mark.parametrize("seed", range(5))
def test_streaming_and_merge_match_exact_rationals(seed):
    rng = np.random.default_rng(seed)
    xs = rng.integers(-50, 50, size=int(rng.integers(1, 40))).tolist()
    n, mu, m2 = _exact(xs)
    st = wf.IDENTITY
    for x in xs:
        st = wf.update(st, x)
    assert st[0] == n
    assert abs(st[1] - float(mu)) <= 1e-13 * max(1.0, abs(float(mu)))
    assert abs(st[2] - float(m2)) <= 1e-12 * max(1.0, float(m2))
    merged = wf.fold_left(wf.inject(x) for x in xs)
    assert abs(merged[1] - float(mu)) <= 1e-13 * max(1.0, abs(float(mu)))
    assert abs(merged[2] - float(m2)) <= 1e-12 * max(1.0, float(m2))


def test_matches_numpy_var():
    x = np.random.default_rng(7).standard_normal((6, 333)) * 3 + 2
    mu, var, rstd = wf.row_stats_ref(x, eps=1e-5)
    np.testing.assert_allclose(mu, x.mean(1), rtol=1e-14)
    np.testing.assert_allclose(var, x.var(1), rtol=1e-13)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(x.var(1) + 1e-5), rtol=1e-13)
    st = wf.two_pass(x[0])
    assert abs(wf.finalize(st, ddof=1)[1] - np.var(x[0], ddof=1)) < 1e-12


def _brackets(items):
    if len(items) == 1:
        yield items[0]
        return
    for i in range(1, len(items)):
        for left in _brackets(items[:i]):
            for right in _brackets(items[i:]):
                yield wf.merge(left, right)


def test_every_bracketing_agrees():
    x = np.random.default_rng(3).standard_normal(6) * 5 + 10
    ref = wf.two_pass(x)
    states = [wf.inject(v) for v in x]
    count = 0
    for st in _brackets(states):
        count += 1
        assert st[0] == ref[0]
        assert abs(st[1] - ref[1]) < 1e-13 * abs(ref[1])
        assert abs(st[2] - ref[2]) < 1e-12 * ref[2]
    assert count == 42  # Catalan(5)


def test_every_chunking_agrees_and_identity():
    x = np.random.default_rng(4).standard_normal(8) * 2 - 1
    ref = wf.two_pass(x)
    for cuts in itertools.product([0, 1], repeat=7):
        bounds = [0] + [i + 1 for i, c in enumerate(cuts) if c] + [8]
        parts = [wf.two_pass(x[a:b]) for a, b in zip(bounds, bounds[1:])]
        st = wf.fold_left(parts)
        assert abs(st[1] - ref[1]) < 1e-13 and abs(st[2] - ref[2]) < 1e-12 * ref[2]
    a = wf.two_pass(x[:3])
    assert wf.merge(a, wf.IDENTITY) == a and wf.merge(wf.IDENTITY, a) == a
    b = wf.two_pass(x[3:])
    ab, ba = wf.merge(a, b), wf.merge(b, a)
    assert ab[0] == ba[0] and abs(ab[1] - ba[1]) < 1e-14 and abs(ab[2] - ba[2]) < 1e-13


def test_twist_is_plain_sums():
    """Merging states equals adding (n, sum x, sum x^2) and twisting back."""
    rng = np.random.default_rng(9)
    a, b = rng.standard_normal(11), rng.standard_normal(5) + 3
    sa, sb = wf.two_pass(a), wf.two_pass(b)
    na, ta, wa = wf.untwist(sa)
    nb, tb, wb = wf.untwist(sb)
    assert abs(ta - a.sum()) < 1e-12 and abs(wa - (a * a).sum()) < 1e-12
    st = wf.twist(na + nb, ta + tb, wa + wb)
    m = wf.merge(sa, sb)
    assert st[0] == m[0] and abs(st[1] - m[1]) < 1e-14 and abs(st[2] - m[2]) < 1e-11


def test_cancellation_case():
    """Samples 1e9 + {0, 1, 2, 3}: exact variance 1.25.  The one-pass
    sum-of-squares formula in float64 loses it; Welford and two-pass keep it."""
    x = 1e9 + np.arange(4.0)
    naive = (x * x).sum() / 4 - (x.sum() / 4) ** 2
    assert abs(naive - 1.25) > 1e-2
    st = wf.fold_left(wf.inject(v) for v in x)
    assert abs(wf.finalize(st)[1] - 1.25) < 1e-6
    assert abs(wf.finalize(wf.two_pass(x))[1] - 1.25) < 1e-6


@pytest.mark.parametrize("S", [1, 2, 7, 64])
def test_chunk_states_combine_to_row_stats(S):
    x = np.random.default_rng(S).standard_normal((5, 100)) * 4 + 7
    n, mu, m2 = wf.chunk_states_ref(x, S)
    assert (n.sum(1) == 100).all()
    cm, cv, cr = wf.combine_ref(n, mu, m2, eps=1e-6)
    rm, rv, rr = wf.row_stats_ref(x, eps=1e-6)
    np.testing.assert_allclose(cm, rm, rtol=1e-13)
    np.testing.assert_allclose(cv, rv, rtol=1e-12)
    np.testing.assert_allclose(cr, rr, rtol=1e-12)


def _bad_merge_no_cross(a, b):
    na, mua, m2a = a
    nb, mub, m2b = b
    if nb == 0:
        return a
    if na == 0:
        return b
    n = na + nb
    return (n, mua + (mub - mua) * nb / n, m2a + m2b)


def _bad_merge_mean(a, b):
    na, mua, m2a = a
    nb, mub, m2b = b
    if nb == 0:
        return a
    if na == 0:
        return b
    n = na + nb
    d = mub - mua
    return (n, mua + d * na / n, m2a + m2b + d * d * na * nb / n)


@pytest.mark.parametrize("bad", [_bad_merge_no_cross, _bad_merge_mean])
def test_planted_mistakes_fail_the_chunking_pin(bad, monkeypatch):
    x = np.random.default_rng(12).standard_normal(9) * 3 + 1
    ref = wf.two_pass(x)
    monkeypatch.setattr(wf, "merge", bad)
    st = wf.fold_left([wf.two_pass(x[:2]), wf.two_pass(x[2:7]), wf.two_pass(x[7:])])
    assert abs(st[1] - ref[1]) > 1e-6 or abs(st[2] - ref[2]) > 1e-6


def test_c_fp32_fold_agrees_with_float64():
    """The fixed-order fp32 C fold of chunk states agrees with the float64
    oracle to fp32 accuracy, leaves identity chunks without effect, and one
    chunk passes through exactly (var = one IEEE division)."""
    from oracle import combine_f32 as cf
    x = np.random.default_rng(21).standard_normal((7, 500)) * 2 + 3
    n, mu, m2 = wf.chunk_states_ref(x, 9)
    n32, mu32, m232 = (a.astype(np.float32) for a in (n, mu, m2))
    mean, var, rstd = cf.welford_combine_f32(n32, mu32, m232, eps=1e-5)
    rm, rv, rr = wf.combine_ref(n32.astype(np.float64), mu32.astype(np.float64),
                                m232.astype(np.float64), eps=1e-5)
    np.testing.assert_allclose(mean, rm, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(var, rv, rtol=1e-5)
    np.testing.assert_allclose(rstd, rr, rtol=1e-5)
    # identity chunks (n = 0) interleaved change no bit
    z = np.zeros((7, 1), np.float32)
    n2 = np.concatenate([z, n32[:, :4], z, n32[:, 4:], z], axis=1)
    mu2 = np.concatenate([z, mu32[:, :4], z, mu32[:, 4:], z], axis=1)
    m22 = np.concatenate([z, m232[:, :4], z, m232[:, 4:], z], axis=1)
    mean2, var2, rstd2 = cf.welford_combine_f32(n2, mu2, m22, eps=1e-5)
    assert (mean2 == mean).all() and (var2 == var).all() and (rstd2 == rstd).all()
    # one chunk: mean passes through, var = M2 / n rounded once
    m1, v1, _ = cf.welford_combine_f32(n32[:, :1], mu32[:, :1], m232[:, :1])
    assert (m1 == mu32[:, 0]).all() and (v1 == m232[:, 0] / n32[:, 0]).all()
