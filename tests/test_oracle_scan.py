"""Pins of the prefix-scan oracle: every prefix equals decode over that
prefix and the matching row of causal attention with the query repeated;
the left-fold scan and the two-sweep tree scan agree with the definition for
lengths that are and are not powers of two; a planted down-sweep mistake
fails; pure-Python brute force on a tiny case."""
import math

import numpy as np
import pytest

from oracle import attention as ora


def _seq(L, D, seed, std=1.5):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(D) * std, rng.standard_normal((L, D)) * std, \
        rng.standard_normal((L, D))


def _states(q, k, v, scale):
    return [ora.inject(scale * float(q @ k[j]), v[j]) for j in range(len(k))]


def test_prefix_equals_decode_and_causal_rows():
    lens = [1, 9, 40]
    D, H = 6, 2
    rng = np.random.default_rng(3)
    T = sum(lens)
    k = rng.standard_normal((T, H, D)) * 2
    v = rng.standard_normal((T, H, D))
    q = rng.standard_normal((3, H, D)) * 2
    cu = np.concatenate([[0], np.cumsum(lens)])
    O, L = ora.prefix_attention_ref(q, k, v, cu, 0.4)
    for b in range(3):
        a = cu[b]
        for i in range(lens[b]):
            cu1 = np.array([0, i + 1])
            o1, l1 = ora.decode_ref(q[b:b + 1], k[a:a + i + 1], v[a:a + i + 1], cu1, 0.4)
            np.testing.assert_allclose(O[a + i], o1[0], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(L[:, a + i], l1[0], rtol=1e-13)
        for h in range(H):
            qrep = np.repeat(q[b, h][None, :], lens[b], axis=0)
            oc, lc = ora.attention_head_ref(qrep, k[a:a + lens[b], h], v[a:a + lens[b], h], 0.4, True)
            np.testing.assert_allclose(O[a:a + lens[b], h], oc, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(L[h, a:a + lens[b]], lc, rtol=1e-13)


@pytest.mark.parametrize("L", [1, 2, 3, 7, 8, 13, 32])
def test_scans_match_definition(L):
    D = 4
    q, k, v = _seq(L, D, L)
    st = _states(q, k, v, 0.7)
    left = ora.scan_left(st, D)
    tree = ora.scan_tree(st, D)
    O, LSE = ora.prefix_attention_ref(q[None, None], k[:, None], v[:, None], [0, L], 0.7)
    for i in range(L):
        for sc in (left[i], tree[i]):
            o, lse = ora.finalize(sc)
            np.testing.assert_allclose(o, O[i, 0], rtol=1e-12, atol=1e-13)
            assert abs(lse - LSE[0, i]) < 1e-12


def test_planted_down_sweep_mistake_fails(monkeypatch):
    """Dropping the exchange of the down-sweep (each node keeps its own
    subtree total) breaks the prefixes."""
    D, L = 3, 8
    q, k, v = _seq(L, D, 99)
    st = _states(q, k, v, 0.9)

    def bad_tree(states, D, base=math.e):
        n = len(states)
        t = list(states)
        step = 1
        while step < n:
            for i in range(2 * step - 1, n, 2 * step):
                t[i] = ora.merge(t[i - step], t[i], base)
            step *= 2
        return t

    good = ora.scan_left(st, D)
    bad = bad_tree(st, D)
    assert any(abs(ora.finalize(g)[1] - ora.finalize(b)[1]) > 1e-6 for g, b in zip(good, bad))


def test_brute_force_tiny():
    q = np.array([1.0, -2.0])
    k = np.array([[0.5, 0.25], [-1.0, 1.0], [2.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 3.0], [-1.0, 1.0]])
    O, L = ora.prefix_attention_ref(q[None, None], k[:, None], v[:, None], [0, 3], 1.0)
    for i in range(3):
        e = [math.exp(q[0] * k[j, 0] + q[1] * k[j, 1]) for j in range(i + 1)]
        den = math.fsum(e)
        for c in range(2):
            assert abs(O[i, 0, c] - math.fsum(e[j] * v[j, c] for j in range(i + 1)) / den) < 1e-14
        assert abs(L[0, i] - math.log(den)) < 1e-14
