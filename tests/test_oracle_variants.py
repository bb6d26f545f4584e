"""Pins of the oracle's mask and cache variants: the causal sliding window,
and split-KV decode over a paged KV cache with grouped query heads.

Each is checked against closed forms, pure-Python brute force, or the plain
(unwindowed, contiguous, one-KV-head-per-query-head) definition it reduces to.
"""
import math

import numpy as np
import pytest

from oracle import attention as ora


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# --- sliding window -----------------------------------------------------------------

def test_window_at_least_n_is_causal():
    N, D = 23, 5
    q, k, v = _rand((N, D), 1, 2), _rand((N, D), 2, 2), _rand((N, D), 3)
    o0, l0 = ora.attention_head_ref(q, k, v, 0.4, True)
    for w in (N, N + 7):
        o1, l1 = ora.attention_head_ref(q, k, v, 0.4, True, window=w)
        np.testing.assert_array_equal(o1, o0)
        np.testing.assert_array_equal(l1, l0)


def test_window_one_sees_only_itself():
    N, D = 9, 4
    q, k, v = _rand((N, D), 4), _rand((N, D), 5), _rand((N, D), 6)
    o, l = ora.attention_head_ref(q, k, v, 0.7, True, window=1)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(l, 0.7 * (q * k).sum(1), rtol=1e-14)


@pytest.mark.parametrize("w", [1, 3, 8])
def test_window_scale_zero_gives_window_means(w):
    N, D = 17, 3
    q, k, v = _rand((N, D), 7), _rand((N, D), 8), _rand((N, D), 9)
    o, l = ora.attention_head_ref(q, k, v, 0.0, True, window=w)
    for i in range(N):
        lo = max(0, i - w + 1)
        np.testing.assert_allclose(o[i], v[lo:i + 1].mean(0), rtol=1e-12, atol=1e-14)
        assert abs(l[i] - math.log(i + 1 - lo)) < 1e-13


@pytest.mark.parametrize("seed", range(4))
def test_window_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    N, D, w = int(rng.integers(2, 8)), int(rng.integers(1, 4)), int(rng.integers(1, 5))
    q, k, v = (rng.standard_normal((N, D)) for _ in range(3))
    o, l = ora.attention_head_ref(q, k, v, 0.9, True, window=w)
    for i in range(N):
        keys = [j for j in range(N) if i - w < j <= i]
        e = {j: math.exp(0.9 * math.fsum(q[i, t] * k[j, t] for t in range(D))) for j in keys}
        den = math.fsum(e.values())
        for t in range(D):
            assert abs(o[i, t] - math.fsum(e[j] * v[j, t] for j in keys) / den) < 1e-12
        assert abs(l[i] - math.log(den)) < 1e-12


# --- paged KV cache with grouped query heads ------------------------------------------

def _paged_case(lens, H, Hkv, D, page, seed, shuffle=True):
    rng = np.random.default_rng(seed)
    B = len(lens)
    nblk = [-(-L // page) for L in lens]
    P = sum(nblk) + 3
    kp = rng.standard_normal((P, page, Hkv, D)) * 2
    vp = rng.standard_normal((P, page, Hkv, D))
    perm = rng.permutation(P) if shuffle else np.arange(P)
    table = np.full((B, max(nblk)), -1, dtype=np.int32)
    i = 0
    for b in range(B):
        for c in range(nblk[b]):
            table[b, c] = perm[i]
            i += 1
    q = rng.standard_normal((B, H, D)) * 2
    return q, kp, vp, table, np.array(lens)


def _contiguous(kp, vp, table, lens):
    """The same caches laid out as packed [T, H_kv, D] with cu_seqlens."""
    ks, vs = [], []
    for b, L in enumerate(lens):
        page = kp.shape[1]
        for t in range(L):
            ks.append(kp[table[b, t // page], t % page])
            vs.append(vp[table[b, t // page], t % page])
    cu = np.concatenate([[0], np.cumsum(lens)])
    return np.array(ks), np.array(vs), cu


def test_paged_equals_contiguous_and_gqa_equals_repeated_heads():
    lens = [1, 5, 16, 17, 100]
    H, Hkv, D, page = 6, 2, 4, 16
    q, kp, vp, table, sl = _paged_case(lens, H, Hkv, D, page, seed=1)
    O, L = ora.decode_paged_ref(q, kp, vp, table, sl, 0.3)
    kc, vc, cu = _contiguous(kp, vp, table, lens)
    # repeat each KV head for its group of query heads: ordinary multi-head decode
    g = H // Hkv
    O2, L2 = ora.decode_ref(q, np.repeat(kc, g, axis=1), np.repeat(vc, g, axis=1), cu, 0.3)
    np.testing.assert_allclose(O, O2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L, L2, rtol=1e-14)


def test_page_order_does_not_matter():
    """Moving pages around the pool and updating the table accordingly leaves
    the logical cache, and so every result, unchanged."""
    lens = [40, 9, 33]
    q, kp, vp, table, sl = _paged_case(lens, 4, 4, 8, 8, seed=2, shuffle=False)
    O1, L1 = ora.decode_paged_ref(q, kp, vp, table, sl, 0.5)
    perm = np.random.default_rng(5).permutation(kp.shape[0])  # new slot of page p: perm[p]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    O2, L2 = ora.decode_paged_ref(q, kp2, vp2, table2, sl, 0.5)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


@pytest.mark.parametrize("S", [1, 3, 16])
def test_paged_chunks_combine_to_unsplit(S):
    lens = [1, 7, 64, 129]
    q, kp, vp, table, sl = _paged_case(lens, 8, 2, 4, 32, seed=S)
    M, Dn, Oc = ora.chunk_states_paged_ref(q, kp, vp, table, sl, S, 0.25)
    O, L = ora.combine_ref(M, Dn, Oc)
    O2, L2 = ora.decode_paged_ref(q, kp, vp, table, sl, 0.25)
    np.testing.assert_allclose(O, O2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, L2, rtol=1e-13)
