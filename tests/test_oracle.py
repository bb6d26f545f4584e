"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check is a hand-derived
worked example, a closed form, an invariant the pages state, brute force in
pure Python, or a library routine on a special case.

Page: "Learning FlashAttention the Hard Way - Part 1" (cloudrift.ai).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import attention as ora

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def val(s: str) -> float:
    s = s.strip()
    if s.startswith("ln(") and s.endswith(")"):
        return math.log(float(Fraction(s[3:-1])))
    return float(Fraction(s))


def arr(x):
    if isinstance(x, str):
        return val(x)
    return np.array([arr(e) for e in x], dtype=np.float64)


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# --- worked examples (hand-derived, tests/golden/hand_examples.json) -------

@pytest.mark.parametrize("mode", ["causal", "noncausal"])
def test_golden_dense_logweights(golden, mode):
    g = golden["dense_logweights"]
    scale = val(g["scale"])
    W = arr(g["W"])
    V = arr(g["V"])
    q = np.log(W) / scale
    k = np.eye(3)
    exp_O = arr(g[mode]["O"])
    exp_L = arr(g[mode]["LSE"])
    for c in [0.0] + [val(x) for x in g["offsets"]]:
        o, l = ora.attention_head_ref(q + c / scale, k, V, scale,
                                      causal=(mode == "causal"))
        np.testing.assert_allclose(o, exp_O, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l, exp_L + c, rtol=1e-13, atol=1e-12)


def test_golden_two_keys(golden):
    g = golden["two_keys"]
    o, l = ora.attention_head_ref(arr(g["q"]), arr(g["k"]), arr(g["v"]),
                                  val(g["scale"]), causal=False)
    np.testing.assert_allclose(o, arr(g["O"]), rtol=1e-14)
    np.testing.assert_allclose(l, arr(g["LSE"]), rtol=1e-14)


def test_golden_base2_states(golden):
    g = golden["base2_states"]
    V = arr(g["V"])
    sig = [arr(c) for c in g["sigma_chunks"]]
    # chunk states by their definition
    sA = ora.row_state(sig[0], V[0:2], base=2.0)
    sB = ora.row_state(sig[1], V[2:3], base=2.0)
    for s, e in zip((sA, sB), g["states"]):
        assert s[0] == val(e["m"]) and s[1] == val(e["d"])
        np.testing.assert_allclose(s[2], arr(e["o"]), rtol=1e-15)
    u = ora.merge(sA, sB, base=2.0)
    assert u[0] == val(g["merged"]["m"]) and u[1] == val(g["merged"]["d"])
    np.testing.assert_allclose(u[2], arr(g["merged"]["o"]), rtol=1e-15)
    O, L = ora.finalize(u, base=2.0)
    np.testing.assert_allclose(O, arr(g["O"]), rtol=1e-14)
    assert abs(L - val(g["LSE"])) < 1e-14
    # the split-KV combine over the same two states
    Oc, Lc = ora.combine_ref(np.array([[sA[0], sB[0]]]),
                             np.array([[sA[1], sB[1]]]),
                             np.array([[sA[2], sB[2]]]))
    np.testing.assert_allclose(Oc[0], arr(g["O"]), rtol=1e-14)
    assert abs(Lc[0] - val(g["LSE"])) < 1e-14


# --- closed forms and invariants -----------------------------------------

def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def test_softmax_rows_sum_to_one():
    s = _rand((7, 33), 0, std=30.0)
    s[2, 5:] = -np.inf
    p = ora.softmax_ref(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert (p >= 0).all() and (p[2, 5:] == 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_gives_means(causal):
    """Identical scores: every visible key weighs the same, so O is the mean
    of the visible V rows and LSE = ln(count)."""
    N, D = 37, 5
    q, k, v = _rand((N, D), 1), _rand((N, D), 2), _rand((N, D), 3)
    o, l = ora.attention_head_ref(q, k, v, 0.0, causal)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[i], v[:n].mean(0), rtol=1e-12, atol=1e-13)
        assert abs(l[i] - math.log(n)) < 1e-13


def test_single_key_gives_v():
    q, k, v = _rand((1, 8), 4), _rand((1, 8), 5), _rand((1, 8), 6)
    o, l = ora.attention_head_ref(q, k, v, 0.3, causal=False)
    np.testing.assert_array_equal(o, v)
    assert abs(l[0] - 0.3 * float(q[0] @ k[0])) < 1e-14
    # causal row 0 only sees key 0
    q, k, v = _rand((6, 8), 7), _rand((6, 8), 8), _rand((6, 8), 9)
    o, _ = ora.attention_head_ref(q, k, v, 0.3, causal=True)
    np.testing.assert_array_equal(o[0], v[0])


@pytest.mark.parametrize("c", [-90.0, -50.0, 50.0, 90.0, 200.0, 800.0])
def test_offset_invariance(c):
    """Append a coordinate so every score of a row moves by c: q' = [q, c/scale],
    k' = [k, 1].  O must not move; LSE moves by c."""
    N, D, scale = 19, 6, 0.4
    q, k, v = _rand((N, D), 10, 3), _rand((N, D), 11, 3), _rand((N, D), 12)
    for causal in (False, True):
        o0, l0 = ora.attention_head_ref(q, k, v, scale, causal)
        q2 = np.concatenate([q, np.full((N, 1), c / scale)], 1)
        k2 = np.concatenate([k, np.ones((N, 1))], 1)
        o1, l1 = ora.attention_head_ref(q2, k2, v, scale, causal)
        assert np.isfinite(o1).all()
        np.testing.assert_allclose(o1, o0, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(l1, l0 + c, rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_sdpa_float64(causal):
    """Library special case: torch's CPU scaled-dot-product attention in
    float64; LSE against torch.logsumexp over the masked score matrix."""
    B, H, N, D = 2, 3, 45, 16
    g = torch.Generator().manual_seed(7)
    q = torch.randn(B, H, N, D, generator=g, dtype=torch.float64) * 2
    k = torch.randn(B, H, N, D, generator=g, dtype=torch.float64) * 2
    v = torch.randn(B, H, N, D, generator=g, dtype=torch.float64)
    scale = 0.21
    O, L = ora.attention_ref(q, k, v, scale, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, is_causal=causal, scale=scale)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-11, atol=1e-12)
    s = (q @ k.transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    np.testing.assert_allclose(L, torch.logsumexp(s, -1).numpy(), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_pure_python(seed):
    """Tiny cases in pure Python with math.exp and math.fsum, straight from
    the definition O_i = sum_j e^{s_ij} v_j / sum_j e^{s_ij}."""
    rng = np.random.default_rng(100 + seed)
    N, D = int(rng.integers(1, 6)), int(rng.integers(1, 4))
    q, k, v = rng.standard_normal((N, D)), rng.standard_normal((N, D)), \
        rng.standard_normal((N, D))
    scale = float(rng.uniform(0.1, 2.0))
    causal = bool(seed % 2)
    o, l = ora.attention_head_ref(q, k, v, scale, causal)
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        s = {j: scale * math.fsum(q[i, t] * k[j, t] for t in range(D))
             for j in keys}
        w = {j: math.exp(s[j]) for j in keys}
        den = math.fsum(w.values())
        for t in range(D):
            assert abs(o[i, t] - math.fsum(w[j] * v[j, t] for j in keys) / den) \
                < 1e-12
        assert abs(l[i] - math.log(den)) < 1e-12


# --- the (m, d, o) monoid ------------------------------------------------------

def _states(N, D, seed, spread=40.0):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal(N) * spread
    v = rng.standard_normal((N, D))
    return s, v, [ora.inject(s[j], v[j]) for j in range(N)]


def _close(u, ref, tol=1e-12):
    assert u[0] == ref[0]
    assert abs(u[1] - ref[1]) <= tol * abs(ref[1])
    np.testing.assert_allclose(u[2], ref[2], rtol=tol, atol=tol * np.abs(ref[2]).max())


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7])
def test_all_bracketings_agree(N):
    """Every bracketing of the fold gives the state of the whole block as
    defined (max, shifted sum, shifted weighted sum)."""
    s, v, st = _states(N, 3, N)
    ref = ora.row_state(s, v)
    trees = ora.all_bracketings(0, N)
    assert len(trees) == math.comb(2 * (N - 1), N - 1) // N  # Catalan number
    for t in trees:
        _close(ora.fold_tree(st, t), ref)


@pytest.mark.parametrize("N", [1, 2, 5, 8])
def test_all_chunkings_agree(N):
    """Every split into contiguous chunks, each chunk's state by its own
    definition, folded left to right, equals the unsplit state; the final
    row equals the attention definition."""
    s, v, _ = _states(N, 4, 50 + N)
    ref = ora.row_state(s, v)
    chunkings = ora.all_chunkings(N)
    assert len(chunkings) == 2 ** (N - 1)
    for ch in chunkings:
        parts = [ora.row_state(s[a:b], v[a:b]) for a, b in ch]
        _close(ora.fold_left(parts, 4), ref)
    o, l = ora.finalize(ref)
    w = np.exp(s - s.max())
    np.testing.assert_allclose(o, (w @ v) / w.sum(), rtol=1e-12)


def test_identity_and_commutativity():
    s, v, st = _states(6, 3, 9)
    e = ora.identity(3)
    for u in st + [ora.row_state(s, v)]:
        for w in (ora.merge(e, u), ora.merge(u, e)):
            assert w[0] == u[0] and w[1] == u[1]
            np.testing.assert_array_equal(w[2], u[2])
    w = ora.merge(e, e)
    assert w[0] == -math.inf and w[1] == 0.0 and not w[2].any()
    for a, b in itertools.combinations(st, 2):
        _close(ora.merge(a, b), ora.merge(b, a), tol=1e-15)


def test_d_range():
    """Every exponent is <= 0 and the argmax term is 1, so 1 <= d <= N."""
    for seed in range(20):
        N = 1 + seed
        s, v, st = _states(N, 2, 200 + seed, spread=100.0)
        u = ora.fold_left(st, 2)
        assert 1.0 <= u[1] <= N


def test_base2_twist():
    """The state over sigma = s log2(e) with 2^x is the same monoid: m scales
    by log2(e), d and o are unchanged, and the read-off row is the same."""
    s, v, _ = _states(11, 3, 77)
    ue = ora.row_state(s, v, base=math.e)
    u2 = ora.row_state(s * ora.LOG2E, v, base=2.0)
    assert abs(u2[0] - ue[0] * ora.LOG2E) < 1e-12 * abs(ue[0])
    assert abs(u2[1] - ue[1]) < 1e-12 * ue[1]
    np.testing.assert_allclose(u2[2], ue[2], rtol=1e-12)
    oe, le = ora.finalize(ue)
    o2, l2 = ora.finalize(u2, base=2.0)
    np.testing.assert_allclose(o2, oe, rtol=1e-12)
    assert abs(l2 - le) < 1e-12 * abs(le)
    # absolute coordinates: d * base^m = sum base^score (no overflow here)
    s_small = s / 20.0
    u = ora.row_state(s_small, v)
    assert abs(u[1] * math.exp(u[0]) - np.exp(s_small).sum()) < 1e-12 * np.exp(s_small).sum()


# --- planted mistakes: the pins above must catch a broken merge ---------------

def _broken_merges():
    def drop_rescale(a, b, base=math.e):   # forgets to shrink the smaller side
        ma, da, oa = a
        mb, db, ob = b
        if mb == -math.inf:
            return a
        if ma == -math.inf:
            return b
        return (max(ma, mb), da + db, oa + ob)

    def wrong_sign(a, b, base=math.e):     # exponent sign flipped
        ma, da, oa = a
        mb, db, ob = b
        if mb == -math.inf:
            return a
        if ma == -math.inf:
            return b
        if ma >= mb:
            f = base ** (ma - mb)
            return (ma, da + db * f, oa + ob * f)
        f = base ** (mb - ma)
        return (mb, da * f + db, oa * f + ob)

    def d_not_o(a, b, base=math.e):        # rescales d but not o
        ma, da, oa = a
        mb, db, ob = b
        if mb == -math.inf:
            return a
        if ma == -math.inf:
            return b
        if ma >= mb:
            return (ma, da + db * base ** (mb - ma), oa + ob)
        return (mb, da * base ** (ma - mb) + db, oa + ob)
    return [drop_rescale, wrong_sign, d_not_o]


@pytest.mark.parametrize("broken", _broken_merges(), ids=lambda f: f.__name__)
def test_pins_catch_planted_merge_mistakes(monkeypatch, broken):
    monkeypatch.setattr(ora, "merge", broken)
    with pytest.raises(AssertionError):
        test_all_chunkings_agree(5)


# --- split-KV chunk states, combine, decode, varlen ---------------------------

@pytest.mark.parametrize("L,S", [(1, 1), (1, 16), (5, 16), (16, 16), (17, 16),
                                 (1000, 16), (1024, 37), (33, 2)])
def test_chunk_bounds_cover(L, S):
    b = ora.chunk_bounds(L, S)
    assert len(b) == S and b[0][0] == 0 and b[-1][1] == L
    for (a0, a1), (b0, _) in zip(b, b[1:]):
        assert a1 == b0 and a0 <= a1
    size = -(-L // S)
    assert all(e - a <= size for a, e in b)


@pytest.mark.parametrize("L,S,align", [(1, 16, 128), (127, 2, 128), (1024, 16, 128),
                                       (1025, 16, 128), (3001, 5, 128), (700, 7, 64)])
def test_chunk_bounds_aligned(L, S, align):
    """Aligned chunking: the chunks still tile [0, L) in order, every
    boundary but the end is a multiple of align, and the chunk length is
    ceil(L / S) rounded up to such a multiple (trailing chunks may be empty)."""
    b = ora.chunk_bounds(L, S, align)
    assert len(b) == S and b[0][0] == 0 and b[-1][1] == L
    for (a0, a1), (b0, _) in zip(b, b[1:]):
        assert a1 == b0 and a0 <= a1
    assert all(a % align == 0 for a, _ in b if a < L)
    size = -(-(-(-L // S)) // align) * align
    assert all(e - a == min(size, max(0, L - a)) for a, e in b)


def _decode_case(B=3, H=2, D=8, lens=(1, 9, 40), seed=0, std=2.0):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q = rng.standard_normal((B, H, D)) * std
    kc = rng.standard_normal((T, H, D)) * std
    vc = rng.standard_normal((T, H, D))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, kc, vc, cu


def test_decode_is_last_causal_row():
    """The newest token sees the whole cache: decode equals the last row of
    causal attention over the sequence with that token's query last."""
    q, kc, vc, cu = _decode_case()
    O, L = ora.decode_ref(q, kc, vc, cu, 0.35)
    for b in range(3):
        a, e = cu[b], cu[b + 1]
        for h in range(2):
            qq = np.array(kc[a:e, h])  # any earlier queries; only the last row is checked
            qq[-1] = q[b, h]
            o, l = ora.attention_head_ref(qq, kc[a:e, h], vc[a:e, h], 0.35, True)
            np.testing.assert_allclose(O[b, h], o[-1], rtol=1e-13)
            assert abs(L[b, h] - l[-1]) < 1e-13


@pytest.mark.parametrize("S", [1, 2, 16, 37])
def test_split_then_combine_equals_unsplit(S):
    q, kc, vc, cu = _decode_case(lens=(1, 9, 40, 300), B=4, seed=S)
    M, Dn, Oc = ora.chunk_states_ref(q, kc, vc, cu, S, 0.35)
    O, L = ora.combine_ref(M, Dn, Oc)
    Or, Lr = ora.decode_ref(q, kc, vc, cu, 0.35)
    np.testing.assert_allclose(O, Or, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lr, rtol=1e-13)
    # empty chunks carry the identity; all others have 1 <= d <= chunk length
    for b, Lb in enumerate((1, 9, 40, 300)):
        for c, (a, e) in enumerate(ora.chunk_bounds(Lb, S)):
            if a == e:
                assert M[b, 0, c] == -math.inf and Dn[b, 0, c] == 0
                assert not Oc[b, 0, c].any()
            else:
                assert 1.0 <= Dn[b, 0, c] <= (e - a)


def test_one_chunk_is_the_whole_state():
    q, kc, vc, cu = _decode_case()
    M, Dn, Oc = ora.chunk_states_ref(q, kc, vc, cu, 1, 0.5)
    for b in range(3):
        a, e = cu[b], cu[b + 1]
        sig = kc[a:e, 1] @ q[b, 1] * 0.5 * ora.LOG2E
        w = 2.0 ** (sig - sig.max())
        assert M[b, 1, 0] == sig.max()
        assert abs(Dn[b, 1, 0] - w.sum()) < 1e-13 * w.sum()
        np.testing.assert_allclose(Oc[b, 1, 0], w @ vc[a:e, 1], rtol=1e-13)


def test_varlen_is_dense_per_sequence():
    rng = np.random.default_rng(3)
    lens = [5, 1, 12]
    H, D = 2, 4
    T = sum(lens)
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out = ora.varlen_ref(q, k, v, cu, 0.7, True)
    # a single sequence is dense attention
    one = ora.varlen_ref(q[:5], k[:5], v[:5], [0, 5], 0.7, True)[0]
    np.testing.assert_array_equal(one[0], out[0][0])
    # sequences do not see each other: changing sequence 0 leaves 2 unchanged
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    k2[:5] += 10.0
    v2[:5] -= 3.0
    out2 = ora.varlen_ref(q2, k2, v2, cu, 0.7, True)
    np.testing.assert_array_equal(out2[2][0], out[2][0])
    np.testing.assert_array_equal(out2[1][0], out[1][0])
    # length-1 sequence: O = v
    np.testing.assert_array_equal(out[1][0][0], v[5])


def test_empty_blocks_are_the_identity():
    """A block with no keys is the identity (-inf, 0, 0): a row that sees no
    key reads off O = 0 and LSE = -inf; a sequence with no tokens has no rows."""
    q = np.ones((2, 3))
    o, l = ora.attention_head_ref(q, np.zeros((0, 3)), np.zeros((0, 3)), 0.5, False)
    assert o.shape == (2, 3) and not o.any() and (l == -np.inf).all()
    out = ora.varlen_ref(np.ones((3, 1, 4)), np.ones((3, 1, 4)), np.ones((3, 1, 4)),
                         [0, 2, 2, 3], 0.5, True)
    assert out[1][0].shape == (0, 1, 4) and out[1][1].shape == (1, 0)
    np.testing.assert_array_equal(out[2][0][0, 0], np.ones(4))
