"""Pins of the float64 backward oracle.  The pages name the backward pass
(recomputation instead of storing P) but give no formulas, so the oracle's
explicit formulas are pinned against things that do not share them: central
finite differences of the forward oracle, torch autograd in float64, and
identities the gradient must satisfy."""
import numpy as np
import pytest
import torch

from oracle import attention as ora


def _case(N, D, seed, std=1.0):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((N, D)) * (std if i < 2 else 1.0) for i in range(4))


def _loss(q, k, v, do, scale, causal):
    o, _ = ora.attention_head_ref(q, k, v, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    """d/dx of <O(q, k, v), dO> by central differences matches every entry."""
    q, k, v, do = _case(5, 3, 1 + causal, std=1.5)
    scale = 0.6
    dq, dk, dv, _ = ora.attention_bwd_head_ref(q, k, v, do, scale, causal)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, do, scale, causal)
            x[idx] = old - h
            lm = _loss(q, k, v, do, scale, causal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_autograd_float64(causal):
    B, H, N, D = 1, 2, 37, 8
    g = torch.Generator().manual_seed(3)
    q, k, v, do = (torch.randn(B, H, N, D, generator=g, dtype=torch.float64) for _ in range(4))
    scale = 0.35
    dq, dk, dv, delta = ora.attention_bwd_ref(q, k, v, do, scale, causal)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=causal,
                                                         scale=scale)
    o.backward(do)
    np.testing.assert_allclose(dq, qq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(delta, (do * o.detach()).sum(-1).numpy(), rtol=1e-12)


def test_gradient_identities():
    """Softmax rows are shift invariant, so dS rows sum to zero: the dQ of a
    constant key shift and sum_j dK_j both vanish; dV sums to sum_i dO_i
    (every row of P sums to 1)."""
    q, k, v, do = _case(11, 4, 7)
    dq, dk, dv, _ = ora.attention_bwd_head_ref(q, k, v, do, 0.8, True)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(0), do.sum(0), rtol=1e-12, atol=1e-12)
    # a single key: the output is v whatever q is, so dq = 0 and dk = 0
    dq1, dk1, dv1, _ = ora.attention_bwd_head_ref(q[:1], k[:1], v[:1], do[:1], 0.8, False)
    np.testing.assert_allclose(dq1, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk1, 0.0, atol=1e-14)
    np.testing.assert_array_equal(dv1, do[:1])


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_equals_full(causal):
    """The row/column-at-a-time backward used at full sizes agrees with the
    whole-matrix one (itself pinned above by finite differences), incl. rows
    and columns at both ends and chunk sizes that do not divide N."""
    N, D = 70, 6
    q, k, v, do = _case(N, D, 11 + causal, std=1.3)
    dq, dk, dv, _ = ora.attention_bwd_head_ref(q, k, v, do, 0.45, causal)
    rows = [0, 1, 33, 68, 69]
    cols = [0, 2, 35, 69]
    sq, sk, sv = ora.attention_bwd_sampled_ref(q, k, v, do, 0.45, causal, rows, cols, chunk=16)
    np.testing.assert_allclose(sq, dq[rows], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sk, dk[cols], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sv, dv[cols], rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_is_per_sequence(causal):
    """One packed sequence equals the dense backward of that sequence; the
    gradients of a sequence do not depend on its neighbours."""
    rng = np.random.default_rng(30 + causal)
    lens = [7, 1, 12]
    T, H, D = sum(lens), 2, 4
    q, k, v, do = (rng.standard_normal((T, H, D)) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lens)])
    dq, dk, dv, delta = ora.attention_bwd_varlen_ref(q, k, v, do, cu, 0.5, causal)
    a, e = cu[2], cu[3]
    sl = lambda x: x[a:e].transpose(1, 0, 2)[None]
    rq, rk, rv, rd = ora.attention_bwd_ref(sl(q), sl(k), sl(v), sl(do), 0.5, causal)
    np.testing.assert_allclose(dq[a:e].transpose(1, 0, 2), rq[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk[a:e].transpose(1, 0, 2), rk[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv[a:e].transpose(1, 0, 2), rv[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(delta[:, a:e], rd[0], rtol=1e-13, atol=1e-14)
    q2 = q.copy()
    q2[:cu[2]] = rng.standard_normal((cu[2], H, D))  # change the other sequences
    g2 = ora.attention_bwd_varlen_ref(q2, k, v, do, cu, 0.5, causal)
    np.testing.assert_array_equal(g2[0][a:e], dq[a:e])
    np.testing.assert_array_equal(g2[1][a:e], dk[a:e])


@pytest.mark.parametrize("w", [1, 2, 4])
def test_window_finite_differences(w):
    """The sliding-window backward against central differences of the
    windowed forward oracle."""
    q, k, v, do = _case(6, 3, 40 + w, std=1.5)
    scale = 0.7
    dq, dk, dv, _ = ora.attention_bwd_head_ref(q, k, v, do, scale, True, window=w)
    h = 1e-6

    def loss():
        o, _ = ora.attention_head_ref(q, k, v, scale, True, window=w)
        return float((o * do).sum())
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss()
            x[idx] = old - h
            lm = loss()
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_window_at_least_n_and_sampled():
    """window >= N is the causal backward; the sampled form equals the full
    one with a window."""
    q, k, v, do = _case(40, 4, 50, std=1.2)
    a = ora.attention_bwd_head_ref(q, k, v, do, 0.5, True)
    b = ora.attention_bwd_head_ref(q, k, v, do, 0.5, True, window=40)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    full = ora.attention_bwd_head_ref(q, k, v, do, 0.5, True, window=7)
    pick = [0, 5, 6, 7, 20, 39]
    sq, sk, sv = ora.attention_bwd_sampled_ref(q, k, v, do, 0.5, True, pick, pick, chunk=16,
                                               window=7)
    np.testing.assert_allclose(sq, full[0][pick], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sk, full[1][pick], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sv, full[2][pick], rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_given_output_shifts_delta_only(causal):
    """A backward call is handed the forward output o and forms Delta_i =
    dO_i . o_i from it.  With o = O + E (E a perturbation, e.g. the rounding
    of O to bf16) only Delta moves, by -dO_i . E_i, so in closed form
        dV' = dV,
        dQ'_i = dQ_i + scale (Delta_i - Delta'_i) sum_j P_ij k_j,
        dK'_j = dK_j + scale sum_i P_ij (Delta_i - Delta'_i) q_i,
    with P the softmax of the scores, here from torch in float64; the
    unperturbed gradients are pinned by finite differences above.  The
    sampled form with o_given agrees with the full form."""
    N, D, scale = 40, 8, 0.45
    q, k, v, do = _case(N, D, 21 + causal, std=1.3)
    rng = np.random.default_rng(5)
    o_exact, _ = ora.attention_head_ref(q, k, v, scale, causal)
    o_given = o_exact + 1e-3 * rng.standard_normal(o_exact.shape)
    dq, dk, dv, delta = ora.attention_bwd_head_ref(q, k, v, do, scale, causal)
    dq2, dk2, dv2, delta2 = ora.attention_bwd_head_ref(q, k, v, do, scale, causal, o=o_given)
    s = torch.from_numpy(q @ k.T * scale)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    p = torch.softmax(s, dim=-1).numpy()
    shift = delta - delta2
    np.testing.assert_allclose(delta2, (do * o_given).sum(1), rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(dv2, dv)
    np.testing.assert_allclose(dq2, dq + scale * shift[:, None] * (p @ k), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dk2, dk + scale * (p * shift[:, None]).T @ q, rtol=1e-9,
                               atol=1e-12)
    picks = [0, 1, 17, N - 1]
    sq, sk, sv = ora.attention_bwd_sampled_ref(q, k, v, do, scale, causal, picks, picks,
                                               chunk=16, o_given=o_given)
    np.testing.assert_allclose(sq, dq2[picks], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sk, dk2[picks], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sv, dv2[picks], rtol=1e-10, atol=1e-12)
