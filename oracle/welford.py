"""Float64 oracle of per-row mean / variance statistics: the Welford carrier
(n, mu, M2) and its Chan-Golub-LeVeque merge.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's CPU baseline, never by the library.

Sources: "Learning FlashAttention the Hard Way - Part 1" (cloudrift.ai),
sections "The Same Move: Welford's Variance" (the carrier, the single-sample
injection (1, x, 0), the streaming update, the symmetric merge with identity
(0, 0, 0), and the final division by n or n - 1), "Why Welford's Combine
Associates" (the merge in deviation form) and "Welford, the Easy Way" (the
carrier as a twist of the three plain sums (n, T, W) = (n, sum x, sum x^2)).
The page's formulas were stripped from the extracted text; the ones below are
the standard forms its prose describes:
    update:  n' = n + 1,  delta = x - mu,  mu' = mu + delta / n',
             M2' = M2 + delta * (x - mu')
    merge:   n = n_a + n_b,  delta = mu_b - mu_a,
             mu = mu_a + delta * n_b / n,
             M2 = M2_a + M2_b + delta^2 * n_a * n_b / n
    twist:   (n, T, W) -> (n, T / n, W - T^2 / n)
Rows are split into column chunks the same way as split-KV decode: chunk c
of S over a length-C row covers [c * ceil(C/S), min(C, (c+1) * ceil(C/S))).
"""
from __future__ import annotations

import numpy as np

IDENTITY = (0.0, 0.0, 0.0)


def inject(x):
    """One sample as a state."""
    return (1.0, float(x), 0.0)


def update(state, x):
    """Fold one more sample into the running state (the streaming form)."""
    n, mu, m2 = state
    n1 = n + 1.0
    delta = float(x) - mu
    mu1 = mu + delta / n1
    return (n1, mu1, m2 + delta * (float(x) - mu1))


def merge(a, b):
    """The associative combine of two states over disjoint samples."""
    na, mua, m2a = a
    nb, mub, m2b = b
    if nb == 0:
        return a
    if na == 0:
        return b
    n = na + nb
    delta = mub - mua
    return (n, mua + delta * nb / n, m2a + m2b + delta * delta * na * nb / n)


def fold_left(states):
    acc = IDENTITY
    for s in states:
        acc = merge(acc, s)
    return acc


def finalize(state, ddof=0):
    """Mean and variance M2 / (n - ddof) (ddof 0: population, 1: sample)."""
    n, mu, m2 = state
    return mu, m2 / (n - ddof)


def twist(n, t, w):
    """The plain sums (n, T, W) mapped to the carrier."""
    if n == 0:
        return IDENTITY
    return (n, t / n, w - t * t / n)


def untwist(state):
    n, mu, m2 = state
    return (n, n * mu, m2 + n * mu * mu)


def two_pass(x):
    """The definition: mu = sum x / n, then M2 = sum (x - mu)^2."""
    x = np.asarray(x, dtype=np.float64)
    n = x.size
    if n == 0:
        return IDENTITY
    mu = x.sum() / n
    return (float(n), float(mu), float(((x - mu) ** 2).sum()))


def chunk_bounds(C, S):
    step = -(-C // S) if C > 0 else 0
    return [(min(C, c * step), min(C, (c + 1) * step)) for c in range(S)]


def to_f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def row_stats_ref(x, eps=0.0):
    """Per row of a [R, C] matrix: mean, population variance and
    1 / sqrt(var + eps) (the LayerNorm statistics), from the two-pass
    definition in float64."""
    x = to_f64(x)
    mu = x.mean(axis=1)
    var = ((x - mu[:, None]) ** 2).mean(axis=1)
    return mu, var, 1.0 / np.sqrt(var + eps)


def chunk_states_ref(x, S):
    """Per row, the states of its S column chunks (two-pass per chunk):
    arrays n, mu, M2 of shape [R, S]."""
    x = to_f64(x)
    R, C = x.shape
    n = np.zeros((R, S))
    mu = np.zeros((R, S))
    m2 = np.zeros((R, S))
    for c, (lo, hi) in enumerate(chunk_bounds(C, S)):
        if hi > lo:
            blk = x[:, lo:hi]
            n[:, c] = hi - lo
            mu[:, c] = blk.mean(axis=1)
            m2[:, c] = ((blk - mu[:, c:c + 1]) ** 2).sum(axis=1)
    return n, mu, m2


def combine_ref(n, mu, m2, eps=0.0):
    """Left fold of each row's chunk states (index order), then mean,
    population variance and 1 / sqrt(var + eps)."""
    R, S = n.shape
    out_mu = np.zeros(R)
    out_var = np.zeros(R)
    for r in range(R):
        st = fold_left((n[r, c], mu[r, c], m2[r, c]) for c in range(S))
        out_mu[r], out_var[r] = finalize(st)
    return out_mu, out_var, 1.0 / np.sqrt(out_var + eps)
