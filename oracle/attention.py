"""Float64 CPU definitions of exact attention and of the (m, d, o) state.

Test infrastructure only (see the package docstring): plain, slow and written
to be checked against the pages by eye.  No tiling, fusion or reordering
beyond what each definition states; NumPy's matmul serves as the dot-product
step.

Page: "Learning FlashAttention the Hard Way - Part 1" (cloudrift.ai).
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np

LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)


def to_f64(x) -> np.ndarray:
    """Exact conversion of a (torch or NumPy) bf16/fp32 tensor to float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Dense attention: the plain definition.
# Section "FlashAttention: Not So Special": S = Q K^T, P = softmax(S) row-wise,
# O = P V, with S never needed by the tiled method but materialised here.
# Section "Softmax Looks Like It Breaks the Rules": the safe softmax subtracts
# the row maximum m before exponentiating and divides by d = sum_j e^{s_j - m}.
# ---------------------------------------------------------------------------

def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = (Q K^T) * scale for one head: q [Nq, D], k [Nk, D] -> [Nq, Nk]."""
    return (q @ k.T) * float(scale)


def causal_mask(s: np.ndarray, q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """Key j is hidden from query i when j > i (positions within a sequence)."""
    s = s.copy()
    s[k_pos[None, :] > q_pos[:, None]] = -np.inf
    return s


def safe_softmax_stats(s: np.ndarray):
    """Row maximum m, shifted weights e^{s - m} and their sum d (three passes:
    max, sum, divide - the last one left to the caller).  A row whose entries
    are all -inf has no maximum; it gets m = -inf, weights 0, d = 0."""
    m = s.max(axis=-1, initial=-np.inf)  # an empty block is the identity
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(s - m_safe[..., None])
    d = w.sum(axis=-1)
    return m, w, d


def softmax_ref(s: np.ndarray) -> np.ndarray:
    """Row-wise safe softmax P = e^{s - m} / d."""
    _, w, d = safe_softmax_stats(s)
    return w / d[..., None]


def window_mask(s: np.ndarray, q_pos: np.ndarray, k_pos: np.ndarray, window: int) -> np.ndarray:
    """Sliding window: key j is hidden from query i when j <= i - window, so
    with the causal mask query i sees keys i - window + 1 .. i."""
    s = s.copy()
    s[k_pos[None, :] <= q_pos[:, None] - int(window)] = -np.inf
    return s


def attention_head_ref(q, k, v, scale, causal, rows=None, window=None):
    """One head.  q [Nq, D], k/v [Nk, D] float64; Nq == Nk when causal.
    Returns O [R, D] and LSE [R] (natural log) for the query rows ``rows``
    (all rows when None).  ``window`` (with causal) keeps only the last
    ``window`` keys of each row.  A fully masked row gives O = 0 and
    LSE = -inf."""
    nq = q.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    s = scores(q[rows], k, scale)
    if causal:
        s = causal_mask(s, rows, np.arange(k.shape[0]))
    if window is not None:
        s = window_mask(s, rows, np.arange(k.shape[0]), window)
    m, w, d = safe_softmax_stats(s)
    num = w @ v
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(d[:, None] > 0, num / np.where(d > 0, d, 1.0)[:, None], 0.0)
        lse = np.where(d > 0, m + np.log(np.where(d > 0, d, 1.0)), -np.inf)
    return o, lse


def attention_ref(q, k, v, scale, causal, rows=None, window=None):
    """Dense [B, H, N, D] inputs (any dtype, converted exactly to float64).
    Returns O [B, H, R, D] and LSE [B, H, R] in float64, looping over heads so
    that at most one head's score matrix is held at a time."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, D = q.shape
    R = N if rows is None else len(rows)
    O = np.zeros((B, H, R, D))
    L = np.zeros((B, H, R))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = attention_head_ref(q[b, h], k[b, h], v[b, h],
                                                  scale, causal, rows, window)
    return O, L


def attention_bwd_head_ref(q, k, v, do, scale, causal, window=None, o=None):
    """Gradients of one head's attention with respect to q, k, v, given the
    output gradient do (all [N, D] float64).  Recomputation, as the tiled
    backward does it: P is rebuilt from the scores and the row log-sum-exp
    (P = e^{S - LSE}), never stored.  With O = P V and S = scale Q K^T:
        dV = P^T dO,  dP = dO V^T,  Delta_i = sum_j P_ij dP_ij = dO_i . O_i,
        dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q.
    ``window`` (with causal): the sliding window of attention_head_ref.
    ``o``: the forward output a backward call is handed ([N, D]); Delta is
    then formed as dO_i . o_i from it, as such a call defines it.  None (the
    default) uses this oracle's own exact O, which gives the exact gradient.
    Returns dq, dk, dv and Delta."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    n = q.shape[0]
    o_own, lse = attention_head_ref(q, k, v, scale, causal, window=window)
    o = o_own if o is None else to_f64(o)
    s = scores(q, k, scale)
    if causal:
        s = causal_mask(s, np.arange(n), np.arange(k.shape[0]))
    if window is not None:
        s = window_mask(s, np.arange(n), np.arange(k.shape[0]), window)
    p = np.exp(s - lse[:, None])  # rows with no visible key do not occur
    dv = p.T @ do
    dp = do @ v.T
    delta = (do * o).sum(axis=1)
    ds = p * (dp - delta[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, delta


def attention_bwd_sampled_ref(q, k, v, do, scale, causal, rows, cols, chunk=1024,
                              window=None, o_given=None):
    """Selected gradient rows of one head, for heads too long for the full
    matrices: dq at the query rows `rows`, dk and dv at the key rows `cols`.
    O and LSE of every query row come from attention_head_ref over row
    chunks; then, per query row i, the row of P and dP; per key row j, the
    column of P and dP (P_ij = e^{s_ij - LSE_i}, hidden keys 0).  The same
    formulas as attention_bwd_head_ref, evaluated one row or column at a time.
    ``o_given``: as ``o`` of attention_bwd_head_ref (Delta from the forward
    output the call is handed; None: this oracle's own O).
    Returns dq[len(rows), D], dk[len(cols), D], dv[len(cols), D]."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    n = q.shape[0]
    o = np.zeros_like(q)
    lse = np.zeros(n)
    for r0 in range(0, n, chunk):
        r = np.arange(r0, min(n, r0 + chunk))
        o[r], lse[r] = attention_head_ref(q, k, v, scale, causal, rows=r, window=window)
    if o_given is not None:
        o = to_f64(o_given)
    delta = (do * o).sum(axis=1)
    pos = np.arange(n)
    dq = np.zeros((len(rows), q.shape[1]))
    for t, i in enumerate(rows):
        s = scale * (k @ q[i])
        vis = pos <= i if causal else np.ones(n, dtype=bool)
        if window is not None:
            vis = vis & (pos > i - window)
        p = np.where(vis, np.exp(s - lse[i]), 0.0)
        ds = p * (v @ do[i] - delta[i])
        dq[t] = scale * (ds @ k)
    dk = np.zeros((len(cols), q.shape[1]))
    dv = np.zeros((len(cols), q.shape[1]))
    for t, j in enumerate(cols):
        s = scale * (q @ k[j])
        vis = pos >= j if causal else np.ones(n, dtype=bool)
        if window is not None:
            vis = vis & (pos < j + window)
        p = np.where(vis, np.exp(s - lse), 0.0)
        ds = p * (do @ v[j] - delta)
        dv[t] = p @ do
        dk[t] = scale * (ds @ q)
    return dq, dk, dv


def attention_bwd_ref(q, k, v, do, scale, causal, window=None, o=None):
    """[B, H, N, D] inputs (any dtype, converted exactly to float64); returns
    dq, dk, dv [B, H, N, D] and Delta [B, H, N] in float64.  ``o``
    ([B, H, N, D] or None): as in attention_bwd_head_ref."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    o = None if o is None else to_f64(o)
    B, H, N, D = q.shape
    dq, dk, dv = (np.zeros((B, H, N, D)) for _ in range(3))
    delta = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h], delta[b, h] = attention_bwd_head_ref(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, window=window,
                o=None if o is None else o[b, h])
    return dq, dk, dv, delta


def varlen_ref(q, k, v, cu_seqlens, scale, causal, seqs=None, rows=None):
    """Packed [T, H, D] inputs with sequence i on tokens
    [cu_seqlens[i], cu_seqlens[i+1]).  Each sequence is its own dense
    attention (positions restart at 0).  Returns {seq: (O [L', H, D],
    LSE [H, L'])} for the chosen sequences (all by default) and query rows
    (local indices, all by default)."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    cu = [int(x) for x in np.asarray(cu_seqlens).tolist()]
    seqs = range(len(cu) - 1) if seqs is None else seqs
    H = q.shape[1]
    out = {}
    for i in seqs:
        a, b = cu[i], cu[i + 1]
        Ls = b - a
        r = np.arange(Ls) if rows is None else np.asarray(
            [x for x in rows if x < Ls], dtype=np.int64)
        O = np.zeros((len(r), H, q.shape[2]))
        LSE = np.zeros((H, len(r)))
        for h in range(H):
            o, l = attention_head_ref(q[a:b, h], k[a:b, h], v[a:b, h], scale,
                                      causal, r)
            O[:, h], LSE[h] = o, l
        out[i] = (O, LSE)
    return out


def decode_ref(q, k_cache, v_cache, cu_seqlens_k, scale, batch=None, heads=None):
    """One query row per sequence, attending to every key of its sequence
    (the newest token sees the whole cache, so there is no mask).
    q [B, H, D]; caches packed [T_k, H, D].  Returns O [B, H, D] and
    LSE [B, H] for the chosen (batch, head) items (others left as NaN)."""
    q, kc, vc = to_f64(q), to_f64(k_cache), to_f64(v_cache)
    cu = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    B, H, D = q.shape
    O = np.full((B, H, D), np.nan)
    LSE = np.full((B, H), np.nan)
    for b in (range(B) if batch is None else batch):
        a, e = cu[b], cu[b + 1]
        for h in (range(H) if heads is None else heads):
            o, l = attention_head_ref(q[b, h][None, :], kc[a:e, h], vc[a:e, h],
                                      scale, False)
            O[b, h], LSE[b, h] = o[0], l[0]
    return O, LSE


def paged_kv_gather(k_pages, v_pages, block_table, seqlen: int, b: int):
    """The KV cache of sequence b as contiguous [L, H_kv, D] arrays: key t
    lives in page block_table[b][t // page_size], row t % page_size.
    Pages are [num_pages, page_size, H_kv, D]."""
    page = k_pages.shape[1]
    idx = np.arange(seqlen)
    pages = np.asarray(block_table)[b][idx // page]
    return k_pages[pages, idx % page], v_pages[pages, idx % page]


def decode_paged_ref(q, k_pages, v_pages, block_table, seqlens, scale,
                     batch=None, heads=None):
    """One query row per sequence against its paged KV cache, with grouped
    query heads: query head h reads KV head h // (H / H_kv).
    q [B, H, D]; pages [P, page_size, H_kv, D]; block_table [B, max_blocks];
    seqlens [B].  Returns O [B, H, D], LSE [B, H] (unselected items NaN)."""
    q, kp, vp = to_f64(q), to_f64(k_pages), to_f64(v_pages)
    B, H, D = q.shape
    Hkv = kp.shape[2]
    group = H // Hkv
    O = np.full((B, H, D), np.nan)
    LSE = np.full((B, H), np.nan)
    for b in (range(B) if batch is None else batch):
        kc, vc = paged_kv_gather(kp, vp, block_table, int(seqlens[b]), b)
        for h in (range(H) if heads is None else heads):
            o, l = attention_head_ref(q[b, h][None, :], kc[:, h // group],
                                      vc[:, h // group], scale, False)
            O[b, h], LSE[b, h] = o[0], l[0]
    return O, LSE


def chunk_states_paged_ref(q, k_pages, v_pages, block_table, seqlens, num_splits,
                           scale, batch=None, heads=None, align=1):
    """Base-2 chunk states of split-KV decode over a paged cache with grouped
    query heads (chunking as chunk_bounds, chunk length rounded up to a
    multiple of ``align`` keys).  Shapes as chunk_states_ref."""
    q, kp, vp = to_f64(q), to_f64(k_pages), to_f64(v_pages)
    B, H, D = q.shape
    group = H // kp.shape[2]
    S = int(num_splits)
    M = np.full((B, H, S), np.nan)
    Dn = np.full((B, H, S), np.nan)
    Ot = np.full((B, H, S, D), np.nan)
    for b in (range(B) if batch is None else batch):
        L = int(seqlens[b])
        kc, vc = paged_kv_gather(kp, vp, block_table, L, b)
        for h in (range(H) if heads is None else heads):
            for c, (a, e) in enumerate(chunk_bounds(L, S, align)):
                sig = (kc[a:e, h // group] @ q[b, h]) * (float(scale) * LOG2E)
                M[b, h, c], Dn[b, h, c], Ot[b, h, c] = row_state(
                    sig, vc[a:e, h // group], base=2.0)
    return M, Dn, Ot


# ---------------------------------------------------------------------------
# The state u = (m, d, o) and its merge.
# Section "The State": over a block of keys, m is the running maximum score,
# d = sum e^{s_j - m} and o = sum e^{s_j - m} v_j (unnormalised output row).
# A single pair (s_j, v_j) enters as (s_j, 1, v_j); the row is read off at the
# end as o / d.
# Section "The Merge, and the Twist": keep the larger maximum and shrink the
# other side toward it, so the exponent is never positive.  Identity
# (-inf, 0, 0) (section "Why Attention's Combine Still Associates").
# Section "Alternative Twist: Base 2": the same monoid over sigma = s log2(e)
# with 2^x in place of e^x.
# ---------------------------------------------------------------------------

def identity(D: int):
    return (-math.inf, 0.0, np.zeros(D))


def inject(s: float, v: np.ndarray):
    """A single key/value pair as a state: (s, 1, v)."""
    return (float(s), 1.0, np.asarray(v, dtype=np.float64).copy())


def merge(a, b, base: float = math.e):
    """(m_a, d_a, o_a) (+) (m_b, d_b, o_b), case-split on the larger max.
    With the identity on either side the other operand is returned (the
    -inf - (-inf) case has no value; it is defined by the identity law)."""
    ma, da, oa = a
    mb, db, ob = b
    if mb == -math.inf:
        return (ma, da, np.array(oa, dtype=np.float64))
    if ma == -math.inf:
        return (mb, db, np.array(ob, dtype=np.float64))
    if ma >= mb:
        f = base ** (mb - ma)
        return (ma, da + db * f, oa + ob * f)
    f = base ** (ma - mb)
    return (mb, da * f + db, oa * f + ob)


def fold_left(states, D: int, base: float = math.e):
    acc = identity(D)
    for u in states:
        acc = merge(acc, u, base)
    return acc


def fold_tree(states, tree, base: float = math.e):
    """Fold following an explicit bracketing: ``tree`` is an int (a leaf
    index) or a pair (left_tree, right_tree)."""
    if isinstance(tree, int):
        return states[tree]
    l, r = tree
    return merge(fold_tree(states, l, base), fold_tree(states, r, base), base)


def finalize(state, base: float = math.e):
    """Output row o / d and log-sum-exp in natural log: ln(base) * m + ln d."""
    m, d, o = state
    if d == 0.0:
        return np.zeros_like(o), -math.inf
    return o / d, math.log(base) * m + math.log(d)


def row_state(s: np.ndarray, v: np.ndarray, base: float = math.e):
    """The state of a whole block by its definition (no merging):
    m = max s, d = sum base^{s - m}, o = sum base^{s - m} v."""
    if s.size == 0:
        return identity(v.shape[-1])
    m = float(s.max())
    if m == -math.inf:
        return identity(v.shape[-1])
    w = np.power(base, s - m)
    return (m, float(w.sum()), w @ v)


# ---------------------------------------------------------------------------
# Split-KV decode: chunk states and their combine.
# Section "Associativity is All You Need": split-K lets separate thread blocks
# own chunks, write partial results to scratch and fold them in a small second
# kernel; "The Merge, and the Twist" gives the fold.  Chunking reading: chunk c
# of a length-L sequence covers keys [c*ceil(L/S), min(L, (c+1)*ceil(L/S))),
# possibly empty.  States are kept in the base-2 coordinates
# (sigma = s * log2(e)).
# ---------------------------------------------------------------------------

def chunk_bounds(L: int, num_splits: int, align: int = 1):
    """Chunk c covers keys [c*C, min(L, (c+1)*C)), C = ceil(L / num_splits)
    rounded up to a multiple of ``align`` (1: no rounding)."""
    size = -(-L // num_splits) if L > 0 else 0
    size = -(-size // align) * align
    out = []
    for c in range(num_splits):
        a = min(L, c * size)
        b = min(L, (c + 1) * size)
        out.append((a, b))
    return out


def chunk_states_ref(q, k_cache, v_cache, cu_seqlens_k, num_splits, scale,
                     batch=None, heads=None):
    """Base-2 states (m2, d, o) of every KV chunk of every (b, h).
    Returns m2 [B, H, S], d [B, H, S], o [B, H, S, D] float64; empty chunks hold
    the identity (-inf, 0, 0).  Items not selected are NaN."""
    q, kc, vc = to_f64(q), to_f64(k_cache), to_f64(v_cache)
    cu = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    B, H, D = q.shape
    S = int(num_splits)
    M = np.full((B, H, S), np.nan)
    Dn = np.full((B, H, S), np.nan)
    Ot = np.full((B, H, S, D), np.nan)
    for b in (range(B) if batch is None else batch):
        a0 = cu[b]
        L = cu[b + 1] - a0
        for h in (range(H) if heads is None else heads):
            for c, (a, e) in enumerate(chunk_bounds(L, S)):
                sig = (kc[a0 + a:a0 + e, h] @ q[b, h]) * (float(scale) * LOG2E)
                m, d, o = row_state(sig, vc[a0 + a:a0 + e, h], base=2.0)
                M[b, h, c], Dn[b, h, c], Ot[b, h, c] = m, d, o
    return M, Dn, Ot


def combine_ref(m2, d, o):
    """Fold the base-2 chunk states of each row left to right (chunk 0 first)
    and finalise: O = o / d, LSE = ln2 * (m2 + log2 d).
    m2, d: [..., S]; o: [..., S, D].  Returns O [..., D], LSE [...]."""
    m2 = np.asarray(m2, dtype=np.float64)
    d = np.asarray(d, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    lead = m2.shape[:-1]
    S = m2.shape[-1]
    D = o.shape[-1]
    Ofl = np.zeros(lead + (D,))
    Lfl = np.zeros(lead)
    for idx in np.ndindex(*lead):
        acc = identity(D)
        for c in range(S):
            acc = merge(acc, (float(m2[idx + (c,)]), float(d[idx + (c,)]),
                              o[idx + (c,)]), base=2.0)
        Ofl[idx], Lfl[idx] = finalize(acc, base=2.0)
    return Ofl, Lfl


# ---------------------------------------------------------------------------
# Enumeration helpers for the associativity pins (brute force, tiny N).
# ---------------------------------------------------------------------------

def all_bracketings(lo: int, hi: int):
    """Every full binary bracketing of leaves lo..hi-1 (Catalan many)."""
    if hi - lo == 1:
        return [lo]
    out = []
    for mid in range(lo + 1, hi):
        for left in all_bracketings(lo, mid):
            for right in all_bracketings(mid, hi):
                out.append((left, right))
    return out


def all_chunkings(n: int) -> list[list[tuple[int, int]]]:
    """Every split of 0..n-1 into contiguous non-empty chunks (2^(n-1))."""
    out = []
    for mask in range(1 << (n - 1)):
        cuts = [0] + [i + 1 for i in range(n - 1) if mask >> i & 1] + [n]
        out.append([(cuts[i], cuts[i + 1]) for i in range(len(cuts) - 1)])
    return out


# ---------------------------------------------------------------------------
# Prefix scan of the (m, d, o) monoid.  "Learning FlashAttention the Hard Way
# - Part 1", section "Why Attention's Combine Still Associates", ties the
# monoid to running exact attention as a parallel prefix scan (the ELSA
# reference, O(log n) depth).  Read here as: for one query vector against a
# sequence of keys, the inclusive scan of the keys' states gives, at every
# position i, the attention over keys 0..i.


def scan_left(states, D: int, base: float = math.e):
    """Inclusive scan by a left fold: prefix i = s_0 (+) ... (+) s_i."""
    out = []
    acc = identity(D)
    for u in states:
        acc = merge(acc, u, base)
        out.append(acc)
    return out


def scan_tree(states, D: int, base: float = math.e):
    """The same prefixes by the two-sweep tree scan (O(log n) depth): the
    up-sweep stores subtree totals at the right child of every pair, the
    down-sweep hands each node the total of everything to its left, and the
    inclusive prefix is that exclusive prefix (+) the element."""
    n = len(states)
    size = 1
    while size < n:
        size *= 2
    t = list(states) + [identity(D) for _ in range(size - n)]
    step = 1
    while step < size:
        for i in range(2 * step - 1, size, 2 * step):
            t[i] = merge(t[i - step], t[i], base)
        step *= 2
    t[size - 1] = identity(D)
    step = size // 2
    while step >= 1:
        for i in range(2 * step - 1, size, 2 * step):
            left = t[i - step]
            t[i - step] = t[i]
            t[i] = merge(t[i], left, base)
        step //= 2
    return [merge(t[i], states[i], base) for i in range(n)]


def prefix_attention_ref(q, k_cache, v_cache, cu_seqlens_k, scale, batch=None, heads=None,
                         positions=None):
    """For every sequence b and head h, the attention of q[b, h] over keys
    0..i of the sequence, at every position i (or at the in-sequence
    positions listed in ``positions[b]``), by the plain definition on each
    prefix.  q [B, H, D]; caches packed [T_k, H, D].  Returns O [T_k, H, D]
    and LSE [H, T_k] (natural log); entries not computed are NaN."""
    q, kc, vc = to_f64(q), to_f64(k_cache), to_f64(v_cache)
    cu = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    B, H, D = q.shape
    T = kc.shape[0]
    O = np.full((T, H, D), np.nan)
    LSE = np.full((H, T), np.nan)
    for b in (range(B) if batch is None else batch):
        a, e = cu[b], cu[b + 1]
        pos = range(e - a) if positions is None else positions[b]
        for h in (range(H) if heads is None else heads):
            for i in pos:
                s = scores(q[b, h][None, :], kc[a:a + i + 1, h], scale)[0]
                m = s.max()
                w = np.exp(s - m)
                O[a + i, h] = (w @ vc[a:a + i + 1, h]) / w.sum()
                LSE[h, a + i] = m + math.log(w.sum())
    return O, LSE


def attention_bwd_varlen_ref(q, k, v, do, cu_seqlens, scale, causal, o=None):
    """Backward over packed sequences: q, k, v, do [T, H, D]; sequence s owns
    tokens [cu[s], cu[s+1]).  Every (sequence, head) is an independent head
    of attention_bwd_head_ref.  ``o`` ([T, H, D] or None): as in
    attention_bwd_head_ref.  Returns dq, dk, dv [T, H, D] and Delta [H, T]
    in float64."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    o = None if o is None else to_f64(o)
    cu = [int(x) for x in np.asarray(cu_seqlens).tolist()]
    T, H, D = q.shape
    dq, dk, dv = (np.zeros((T, H, D)) for _ in range(3))
    delta = np.zeros((H, T))
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        if e == a:
            continue
        for h in range(H):
            g = attention_bwd_head_ref(q[a:e, h], k[a:e, h], v[a:e, h], do[a:e, h], scale, causal,
                                       o=None if o is None else o[a:e, h])
            dq[a:e, h], dk[a:e, h], dv[a:e, h], delta[h, a:e] = g
    return dq, dk, dv, delta
