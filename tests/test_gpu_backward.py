"""GPU parity of the backward by recomputation (fa_bwd through the binding)
against the float64 oracle on the same seeded inputs: small shapes element by
element, the full-size causal head on sampled rows and columns, the
degenerate scale 0, determinism and argument checks.

The backward is handed the forward's O and LSE.  In the parity tests these
come from the oracle's forward, rounded as a bf16 forward returns them (O to
bf16, LSE to fp32), so no oracle input comes from the GPU.  Each gradient is
checked row by row against the oracle's gradient formed with that same bf16
O (Delta_i = dO_i . O_i, as the call defines it), and as a tensor against
the exact gradient (Delta from the exact O)."""
import ctypes

import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from tests.gpu_common import check_grad, check_grad_exact, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _run(fa, case, do):
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    o, lse = fa.fa_fwd(q, k, v, case.scale, case.causal)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do.cuda(), lse, case.scale, case.causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    return dq, dk, dv


def _oracle_fwd(q, k, v, scale, causal, window=None):
    """The oracle's O and LSE, rounded as a bf16 forward returns them."""
    O, L = ora.attention_ref(q, k, v, scale, causal, window=window)
    return torch.from_numpy(O).to(torch.bfloat16), torch.from_numpy(L).to(torch.float32)


def _check_both(grads, ref_given, ref_exact, tag):
    for name, g, rg, re in zip(("dq", "dk", "dv"), grads, ref_given, ref_exact):
        check_grad(np64(g), rg, f"{name} {tag}")
        check_grad_exact(np64(g), re, f"{name} {tag} (exact gradient)")


def _bwd_dense_checked(fa, case, do, causal, tag, window=None):
    o_in, lse_in = _oracle_fwd(case.q, case.k, case.v, case.scale, causal, window)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    if window is None:
        g = fa.fa_bwd(q, k, v, o_in.cuda(), do.cuda(), lse_in.cuda(), case.scale, causal)
    else:
        g = fa.fa_bwd_window(q, k, v, o_in.cuda(), do.cuda(), lse_in.cuda(), window, case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    rg = ora.attention_bwd_ref(case.q, case.k, case.v, do, case.scale, causal, window=window,
                               o=o_in)[:3]
    re = ora.attention_bwd_ref(case.q, case.k, case.v, do, case.scale, causal,
                               window=window)[:3]
    _check_both(g, rg, re, tag)
    return g


SHAPES = [
    # (B, H, N, D, causal): one row, exact tiles, ragged tails, both head dims
    (1, 1, 1, 64, False),
    (1, 1, 1, 128, True),
    (1, 2, 128, 128, True),
    (1, 2, 129, 64, True),
    (2, 1, 300, 128, False),
    (2, 2, 256, 64, True),
    (1, 2, 517, 128, True),
    (1, 1, 640, 64, False),
]


@pytest.mark.parametrize("B,H,N,D,causal", SHAPES)
def test_bwd_small(fa, B, H, N, D, causal):
    case = inp.dense(B, H, N, D, seed=900 + N + D, causal=causal)
    do = inp.output_grad((B, H, N, D), seed=901 + N)
    _bwd_dense_checked(fa, case, do, causal, (B, H, N, D, causal))


def test_bwd_large_scores(fa):
    """q, k with std 2 (peaked softmax rows, large LSE)."""
    case = inp.dense(1, 2, 384, 128, seed=930, causal=True, qk_std=2.0)
    do = inp.output_grad((1, 2, 384, 128), seed=931)
    _bwd_dense_checked(fa, case, do, True, "std2")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_scale_zero(fa, causal):
    """scale 0: uniform weights, dQ = dK = 0 exactly, dV = P^T dO."""
    case = inp.dense(1, 2, 200, 64, seed=940, causal=causal, scale=0.0)
    do = inp.output_grad((1, 2, 200, 64), seed=941)
    dq, dk, dv = _run(fa, case, do)
    assert not dq.any() and not dk.any()
    _, _, rv, _ = ora.attention_bwd_ref(case.q, case.k, case.v, do, 0.0, causal)
    check_grad_exact(np64(dv), rv, "dv scale0")
    check_grad(np64(dv), rv, "dv scale0")  # dV does not depend on Delta


def test_bwd_deterministic(fa):
    case = inp.dense(1, 4, 700, 128, seed=950, causal=True)
    do = inp.output_grad((1, 4, 700, 128), seed=951)
    a = _run(fa, case, do)
    b = _run(fa, case, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_full_size_sampled(fa):
    """The causal prefill workload (B=1, H=32, N=16384, D=128): heads 0 and 31,
    dq at sampled query rows, dk and dv at sampled key rows (tile edges, both
    ends, random interior)."""
    B, H, N, D = 1, 32, 16384, 128
    case = inp.dense(B, H, N, D, seed=960, causal=True)
    do = inp.output_grad((B, H, N, D), seed=961)
    rng = np.random.default_rng(962)
    picks = sorted(set([0, 1, 127, 128, 8191, 8192, N - 129, N - 128, N - 1]) |
                   set(rng.integers(0, N, 23).tolist()))
    _full_size_sampled(fa, case, do, picks, "")


def _full_size_sampled(fa, case, do, picks, tag, window=None):
    """Heads 0 and H-1 of a [1, H, N, D] problem: their O and LSE from the
    oracle (rounded as the bf16 forward returns them), the other heads' from
    the GPU forward (not checked); sampled rows of dq, dk, dv against both
    oracle gradients."""
    B, H, N, D = case.q.shape
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    if window is None:
        o, lse = fa.fa_fwd(q, k, v, case.scale, True)
    else:
        o, lse = fa.fa_fwd_window(q, k, v, window, case.scale)
    heads = (0, H - 1)
    o_in = {}
    for h in heads:
        O = np.zeros((N, D))
        L = np.zeros(N)
        for r0 in range(0, N, 2048):
            r = np.arange(r0, min(N, r0 + 2048))
            O[r], L[r] = ora.attention_head_ref(ora.to_f64(case.q[0, h]), ora.to_f64(case.k[0, h]),
                                                ora.to_f64(case.v[0, h]), case.scale, True,
                                                rows=r, window=window)
        o_in[h] = torch.from_numpy(O).to(torch.bfloat16)
        o[0, h] = o_in[h].cuda()
        lse[0, h] = torch.from_numpy(L).to(torch.float32).cuda()
    if window is None:
        dq, dk, dv = fa.fa_bwd(q, k, v, o, do.cuda(), lse, case.scale, True)
    else:
        dq, dk, dv = fa.fa_bwd_window(q, k, v, o, do.cuda(), lse, window, case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    for h in heads:
        args = (case.q[0, h], case.k[0, h], case.v[0, h], do[0, h], case.scale, True, picks, picks)
        rg = ora.attention_bwd_sampled_ref(*args, window=window, o_given=o_in[h])
        re = ora.attention_bwd_sampled_ref(*args, window=window)
        got = (dq[0, h, picks], dk[0, h, picks], dv[0, h, picks])
        _check_both(got, rg, re, f"{tag}head {h}")


def test_bwd_invalid_args(fa):
    lib = fa.load_library()
    x = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 64), dtype=torch.float32, device="cuda")
    ws = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    args = [p, p, p, p, p, lse.data_ptr(), p, p, p, ws.data_ptr()]
    # head dim 96
    assert lib.fa_bwd(*args, 1, 1, 64, 96, 0.1, 1, s) == fa.FA_ERR_INVALID_ARG
    # misaligned dO
    bad = list(args)
    bad[4] = p + 2
    assert lib.fa_bwd(*bad, 1, 1, 64, 128, 0.1, 1, s) == fa.FA_ERR_INVALID_ARG
    # negative scale, NULL dq
    assert lib.fa_bwd(*args, 1, 1, 64, 128, -1.0, 1, s) == fa.FA_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = None
    assert lib.fa_bwd(*bad, 1, 1, 64, 128, 0.1, 1, s) == fa.FA_ERR_INVALID_ARG
    # empty problem: FA_OK, nothing touched
    assert lib.fa_bwd(None, None, None, None, None, None, None, None, None, None,
                      1, 1, 0, 128, 0.1, 1, s) == fa.FA_OK
    assert lib.fa_bwd_workspace_bytes(2, 3, 5) == 2 * 3 * 5 * 4


# --- packed sequences -------------------------------------------------------------

def _varlen_checked(fa, case, do, causal, tag):
    """Packed backward on the oracle's O and LSE (rounded as the bf16
    forward returns them), checked against both oracle gradients."""
    T, H, D = case.q.shape
    ref = ora.varlen_ref(case.q, case.k, case.v, case.cu_seqlens, case.scale, causal)
    cuh = case.cu_seqlens.tolist()
    O = np.zeros((T, H, D))
    L = np.zeros((H, T))
    for s_, (Os, Ls) in ref.items():
        O[cuh[s_]:cuh[s_ + 1]] = Os
        L[:, cuh[s_]:cuh[s_ + 1]] = Ls
    o_in = torch.from_numpy(O).to(torch.bfloat16)
    lse_in = torch.from_numpy(L).to(torch.float32)
    cu = case.cu_seqlens.cuda()
    g = fa.fa_bwd_varlen(case.q.cuda(), case.k.cuda(), case.v.cuda(), o_in.cuda(), do.cuda(),
                         lse_in.cuda(), cu, case.max_seqlen, case.scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    rg = ora.attention_bwd_varlen_ref(case.q, case.k, case.v, do, case.cu_seqlens, case.scale,
                                      causal, o=o_in)[:3]
    re = ora.attention_bwd_varlen_ref(case.q, case.k, case.v, do, case.cu_seqlens, case.scale,
                                      causal)[:3]
    _check_both(g, rg, re, tag)


def _varlen_run(fa, case, do, causal):
    cu = case.cu_seqlens.cuda()
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    o, lse = fa.fa_fwd_varlen(q, k, v, cu, case.max_seqlen, case.scale, causal)
    g = fa.fa_bwd_varlen(q, k, v, o, do.cuda(), lse, cu, case.max_seqlen, case.scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    return g


@pytest.mark.parametrize("D,causal", [(64, True), (128, True), (128, False)])
def test_bwd_varlen(fa, D, causal):
    """Sequences of 1, 100, 128, 129 and 300 tokens packed together: every
    tile boundary case, rows of the next sequence inside tail tiles."""
    lens = [1, 100, 128, 129, 300]
    case = inp.varlen(lens, H=2, D=D, seed=970 + D, causal=causal)
    do = inp.output_grad(tuple(case.q.shape), seed=971)
    _varlen_checked(fa, case, do, causal, f"varlen D={D}")


def test_bwd_varlen_one_sequence_equals_dense(fa):
    """One packed sequence runs the same tiles in the same order as the dense
    backward: the gradients agree bit for bit."""
    N, H, D = 333, 2, 128
    case = inp.varlen([N], H=H, D=D, seed=975, causal=True)
    do = inp.output_grad((N, H, D), seed=976)
    a = _varlen_run(fa, case, do, True)
    dense = lambda t: t.permute(1, 0, 2).unsqueeze(0).contiguous().cuda()
    q, k, v = dense(case.q), dense(case.k), dense(case.v)
    o, lse = fa.fa_fwd(q, k, v, case.scale, True)
    b = fa.fa_bwd(q, k, v, o, dense(do), lse, case.scale, True)
    for x, y in zip(a, b):
        assert torch.equal(x.permute(1, 0, 2).unsqueeze(0), y)


def test_bwd_varlen_bad_offsets_reported(fa):
    case = inp.varlen([50, 70], H=2, D=64, seed=977, causal=True)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    cu = case.cu_seqlens.cuda()
    o, lse = fa.fa_fwd_varlen(q, k, v, cu, case.max_seqlen, case.scale, True)
    bad = torch.tensor([0, 50, 400], dtype=torch.int32, device="cuda")  # past T = 120
    fa.fa_bwd_varlen(q, k, v, o, torch.zeros_like(q), lse, bad, 400, case.scale, True)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS
    assert fa.fa_check_device_status() == fa.FA_OK


# --- causal sliding window ------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("w", [1, 37, 128, 129, 300, 600])
def test_bwd_window(fa, D, w):
    N = 517
    case = inp.dense(1, 2, N, D, seed=980 + w, causal=True)
    do = inp.output_grad((1, 2, N, D), seed=981 + w)
    _bwd_dense_checked(fa, case, do, True, f"window {w} D={D}", window=w)


def test_bwd_window_at_least_n_equals_causal(fa):
    """A window of N or more is causal attention: the same gradients bit for
    bit as fa_bwd (no edge tile exists, so the same products run)."""
    N = 300
    case = inp.dense(1, 2, N, 128, seed=985, causal=True)
    do = inp.output_grad((1, 2, N, 128), seed=986).cuda()
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    o, lse = fa.fa_fwd(q, k, v, case.scale, True)
    a = fa.fa_bwd(q, k, v, o, do, lse, case.scale, True)
    b = fa.fa_bwd_window(q, k, v, o, do, lse, N, case.scale)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_window_full_size_sampled(fa):
    """B=1 H=32 N=16384 D=128, window 4096: heads 0 and 31 on sampled rows."""
    B, H, N, D, w = 1, 32, 16384, 128, 4096
    case = inp.dense(B, H, N, D, seed=987, causal=True)
    do = inp.output_grad((B, H, N, D), seed=988)
    rng = np.random.default_rng(989)
    picks = sorted(set([0, 127, 128, w - 1, w, 8191, N - 1]) | set(rng.integers(0, N, 13).tolist()))
    _full_size_sampled(fa, case, do, picks, "window ", window=w)
