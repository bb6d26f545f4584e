"""GPU parity of the dense and varlen forward (C ABI through the binding)
against the float64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from tests.gpu_common import (check_lse, check_o_bf16, check_o_f32, np64,
                              TOL_F32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _dense_gpu(case):
    return (case.q.cuda(), case.k.cuda(), case.v.cuda())


# --- fp32 FFMA path -----------------------------------------------------------

def test_config1_fp32(fa):
    case = inp.config1()
    q, k, v = _dense_gpu(case)
    o, lse = fa.fa_fwd_f32(q, k, v, case.scale, case.causal)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, case.causal)
    assert np.abs(np64(o) - O).max() <= TOL_F32
    assert np.abs(np64(lse) - L).max() <= TOL_F32


@pytest.mark.parametrize("N,D,causal", [(1, 64, False), (63, 64, True), (200, 128, False),
                                        (333, 128, True), (129, 64, True), (70, 64, False),
                                        (1000, 64, True), (2048, 64, False)])
def test_fp32_shapes(fa, N, D, causal):
    case = inp.dense(2, 3, N, D, seed=10 + N, causal=causal, dtype=torch.float32,
                     qk_std=2.0)
    o, lse = fa.fa_fwd_f32(*_dense_gpu(case), case.scale, causal)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, causal)
    assert np.abs(np64(o) - O).max() <= TOL_F32
    assert np.abs(np64(lse) - L).max() <= TOL_F32


def test_fp32_large_grid(fa):
    """A grid that fills the GPU runs two threads per row (small problems
    eight): both against the oracle on sampled heads."""
    case = inp.dense(4, 8, 640, 64, seed=77, causal=True, dtype=torch.float32)
    o, lse = fa.fa_fwd_f32(*_dense_gpu(case), case.scale, True)
    O, L = ora.attention_ref(case.q[:1, :2], case.k[:1, :2], case.v[:1, :2], case.scale, True)
    assert np.abs(np64(o[:1, :2]) - O).max() <= TOL_F32
    assert np.abs(np64(lse[:1, :2]) - L).max() <= TOL_F32


# --- bf16 tensor-core path -------------------------------------------------------

SHAPES = [
    # (B, H, N, D, causal): several tiles and ragged tails, both head dims
    (1, 1, 1, 128, False),
    (1, 2, 127, 64, True),
    (2, 2, 128, 128, True),
    (1, 3, 129, 128, False),
    (2, 1, 255, 64, False),
    (1, 2, 300, 128, True),
    (1, 2, 517, 64, True),
    (2, 2, 640, 128, False),
]


@pytest.mark.parametrize("B,H,N,D,causal", SHAPES)
def test_bf16_small(fa, B, H, N, D, causal):
    case = inp.dense(B, H, N, D, seed=N * 7 + D, causal=causal)
    q, k, v = _dense_gpu(case)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, causal)
    o32, lse32 = fa.fa_fwd_ex(q, k, v, case.scale, causal, o_dtype=torch.float32)
    check_o_f32(np64(o32), O, f"fp32 out {B,H,N,D,causal}")
    check_lse(np64(lse32), L)
    o16, lse16 = fa.fa_fwd(q, k, v, case.scale, causal)
    check_o_bf16(np64(o16), O, f"bf16 out {B,H,N,D,causal}")
    check_lse(np64(lse16), L)
    # the bf16 output is the nearest-even rounding of the fp32 one
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(lse16, lse32)
    assert fa.fa_check_device_status() == fa.FA_OK


def test_config2_full(fa):
    """B=4 H=16 N=2048 D=128 causal: every output element against the oracle."""
    case = inp.config2()
    q, k, v = _dense_gpu(case)
    o, lse = fa.fa_fwd(q, k, v, case.scale, True)
    o32, _ = fa.fa_fwd_ex(q, k, v, case.scale, True, o_dtype=torch.float32)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, True)
    check_o_bf16(np64(o), O, "config2 bf16")
    check_o_f32(np64(o32), O, "config2 fp32-out")
    check_lse(np64(lse), L)


@pytest.mark.parametrize("D,ramp", [(64, False), (128, False), (64, True), (128, True)])
def test_persistent_equals_one_item(fa, D, ramp):
    """B=4 H=16 causal with N=2048 at D=128 and N=1024 at D=64 (1024 or 512
    query tiles, more than the SMs; short enough for the persistent launch)
    runs on persistent CTAs; each head alone runs one tile per CTA.  The
    per-tile arithmetic is the same, so the outputs agree bit for bit.  With
    keys that grow along the sequence (ramp) rows move their reference on
    many tiles, where the one-item kernel redoes the weights it computed
    against the old reference."""
    N = 2048 if D == 128 else 1024
    case = inp.dense(4, 16, N, D, seed=60 + D, causal=True, qk_std=3.0 if ramp else 1.0)
    q, k, v = _dense_gpu(case)
    if ramp:
        r = (1.0 + 4.0 * torch.arange(N, dtype=torch.float32, device="cuda") / N)
        k = (k.float() * r.view(1, 1, -1, 1)).to(torch.bfloat16)
    o, lse = fa.fa_fwd(q, k, v, case.scale, True)
    for b in range(4):
        for h in range(16):
            sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
            o1, l1 = fa.fa_fwd(sl(q), sl(k), sl(v), case.scale, True)
            assert torch.equal(o1[0, 0], o[b, h]), (b, h)
            assert torch.equal(l1[0, 0], lse[b, h]), (b, h)
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("c", [-90.0, 50.0, 90.0, 200.0])
def test_offset_invariance(fa, c):
    """Append a coordinate so every score of a row moves by c (q' = [q, c/scale],
    k' = [k, 1]): O is unchanged and LSE moves by c."""
    B, H, N, D = 1, 2, 300, 128
    case = inp.dense(B, H, N, D - 1, seed=21, causal=True, dtype=torch.float32)
    scale = 1.0 / math.sqrt(D)
    col = torch.full((B, H, N, 1), c / scale)
    # c/scale must be exact in bf16 for the shift to be exactly c
    col = col.to(torch.bfloat16).float()
    shift = float(col[0, 0, 0, 0]) * scale
    q = torch.cat([case.q, col], -1).to(torch.bfloat16)
    k = torch.cat([case.k, torch.ones(B, H, N, 1)], -1).to(torch.bfloat16)
    v = torch.cat([case.v, torch.zeros(B, H, N, 1)], -1).to(torch.bfloat16)
    q0 = torch.cat([case.q, torch.zeros(B, H, N, 1)], -1).to(torch.bfloat16)
    O, L = ora.attention_ref(q0, k, v, scale, True)
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), scale, True, o_dtype=torch.float32)
    check_o_f32(np64(o), O, f"offset {c}")
    check_lse(np64(lse) - shift, L, tol=2e-3)


@pytest.mark.parametrize("D", [64, 128])
def test_scale_zero_prefix_means(fa, D):
    """Identical scores: causal rows are prefix means of V, LSE = ln(i+1)."""
    case = inp.dense(1, 2, 260, D, seed=5, causal=True)
    o, lse = fa.fa_fwd_ex(*_dense_gpu(case), 0.0, True, o_dtype=torch.float32)
    v = np64(case.v)
    ref = np.cumsum(v, axis=2) / np.arange(1, 261)[None, None, :, None]
    check_o_f32(np64(o), ref, "scale 0")
    check_lse(np64(lse), np.log(np.arange(1, 261))[None, None, :].repeat(2, 1))


def test_empty_and_invalid(fa):
    z = torch.empty((0, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fa_fwd(z, z, z)
    assert o.shape == z.shape
    q = torch.randn(1, 1, 16, 96, device="cuda").to(torch.bfloat16)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(q, q, q)
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    q = torch.randn(1, 1, 16, 64, device="cuda").to(torch.bfloat16)
    o = torch.full_like(q, 7.0)
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(q, q, q, scale=-1.0, o=o)
    assert e.value.code == fa.FA_ERR_INVALID_ARG
    assert (o == 7.0).all()  # nothing launched, output untouched


def test_output_tail_untouched(fa):
    """The O stores stop at the tensor's end: with O the head of a larger
    buffer, rows past the last sequence (dense N = 300 and 129: the last
    tile's warps straddle or pass N; varlen: a packed tail) leave the rest of
    the buffer as it was, and the outputs still match the oracle."""
    sentinel = 0x7FC1  # a NaN bit pattern no store produces
    for (B, H, N, D) in [(1, 2, 300, 128), (2, 1, 129, 128), (1, 1, 300, 64)]:
        case = inp.dense(B, H, N, D, seed=N + D, causal=True)
        q, k, v = _dense_gpu(case)
        n = B * H * N * D
        buf = torch.full((n + 8192,), sentinel, dtype=torch.int16, device="cuda")
        o = buf[:n].view(torch.bfloat16).view(B, H, N, D)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        fa.fa_fwd(q, k, v, case.scale, True, o=o, lse=lse)
        torch.cuda.synchronize()
        assert bool((buf[n:] == sentinel).all()), f"store past the end {B, H, N, D}"
        O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, True)
        check_o_bf16(np64(o), O, f"dense {B, H, N, D}")
        check_lse(np64(lse), L)
    for D in (64, 128):
        case = inp.varlen([300, 129, 37], H=2, D=D, seed=3 * D, causal=True)
        q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
        T = sum(case.meta["lens"])
        n = T * 2 * D
        buf = torch.full((n + 8192,), sentinel, dtype=torch.int16, device="cuda")
        o = buf[:n].view(torch.bfloat16).view(T, 2, D)
        lse = torch.empty((2, T), dtype=torch.float32, device="cuda")
        fa.fa_fwd_varlen(q, k, v, case.cu_seqlens.cuda(), case.max_seqlen, case.scale, True,
                         o=o, lse=lse)
        torch.cuda.synchronize()
        assert bool((buf[n:] == sentinel).all()), f"varlen store past the end D={D}"
        ref = ora.varlen_ref(case.q, case.k, case.v, case.cu_seqlens, case.scale, True)
        cuh = case.cu_seqlens.tolist()
        for s_, (O, L) in ref.items():
            check_o_bf16(np64(o[cuh[s_]:cuh[s_ + 1]]), O, f"varlen seq {s_} D={D}")
            check_lse(np64(lse[:, cuh[s_]:cuh[s_ + 1]]), L)
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("N,D,causal,qk_std", [(65536, 128, True, 3.0), (32768, 64, False, 1.0)])
def test_long_sequence_sampled(fa, N, D, causal, qk_std):
    """Sequences 2-4x config 3's length: sampled rows (the first and last,
    both sides of tile edges, random ones) of both heads against the oracle.
    The causal case keeps config 3's score spread, so the lagging reference
    maximum runs over 512 key tiles."""
    case = inp.dense(1, 2, N, D, seed=N + D, causal=causal, qk_std=qk_std)
    q, k, v = _dense_gpu(case)
    o, lse = fa.fa_fwd(q, k, v, case.scale, causal)
    torch.cuda.synchronize()
    rng = np.random.default_rng(N)
    rows = sorted(set([0, 1, 127, 128, 4095, 4096, N // 2, N - 129, N - 128, N - 1])
                  | set(rng.integers(0, N, 20).tolist()))
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, causal, rows=rows)
    idx = torch.tensor(rows, device="cuda")
    check_o_bf16(np64(o[:, :, idx]), O, f"N={N} D={D}")
    check_lse(np64(lse[:, :, idx]), L)
    assert fa.fa_check_device_status() == fa.FA_OK


# --- varlen -------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_two_group_odd_tile_counts(fa, causal):
    """D = 64 splits a query tile's key tiles between two softmax groups
    (even and odd tiles) and merges their states: sequences of 1, 2, 3 and
    5 key tiles (group 1 with no tile, one, or fewer than group 0), ragged
    tails, keys that grow along the sequence so that the reference maximum
    moves inside each group."""
    for N in (100, 200, 300, 600):
        case = inp.dense(1, 3, N, 64, seed=70 + N, causal=causal, qk_std=3.0)
        ramp = (1.0 + 3.0 * torch.arange(N, dtype=torch.float32) / N).view(1, 1, -1, 1)
        k = (case.k.float() * ramp).to(torch.bfloat16)
        o, lse = fa.fa_fwd_ex(case.q.cuda(), k.cuda(), case.v.cuda(), case.scale, causal,
                              o_dtype=torch.float32)
        O, L = ora.attention_ref(case.q, k, case.v, case.scale, causal)
        check_o_f32(np64(o), O, f"two groups N={N} causal={causal}")
        check_lse(np64(lse), L)
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_small(fa, D):
    lens = [1, 127, 128, 129, 0, 300, 5, 257]
    case = inp.varlen(lens, H=3, D=D, seed=D, causal=True)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    cu = case.cu_seqlens.cuda()
    o, lse = fa.fa_fwd_varlen(q, k, v, cu, case.max_seqlen, case.scale, True)
    ref = ora.varlen_ref(case.q, case.k, case.v, case.cu_seqlens, case.scale, True)
    cuh = case.cu_seqlens.tolist()
    for s, (O, L) in ref.items():
        a, b = cuh[s], cuh[s + 1]
        check_o_bf16(np64(o[a:b]), O, f"seq {s}")
        check_lse(np64(lse[:, a:b]), L)
        # the same sequence alone through the dense entry point: same bits
        if b > a:
            qs, ks, vs = (t[a:b].permute(1, 0, 2).unsqueeze(0).contiguous() for t in (q, k, v))
            od, ld = fa.fa_fwd(qs, ks, vs, case.scale, True)
            assert torch.equal(od[0].permute(1, 0, 2), o[a:b])
            assert torch.equal(ld[0], lse[:, a:b])
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_moving_reference(fa, D):
    """Packed sequences whose keys grow along each sequence (scores with a
    spread of many units), so rows move their reference on many tiles: the
    one-item kernel redoes the weights of those tiles.  Every row against
    the oracle, and each sequence alone through the dense entry point bit
    for bit."""
    lens = [300, 700, 129, 1000, 1]
    case = inp.varlen(lens, H=2, D=D, seed=70 + D, causal=True)
    cuh = case.cu_seqlens.tolist()
    ramp = torch.ones(case.k.shape[0])
    for s_ in range(len(lens)):
        a, b = cuh[s_], cuh[s_ + 1]
        ramp[a:b] = 1.0 + 4.0 * torch.arange(b - a, dtype=torch.float32) / max(1, b - a)
    qh = (case.q.float() * 3.0).to(torch.bfloat16)
    kh = (case.k.float() * 3.0 * ramp.view(-1, 1, 1)).to(torch.bfloat16)
    q, k, v = qh.cuda(), kh.cuda(), case.v.cuda()
    cu = case.cu_seqlens.cuda()
    o, lse = fa.fa_fwd_varlen(q, k, v, cu, case.max_seqlen, case.scale, True)
    ref = ora.varlen_ref(qh, kh, case.v, case.cu_seqlens, case.scale, True)
    for s_, (O, L) in ref.items():
        a, b = cuh[s_], cuh[s_ + 1]
        check_o_bf16(np64(o[a:b]), O, f"seq {s_}")
        check_lse(np64(lse[:, a:b]), L)
        qs, ks, vs = (t[a:b].permute(1, 0, 2).unsqueeze(0).contiguous() for t in (q, k, v))
        od, ld = fa.fa_fwd(qs, ks, vs, case.scale, True)
        assert torch.equal(od[0].permute(1, 0, 2), o[a:b])
        assert torch.equal(ld[0], lse[:, a:b])
    assert fa.fa_check_device_status() == fa.FA_OK


def test_varlen_bad_offsets_reported(fa):
    """cu_seqlens that decrease are caught by the kernel's own check and
    reported as FA_ERR_DEVICE_BOUNDS; nothing is read out of range."""
    case = inp.varlen([100, 50], H=2, D=64, seed=1)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    bad = torch.tensor([0, 120, 100], dtype=torch.int32, device="cuda")
    fa.fa_fwd_varlen(q, k, v, bad, 150, case.scale, True)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS
    assert fa.fa_check_device_status() == fa.FA_OK  # the word was cleared


# --- run-to-run determinism -------------------------------------------------------

def test_forward_deterministic(fa):
    """No atomics and a fixed merge order in every path: repeated launches on
    the same inputs give the same bits (dense causal with a window edge,
    packed sequences, and the fp32 path)."""
    case = inp.dense(1, 8, 3000, 128, seed=31, causal=True, qk_std=3.0)
    q, k, v = _dense_gpu(case)
    runs = [fa.fa_fwd(q, k, v, case.scale, True) for _ in range(3)]
    runs += [fa.fa_fwd(q, k, v, case.scale, True) for _ in range(2)]
    for o, lse in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
    wins = [fa.fa_fwd_window(q, k, v, 700, case.scale) for _ in range(3)]
    for o, lse in wins[1:]:
        assert torch.equal(o, wins[0][0]) and torch.equal(lse, wins[0][1])

    vcase = inp.varlen([1, 129, 700, 2048, 5], H=4, D=64, seed=32, causal=True)
    vq, vk, vv, cu = vcase.q.cuda(), vcase.k.cuda(), vcase.v.cuda(), vcase.cu_seqlens.cuda()
    vruns = [fa.fa_fwd_varlen(vq, vk, vv, cu, vcase.max_seqlen, vcase.scale, True)
             for _ in range(3)]
    for o, lse in vruns[1:]:
        assert torch.equal(o, vruns[0][0]) and torch.equal(lse, vruns[0][1])

    fcase = inp.dense(2, 3, 700, 64, seed=33, causal=True, dtype=torch.float32)
    fq, fk, fv = _dense_gpu(fcase)
    fruns = [fa.fa_fwd_f32(fq, fk, fv, fcase.scale, True) for _ in range(3)]
    for o, lse in fruns[1:]:
        assert torch.equal(o, fruns[0][0]) and torch.equal(lse, fruns[0][1])
    assert fa.fa_check_device_status() == fa.FA_OK


# --- the reference maximum: moves, and range -----------------------------------------

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_reference_moves(fa, causal, D):
    """Keys that grow along the sequence make later tiles' maxima exceed the
    reference a row set on its first tile by far more than the move
    threshold, so rows move their reference (and warps rescale O) many
    times; the result still matches the oracle.  (At D = 64 both softmax
    groups rescale their own accumulators between their P V products.)"""
    case = inp.dense(1, 2, 1100, D, seed=41, causal=causal, qk_std=3.0)
    ramp = (1.0 + 4.0 * torch.arange(1100, dtype=torch.float32) / 1100).view(1, 1, -1, 1)
    k = (case.k.float() * ramp).to(torch.bfloat16)
    o, lse = fa.fa_fwd(case.q.cuda(), k.cuda(), case.v.cuda(), case.scale, causal)
    O, L = ora.attention_ref(case.q, k, case.v, case.scale, causal)
    check_o_bf16(np64(o), O, "moving reference")
    check_lse(np64(lse), L)
    o32, lse32 = fa.fa_fwd_ex(case.q.cuda(), k.cuda(), case.v.cuda(), case.scale, causal,
                              o_dtype=torch.float32)
    check_o_f32(np64(o32), O, "moving reference, fp32 out")


def test_large_values_in_range(fa):
    """|V| around 1e15 at N = 2048 sits far inside the range the lagging
    reference keeps (N * 2^32 * max|V| below fp32's limit): finite outputs
    within the relative tolerance of the oracle."""
    case = inp.dense(1, 2, 2048, 128, seed=42, causal=True, qk_std=3.0, v_std=1e15)
    o, lse = fa.fa_fwd_ex(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.scale, True,
                          o_dtype=torch.float32)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, True)
    o = np64(o)
    assert np.isfinite(o).all()
    assert np.abs(o - O).max() <= 1e-2 * np.abs(O).max()
    check_lse(np64(lse), L)
