"""GPU parity of the mask and cache variants against the float64 oracle:
the causal sliding window (fa_fwd_window) and split-KV decode over a paged KV
cache with grouped query heads (fa_decode_paged_splitkv)."""
import math

import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from tests.gpu_common import check_lse, check_o_bf16, check_o_f32, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


# --- sliding window -----------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("w", [1, 37, 128, 129, 300, 600])
def test_window_small(fa, D, w):
    case = inp.dense(1, 2, 517, D, seed=w + D, causal=True, qk_std=2.0)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    o, lse = fa.fa_fwd_window(q, k, v, w, case.scale)
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, True, window=w)
    check_o_bf16(np64(o), O, f"window {w}")
    check_lse(np64(lse), L)
    if w >= 517:  # a window covering the sequence is plain causal attention
        oc, lc = fa.fa_fwd(q, k, v, case.scale, True)
        assert torch.equal(o, oc) and torch.equal(lse, lc)
    assert fa.fa_check_device_status() == fa.FA_OK


def test_window_long_sampled(fa):
    """N=16384, window 4096: sampled rows (including both edges of the first
    full window) against the oracle."""
    case = inp.dense(1, 2, 16384, 128, seed=77, causal=True, qk_std=3.0, device="cuda")
    o, lse = fa.fa_fwd_window(case.q, case.k, case.v, 4096, case.scale)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 4094, 4095, 4096, 4097, 8191, 12345, 16383])
    O, L = ora.attention_ref(case.q.cpu(), case.k.cpu(), case.v.cpu(), case.scale, True,
                             rows=rows, window=4096)
    ri = torch.as_tensor(rows, device="cuda")
    check_o_bf16(np64(o.index_select(2, ri)), O, "window 4096")
    check_lse(np64(lse.index_select(2, ri)), L)


@pytest.mark.parametrize("D,w", [(128, 300), (64, 300), (64, 129)])
def test_window_persistent(fa, D, w):
    """B=2 H=40 with N=1300 at D=128 and N=1000 at D=64 (880 or 640 query
    tiles, more than the SMs; short enough for the persistent launch) runs on
    persistent CTAs: window edges inside items, items whose key range starts
    past the first tile.  Two heads against the oracle, every head against
    the same head launched alone (one tile per CTA) bit for bit."""
    N = 1300 if D == 128 else 1000
    case = inp.dense(2, 40, N, D, seed=w + 3 * D, causal=True, qk_std=2.0)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    o, lse = fa.fa_fwd_window(q, k, v, w, case.scale)
    O, L = ora.attention_ref(case.q[:, :1], case.k[:, :1], case.v[:, :1], case.scale, True,
                             window=w)
    check_o_bf16(np64(o[:, :1]), O, f"window {w} D={D}")
    check_lse(np64(lse[:, :1]), L)
    for b in range(2):
        for h in range(0, 40, 7):
            sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
            o1, l1 = fa.fa_fwd_window(sl(q), sl(k), sl(v), w, case.scale)
            assert torch.equal(o1[0, 0], o[b, h]) and torch.equal(l1[0, 0], lse[b, h]), (b, h)
    assert fa.fa_check_device_status() == fa.FA_OK


def test_window_invalid(fa):
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_window(q, q, q, 0)
    assert e.value.code == fa.FA_ERR_INVALID_ARG


# --- paged KV cache, grouped query heads -------------------------------------------

def _paged_align(H, Hkv, page, D):
    """Chunk length granularity of fa_decode_paged_splitkv: whole 128-key
    tiles on the grouped-head tensor-core path, single keys otherwise."""
    return 128 if D == 128 and 2 <= H // Hkv <= 16 and page >= 8 else 1


def _paged_gpu(case):
    return (case.q.cuda(), case.k_pages.cuda(), case.v_pages.cuda(),
            case.block_table.cuda(), case.seqlens.cuda())


@pytest.mark.parametrize("H,Hkv,page,S,D", [(8, 8, 16, 1, 128), (8, 2, 16, 7, 128),
                                            (8, 4, 64, 16, 64), (16, 1, 32, 16, 128)])
def test_paged_decode(fa, H, Hkv, page, S, D):
    lens = [1, 63, 64, 65, 1000, 5000]
    case = inp.paged_decode(len(lens), H, Hkv, D, page, seed=H + page + S, num_splits=S,
                            lens=lens)
    args = _paged_gpu(case)
    pm, pd, po = fa.fa_decode_paged_splitkv(*args, S, case.scale)
    M, Dn, Oc = ora.chunk_states_paged_ref(case.q, case.k_pages, case.v_pages,
                                           case.block_table, case.seqlens, S, case.scale,
                                           align=_paged_align(H, Hkv, page, D))
    full = np.isfinite(M)
    assert (np64(pm)[~full] == -np.inf).all() and (np64(pd)[~full] == 0).all()
    assert np.abs(np64(pm)[full] - M[full]).max() <= 1e-4 * max(1.0, np.abs(M[full]).max())
    assert np.abs(np64(pd)[full] / Dn[full] - 1).max() <= 1e-4
    O, L = ora.decode_paged_ref(case.q, case.k_pages, case.v_pages, case.block_table,
                                case.seqlens, case.scale)
    o32, lse = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    check_o_f32(np64(o32), O, "paged decode")
    check_lse(np64(lse), L)
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("H,Hkv,page,S", [(8, 4, 8, 3), (8, 2, 16, 7), (32, 8, 64, 16),
                                          (16, 2, 128, 5), (16, 1, 256, 2), (12, 3, 32, 1)])
def test_paged_decode_tensor_core_groups(fa, H, Hkv, page, S):
    """D = 128 with 2..16 query heads per KV head runs the tensor-core kernel:
    chunk states against the oracle's, the combined output against decode."""
    lens = [1, 127, 128, 129, 700, 3001]
    D = 128
    case = inp.paged_decode(len(lens), H, Hkv, D, page, seed=H * 3 + page + S, num_splits=S,
                            lens=lens)
    args = _paged_gpu(case)
    pm, pd, po = fa.fa_decode_paged_splitkv(*args, S, case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    M, Dn, Oc = ora.chunk_states_paged_ref(case.q, case.k_pages, case.v_pages,
                                           case.block_table, case.seqlens, S, case.scale,
                                           align=128)
    full = np.isfinite(M)
    assert (np64(pm)[~full] == -np.inf).all() and (np64(pd)[~full] == 0).all()
    assert np.abs(np64(pm)[full] - M[full]).max() <= 1e-4 * max(1.0, np.abs(M[full]).max())
    assert np.abs(np64(pd)[full] / Dn[full] - 1).max() <= 1e-4
    O, L = ora.decode_paged_ref(case.q, case.k_pages, case.v_pages, case.block_table,
                                case.seqlens, case.scale)
    o32, lse = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    check_o_f32(np64(o32), O, "paged decode (tensor cores)")
    check_lse(np64(lse), L)


def test_paged_tensor_core_stale_tail_rows(fa):
    """Rows past a sequence's end inside its last page hold NaN: they must not
    reach the output."""
    lens = [200, 70]
    case = inp.paged_decode(len(lens), 8, 2, 128, 64, seed=41, num_splits=2, lens=lens)
    kp, vp = case.k_pages.clone(), case.v_pages.clone()
    for b, L in enumerate(lens):
        last = int(case.block_table[b, (L - 1) // 64])
        kp[last, L % 64:] = float("nan")
        vp[last, L % 64:] = float("nan")
    q, _, _, table, sl = _paged_gpu(case)
    pm, pd, po = fa.fa_decode_paged_splitkv(q, kp.cuda(), vp.cuda(), table, sl, 2, case.scale)
    o32, lse = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    O, L = ora.decode_paged_ref(case.q, case.k_pages, case.v_pages, case.block_table,
                                case.seqlens, case.scale)
    check_o_f32(np64(o32), O, "stale tail rows")
    check_lse(np64(lse), L)


def test_paged_tensor_core_bad_page_reported(fa):
    case = inp.paged_decode(2, 8, 2, 128, 16, seed=43, num_splits=4, lens=[300, 90])
    q, kp, vp, table, sl = _paged_gpu(case)
    table[0, 3] = case.meta["pages"] + 7  # past the pool
    fa.fa_decode_paged_splitkv(q, kp, vp, table, sl, 4, case.scale)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS
    assert fa.fa_check_device_status() == fa.FA_OK


def test_paged_identity_layout_equals_packed_decode(fa):
    """Pages laid out in order with one KV head per query head hold the same
    keys as a packed cache: the two entry points give the same bits."""
    lens = [100, 37, 256]
    H, D, page = 4, 128, 16
    case = inp.paged_decode(len(lens), H, H, D, page, seed=5, num_splits=8, lens=lens,
                            spare_pages=0)
    nblk = [-(-L // page) for L in lens]
    # renumber pages so sequence b's pages are consecutive and in key order
    order = [int(case.block_table[b, c]) for b in range(len(lens)) for c in range(nblk[b])]
    kp = case.k_pages[order]
    vp = case.v_pages[order]
    table = torch.full_like(case.block_table, -1)
    i = 0
    for b in range(len(lens)):
        for c in range(nblk[b]):
            table[b, c] = i
            i += 1
    packed_k = torch.cat([kp[sum(nblk[:b]):sum(nblk[:b + 1])].reshape(-1, H, D)[:lens[b]]
                          for b in range(len(lens))])
    packed_v = torch.cat([vp[sum(nblk[:b]):sum(nblk[:b + 1])].reshape(-1, H, D)[:lens[b]]
                          for b in range(len(lens))])
    cu = inp.cu_from_lengths(lens)
    q = case.q.cuda()
    a = fa.fa_decode_paged_splitkv(q, kp.cuda(), vp.cuda(), table.cuda(),
                                   case.seqlens.cuda(), 8, case.scale)
    b = fa.fa_decode_splitkv(q, packed_k.cuda(), packed_v.cuda(), cu.cuda(), 8, case.scale)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_paged_bad_page_reported(fa):
    case = inp.paged_decode(2, 4, 2, 64, 16, seed=3, num_splits=4, lens=[40, 20])
    q, kp, vp, table, sl = _paged_gpu(case)
    table[1, 0] = case.meta["pages"] + 5  # past the pool
    fa.fa_decode_paged_splitkv(q, kp, vp, table, sl, 4, case.scale)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS
