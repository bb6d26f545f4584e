"""GPU parity of prefix attention (fa_prefix_attention, the inclusive scan
of the (m, d, o) states over each sequence's keys) against the float64
oracle: every position on small ragged sequences, sampled positions on the
decode workload's caches, the last position against split-KV decode, and
the device bounds check."""
import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from tests.gpu_common import check_lse, check_o_bf16, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _run(fa, case):
    cu = case.cu_seqlens_k.cuda()
    o, lse = fa.fa_prefix_attention(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(),
                                    cu, case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("D", [64, 128])
def test_every_position_small(fa, D):
    lens = [1, 5, 0, 127, 128, 129, 300, 1000]
    case = inp.decode(len(lens), 4, D, seed=70 + D, num_splits=1, lens=lens)
    o, lse = _run(fa, case)
    O, L = ora.prefix_attention_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k,
                                    case.scale)
    check_o_bf16(np64(o), O, f"prefix D={D}")
    check_lse(np64(lse), L)


def test_peaked_scores(fa):
    """q, k with std 3: scores in the tens, maxima that move often."""
    lens = [700, 257]
    case = inp.decode(2, 3, 128, seed=75, num_splits=1, lens=lens)
    case.q.mul_(3)
    case.k_cache.mul_(3)
    o, lse = _run(fa, case)
    O, L = ora.prefix_attention_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k,
                                    case.scale)
    check_o_bf16(np64(o), O, "peaked")
    check_lse(np64(lse), L)


def test_decode_workload_sampled(fa):
    """The decode workload's caches (B=64, H=32, D=128, L ~ U[1024, 32768]):
    sampled positions (window edges, both ends, random) of sampled heads."""
    case = inp.decode(64, 32, 128, seed=4, num_splits=16)
    o, lse = _run(fa, case)
    lens = case.meta["lens"]
    rng = np.random.default_rng(1)
    batch = [0, 17, 63]
    pos = {b: sorted(set([0, 1, 127, 128, 129, lens[b] - 1]) |
                     set(rng.integers(0, lens[b], 6).tolist())) for b in batch}
    heads = [0, 31]
    O, L = ora.prefix_attention_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k,
                                    case.scale, batch=batch, heads=heads, positions=pos)
    cu = case.cu_seqlens_k.tolist()
    for b in batch:
        rows = [cu[b] + i for i in pos[b]]
        for h in heads:
            check_o_bf16(np64(o[rows, h]), O[rows, h], f"b{b} h{h}")
            check_lse(np64(lse[h, rows]), L[h, rows])


def test_last_position_is_decode(fa):
    case = inp.decode(6, 8, 128, seed=80, num_splits=4, lens=[3000, 1, 128, 4097, 50, 999])
    o, lse = _run(fa, case)
    cu = case.cu_seqlens_k.cuda()
    od, ld = fa.decode(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), cu, 4,
                       case.scale)
    last = (case.cu_seqlens_k[1:] - 1).long().cuda()
    a = o[last].float()
    b = od.float()
    assert (a - b).abs().max().item() <= 2 ** -7 * b.abs().max().item() + 1e-3
    assert (lse[:, last].t() - ld).abs().max().item() <= 1e-4


def test_bad_offsets_report_bounds(fa):
    case = inp.decode(2, 2, 64, seed=81, num_splits=1, lens=[10, 20])
    cu = torch.tensor([0, 10, 40], dtype=torch.int32, device="cuda")  # past T = 30
    fa.fa_prefix_attention(case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(), cu,
                           case.scale)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS
    assert fa.fa_check_device_status() == fa.FA_OK


@pytest.mark.parametrize("D,S", [(64, 2), (128, 7), (128, 16)])
def test_chunked_every_position(fa, D, S):
    """Rows cut into S chunks scanned at once from the split-KV states of the
    earlier chunks: every position against the oracle, empty chunks incl."""
    lens = [1, 5, 0, 127, 300, 1000]
    case = inp.decode(len(lens), 4, D, seed=90 + S, num_splits=S, lens=lens)
    cu = case.cu_seqlens_k.cuda()
    o, lse = fa.fa_prefix_attention_chunked(case.q.cuda(), case.k_cache.cuda(),
                                            case.v_cache.cuda(), cu, S, case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    O, L = ora.prefix_attention_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k,
                                    case.scale)
    check_o_bf16(np64(o), O, f"chunked S={S}")
    check_lse(np64(lse), L)


def test_chunked_long_row(fa):
    """One long sequence (2 heads, 200000 keys) in 64 chunks: sampled positions
    at chunk edges and inside, against the oracle."""
    L_ = 200000
    case = inp.decode(1, 2, 128, seed=95, num_splits=64, lens=[L_], device="cuda")
    cu = case.cu_seqlens_k.cuda()
    o, lse = fa.fa_prefix_attention_chunked(case.q, case.k_cache, case.v_cache, cu, 64,
                                            case.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    csize = -(-L_ // 64)
    rng = np.random.default_rng(3)
    pos = sorted(set([0, 1, csize - 1, csize, csize + 1, 31 * csize, L_ - 1]) |
                 set(rng.integers(0, L_, 8).tolist()))
    O, L = ora.prefix_attention_ref(case.q.cpu(), case.k_cache.cpu(), case.v_cache.cpu(),
                                    case.cu_seqlens_k, case.scale, positions={0: pos})
    check_o_bf16(np64(o[pos]), O[pos], "long row")
    check_lse(np64(lse[:, pos]), L[:, pos])
