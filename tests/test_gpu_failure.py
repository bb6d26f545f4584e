"""The device-side failure path of the tensor-core forward, made to run on
purpose without faulting anything.

Every pipeline wait in the kernels is bounded; when one runs out the kernel
records FA_ERR_DEVICE_TIMEOUT in the device status word, lets the copies and
tensor-core products it has already issued complete, frees its tensor memory
and returns.  fa_fwd_fault_inject makes that happen: the producer never
requests one key tile (a flag nothing else sets), and the waits give up after
a short limit.  The test then checks that the status reports the timeout once
and is cleared, that query tiles which never needed the missing key tile
still wrote correct rows, and that the next ordinary call on the same
context matches the oracle.
"""
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


@pytest.mark.parametrize("D,causal,H", [(128, False, 2), (64, False, 2), (128, True, 2),
                                         (128, False, 80), (64, False, 80)])
def test_wait_timeout_unwinds(fa, D, causal, H):
    """H = 80 gives 320 query tiles, more than the GPU's SMs, so the short
    sequence runs on persistent CTAs (a CTA that gives up leaves its later
    items unwritten); H = 2 runs one CTA per query tile."""
    B, N = 1, 512  # four query tiles, four key tiles per head
    case = inp.dense(B, H, N, D, seed=50 + D, causal=causal)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    assert fa.fa_check_device_status() == fa.FA_OK
    o = torch.full((B, H, N, D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, N), 7.0, dtype=torch.float32, device="cuda")
    fa.fa_fwd_fault_inject(q, k, v, 1, 2000, case.scale, causal, o=o, lse=lse)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_check_device_status() == fa.FA_OK  # reported once, then cleared
    O, L = ora.attention_ref(case.q, case.k, case.v, case.scale, causal)
    if causal:
        # query tile 0 sees key tile 0 only: it finished and wrote its rows;
        # the tiles that reached the missing key tile gave up without writing
        check_o_bf16(np64(o[:, :, :128]), O[:, :, :128], "tile 0")
        check_lse(np64(lse[:, :, :128]), L[:, :, :128])
        assert bool((o[:, :, 128:] == 7.0).all()) and bool((lse[:, :, 128:] == 7.0).all())
    else:
        assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    # the context is usable: an ordinary call matches the oracle
    o2, l2 = fa.fa_fwd(q, k, v, case.scale, causal)
    check_o_bf16(np64(o2), O, "after the timeout")
    check_lse(np64(l2), L)
    assert fa.fa_check_device_status() == fa.FA_OK
    # a tile index past the last key tile injects nothing: the same bits
    o3, l3 = fa.fa_fwd_fault_inject(q, k, v, N // 128, 2000, case.scale, causal)
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.equal(o3, o2) and torch.equal(l3, l2)
