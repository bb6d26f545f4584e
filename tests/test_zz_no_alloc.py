"""The no-allocation split-KV decode entry point.

Some callers are handed only their input and output buffers and may not
allocate device memory (a plugin interface without a workspace, a serving
loop whose memory is fixed at start-up).  fa_decode_splitkv_noalloc keeps its
partial states in a static device array of the library instead.  This file
checks, through the C ABI, that it returns what the allocating path
(fa_decode_splitkv into a caller workspace, then fa_combine_states) returns,
on two calls in a row with different inputs, so that nothing left in the
shared array by the first call leaks into the second.  It is named to be
collected last.
"""
import pytest
import torch

import fa_inputs as inp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _both_paths(fa, case, o_dtype):
    q, kc, vc = case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda()
    cu = case.cu_seqlens_k.cuda()
    pm, pd, po = fa.fa_decode_splitkv(q, kc, vc, cu, case.num_splits, case.scale)
    ref_o, ref_l = fa.fa_combine_states(pm, pd, po, o_dtype=o_dtype)
    o, l = fa.fa_decode_splitkv_noalloc(q, kc, vc, cu, case.num_splits, case.scale,
                                        o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o, l, ref_o, ref_l


def test_noalloc_matches_allocating_path_twice(fa):
    """Both paths run the same two kernels, with the same fixed chunk order,
    on the same inputs, so their outputs must be equal bit for bit; a state
    left over from the first call would change some bits of the second."""
    first = inp.decode(6, 4, 128, seed=31, num_splits=16,
                       lens=[1, 5, 300, 2048, 4097, 9000])
    second = inp.decode(3, 8, 64, seed=32, num_splits=7, lens=[700, 2, 1500])
    for case, o_dtype in ((first, torch.bfloat16), (second, torch.float32)):
        o, l, ref_o, ref_l = _both_paths(fa, case, o_dtype)
        assert torch.equal(o, ref_o), "no-alloc O differs from the workspace path"
        assert torch.equal(l, ref_l), "no-alloc LSE differs from the workspace path"
    assert fa.fa_check_device_status() == fa.FA_OK


def test_noalloc_refuses_oversized_problem(fa):
    # 64 x 64 x 64 states x (128 + 2) floats = 136 MB > 32 MiB
    q = torch.zeros((64, 64, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((64, 64, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.arange(65, dtype=torch.int32, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_decode_splitkv_noalloc(q, kv, kv, cu, 64)
    assert e.value.code == fa.FA_ERR_SCRATCH_CAPACITY
