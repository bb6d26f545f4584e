"""GPU parity of split-KV decode and of the state combine.

* fa_decode_splitkv's chunk states against the oracle's chunk states;
* decode + combine against the unsplit float64 decode, for several chunk
  counts (the split must not change the result beyond rounding);
* fa_combine_states bit for bit against the plain C fp32 fold, on states the
  oracle produced (never on states from the GPU).
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from oracle import combine_f32 as cf
from tests.gpu_common import check_lse, check_o_bf16, check_o_f32, check_states, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _gpu(case):
    return (case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda(),
            case.cu_seqlens_k.cuda())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 16, 37])
def test_decode_small(fa, D, S):
    lens = [1, 2, 15, 16, 17, 100, 1000, 2049]
    case = inp.decode(len(lens), 4, D, seed=S + D, num_splits=S, lens=lens)
    q, kc, vc, cu = _gpu(case)
    pm, pd, po = fa.fa_decode_splitkv(q, kc, vc, cu, S, case.scale)
    M, Dn, Oc = ora.chunk_states_ref(case.q, case.k_cache, case.v_cache,
                                     case.cu_seqlens_k, S, case.scale)
    check_states(pm, pd, po, M, Dn, Oc, f"states S={S}")
    O, L = ora.decode_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k, case.scale)
    o32, lse = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    check_o_f32(np64(o32), O, "decode fp32-out")
    check_lse(np64(lse), L)
    o16, lse16 = fa.fa_combine_states(pm, pd, po, o_dtype=torch.bfloat16)
    check_o_bf16(np64(o16), O, "decode bf16")
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(lse16, lse)
    assert fa.fa_check_device_status() == fa.FA_OK


def test_decode_empty_sequence(fa):
    """A zero-length cache: every chunk is the identity, O = 0, LSE = -inf."""
    case = inp.decode(3, 2, 128, seed=9, num_splits=4, lens=[5, 0, 3])
    q, kc, vc, cu = _gpu(case)
    pm, pd, po = fa.fa_decode_splitkv(q, kc, vc, cu, 4, case.scale)
    o, lse = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    assert (pm[1] == -math.inf).all() and (pd[1] == 0).all() and (po[1] == 0).all()
    assert (o[1] == 0).all() and (lse[1] == -math.inf).all()
    O, L = ora.decode_ref(case.q, case.k_cache, case.v_cache, case.cu_seqlens_k,
                          case.scale, batch=[0, 2])
    check_o_f32(np64(o[[0, 2]]), O[[0, 2]])
    check_lse(np64(lse[[0, 2]]), L[[0, 2]])


def test_decode_bad_offsets_reported(fa):
    case = inp.decode(2, 2, 64, seed=2, num_splits=4, lens=[10, 10])
    q, kc, vc, _ = _gpu(case)
    bad = torch.tensor([0, 10, 25], dtype=torch.int32, device="cuda")  # 25 > T_k = 20
    fa.fa_decode_splitkv(q, kc, vc, bad, 4, case.scale)
    assert fa.fa_check_device_status() == fa.FA_ERR_DEVICE_BOUNDS


# --- combine: bit-exact against the C fold ------------------------------------------

def _oracle_states(S, D, seed):
    """States from the oracle's chunk definition (float64, rounded to fp32)."""
    lens = [1, 3, 40, 333, 1024, 4000]
    case = inp.decode(len(lens), 3, D, seed=seed, num_splits=S, lens=lens)
    M, Dn, Oc = ora.chunk_states_ref(case.q, case.k_cache, case.v_cache,
                                     case.cu_seqlens_k, S, case.scale)
    return (M.astype(np.float32), Dn.astype(np.float32), Oc.astype(np.float32))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 16, 37])
def test_combine_bit_exact(fa, D, S):
    M, Dn, Oc = _oracle_states(S, D, seed=S * D)
    rows = M.shape[0] * M.shape[1]
    ref_o, ref_b, ref_l = cf.combine_f32(M.reshape(rows, S), Dn.reshape(rows, S),
                                         Oc.reshape(rows, S, D))
    pm, pd, po = (torch.from_numpy(x).cuda() for x in (M, Dn, Oc))
    o32, l32 = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    o16, l16 = fa.fa_combine_states(pm, pd, po, o_dtype=torch.bfloat16)
    got_o = o32.cpu().numpy().reshape(rows, D)
    got_b = o16.cpu().view(torch.int16).numpy().reshape(rows, D).view(np.uint16)
    got_l = l32.cpu().numpy().reshape(rows)
    assert (got_o.view(np.uint32) == ref_o.view(np.uint32)).all()
    assert (got_b == ref_b).all()
    assert (got_l.view(np.uint32) == ref_l.view(np.uint32)).all()
    assert torch.equal(l16, l32)


def test_combine_random_states_bit_exact(fa):
    """Random states with identity chunks in arbitrary places, 1000 rows."""
    rng = np.random.default_rng(11)
    rows, S, D = 1000, 16, 128
    m = (rng.standard_normal((rows, S)) * 30).astype(np.float32)
    d = rng.uniform(1, 900, (rows, S)).astype(np.float32)
    o = (rng.standard_normal((rows, S, D)) * 100).astype(np.float32)
    e = rng.uniform(size=(rows, S)) < 0.3
    m[e], d[e], o[e] = -np.inf, 0, 0
    ref_o, ref_b, ref_l = cf.combine_f32(m, d, o)
    go, gl = fa.fa_combine_states(*(torch.from_numpy(x).cuda() for x in (m, d, o)),
                                  o_dtype=torch.float32)
    assert (go.cpu().numpy().view(np.uint32) == ref_o.view(np.uint32)).all()
    assert (gl.cpu().numpy().view(np.uint32) == ref_l.view(np.uint32)).all()
