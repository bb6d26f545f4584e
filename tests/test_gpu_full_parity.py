"""Full-output parity of the benchmark workloads at their full sizes, in the
launch configuration the bench times: every output element against the
float64 oracle on the same seeded inputs.

  * causal prefill, B=1 H=32 N=16384 D=128, Q and K ~ N(0, 9) (scaled scores
    reach the high tens): all 524,288 rows, bf16 and fp32 output, and LSE;
  * split-KV decode, B=64 H=32 D=128, lengths U[1024, 32768], 16 chunks:
    every (sequence, head) row's 16 chunk states, then O (bf16 and fp32
    output) and LSE after the combine;
  * packed causal prefill, 65536 tokens in sequences of lengths U[1, 8192],
    H=16, D=64 and D=128: every row of every sequence and head.

The method reaches the plain result exactly up to rounding ("Learning
FlashAttention the Hard Way - Part 1", "FlashAttention: Not So Special";
"Understanding FlashAttention Pt 1", Introduction: without approximating
attention), so the bounds are the rounding tolerances of tests/gpu_common.py,
applied to every element.  The oracle runs in spawned worker processes, one
head per task.  Set FA_PARITY_REPORT to a file name to record the measured
errors.
"""
import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import attention as ora
from tests import oracle_pool
from tests.gpu_common import (ErrorStats, TOL_LSE, TOL_O, TOL_REL_L2, check_states,
                              np64, report)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _assert_f32(st: ErrorStats, what):
    assert st.finite, f"{what}: non-finite output"
    assert st.max_abs <= TOL_O, f"{what}: max abs {st.max_abs:.3e} > {TOL_O} at {st.worst}"
    assert st.rel_l2 <= TOL_REL_L2, f"{what}: rel-L2 {st.rel_l2:.3e}"


def _assert_bf16(st: ErrorStats, what):
    assert st.finite, f"{what}: non-finite output"
    assert st.max_excess <= TOL_O, \
        f"{what}: max(|err| - u|ref|) {st.max_excess:.3e} > {TOL_O} at {st.worst}"
    assert st.rel_l2 <= TOL_REL_L2, f"{what}: rel-L2 {st.rel_l2:.3e}"


def _assert_lse(st: ErrorStats, what):
    assert st.finite, f"{what}: non-finite LSE"
    assert st.max_abs <= TOL_LSE, f"{what}: LSE max abs {st.max_abs:.3e} at {st.worst}"


def test_config3_full(fa):
    case = inp.config3(device="cuda")
    B, H, N, D = case.q.shape
    scale = case.scale
    o16, lse16 = fa.fa_fwd(case.q, case.k, case.v, case.scale, True)
    o32, lse32 = fa.fa_fwd_ex(case.q, case.k, case.v, case.scale, True, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    # the bf16 output is the nearest-even rounding of the fp32 one
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(lse16, lse32)
    g16, g32, gl = np64(o16[0]), np64(o32[0]), np64(lse32[0])
    qc, kc, vc = (t[0].float().cpu().numpy() for t in (case.q, case.k, case.v))
    del o16, o32, lse16, lse32, case
    s32, s16, sl = ErrorStats(), ErrorStats(), ErrorStats()
    lse_max = -np.inf
    tasks = [(qc[h], kc[h], vc[h], scale, True) for h in range(H)]
    with oracle_pool.pool() as p:
        for h, (O, L) in enumerate(p.imap(oracle_pool.head_ref, tasks)):
            s32.add(g32[h], O, ("head", h))
            s16.add(g16[h], O, ("head", h))
            sl.add(gl[h], L, ("head", h))
            lse_max = max(lse_max, float(L.max()))
    report("config3_full", rows=B * H * N, o_f32=s32.summary(), o_bf16=s16.summary(),
           lse=sl.summary(), oracle_lse_max=lse_max)
    assert s32.count == B * H * N * D and sl.count == B * H * N
    _assert_f32(s32, "config3 fp32-out")
    _assert_bf16(s16, "config3 bf16")
    _assert_lse(sl, "config3")
    # the scores really are in the overflow range of a naive fp32 exp
    assert lse_max > 40.0


def test_config4_full(fa):
    case = inp.config4(device="cuda")
    B, H, D = case.q.shape
    S = case.num_splits
    cu = case.cu_seqlens_k.cuda()
    pm, pd, po = fa.fa_decode_splitkv(case.q, case.k_cache, case.v_cache, cu, S, case.scale)
    o16, lse16 = fa.fa_combine_states(pm, pd, po)
    o32, lse32 = fa.fa_combine_states(pm, pd, po, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(lse16, lse32)
    cuh = case.cu_seqlens_k.tolist()
    s32, s16, sl = ErrorStats(), ErrorStats(), ErrorStats()
    for b in range(B):
        a, e = cuh[b], cuh[b + 1]
        kc = case.k_cache[a:e].cpu().double().numpy()
        vc = case.v_cache[a:e].cpu().double().numpy()
        q = case.q[b:b + 1].cpu().double().numpy()
        cu1 = np.array([0, e - a])
        M, Dn, Oc = ora.chunk_states_ref(q, kc, vc, cu1, S, case.scale)
        check_states(pm[b:b + 1], pd[b:b + 1], po[b:b + 1], M, Dn, Oc, f"states b={b}")
        O, L = ora.decode_ref(q, kc, vc, cu1, case.scale)
        s32.add(np64(o32[b:b + 1]), O, ("seq", b))
        s16.add(np64(o16[b:b + 1]), O, ("seq", b))
        sl.add(np64(lse32[b:b + 1]), L, ("seq", b))
    report("config4_full", rows=B * H, o_f32=s32.summary(), o_bf16=s16.summary(),
           lse=sl.summary())
    assert sl.count == B * H
    _assert_f32(s32, "config4 fp32-out")
    _assert_bf16(s16, "config4 bf16")
    _assert_lse(sl, "config4")


@pytest.mark.parametrize("D", [64, 128])
def test_config5_full(fa, D):
    case = inp.config5(D)
    T, H, _ = case.q.shape
    o, lse = fa.fa_fwd_varlen(case.q.cuda(), case.k.cuda(), case.v.cuda(),
                              case.cu_seqlens.cuda(), case.max_seqlen, case.scale, True)
    torch.cuda.synchronize()
    assert fa.fa_check_device_status() == fa.FA_OK
    go, gl = np64(o), np64(lse)
    cuh = case.cu_seqlens.tolist()
    qf, kf, vf = (t.float().numpy() for t in (case.q, case.k, case.v))
    tasks, where = [], []
    for s in range(len(cuh) - 1):
        a, b = cuh[s], cuh[s + 1]
        for h in range(H):
            tasks.append((np.ascontiguousarray(qf[a:b, h]), np.ascontiguousarray(kf[a:b, h]),
                          np.ascontiguousarray(vf[a:b, h]), case.scale, True))
            where.append((s, h, a, b))
    s16, sl = ErrorStats(), ErrorStats()
    with oracle_pool.pool() as p:
        for (s, h, a, b), (O, L) in zip(where, p.imap(oracle_pool.head_ref, tasks)):
            s16.add(go[a:b, h], O, ("seq", s, "head", h))
            sl.add(gl[h, a:b], L, ("seq", s, "head", h))
    report(f"config5_full_D{D}", rows=T * H, seqs=len(cuh) - 1, o_bf16=s16.summary(),
           lse=sl.summary())
    assert s16.count == T * H * D and sl.count == T * H
    _assert_bf16(s16, f"config5 D={D} bf16")
    _assert_lse(sl, f"config5 D={D}")
