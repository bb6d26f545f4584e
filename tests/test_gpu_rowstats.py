"""GPU parity of the Welford row statistics (fa_row_stats, the split-K
partials and the combine) against the float64 oracle, and of the combine
against the fixed-order C fp32 fold bit for bit."""
import numpy as np
import pytest
import torch

import fa_inputs as inp
from oracle import combine_f32 as cf
from oracle import welford as wf
from tests.gpu_common import np64

pytestmark = pytest.mark.gpu

# fp32 accumulation against float64.  With a row mean mu and spread sigma,
# the pack means and merge deltas carry absolute errors ~ u (|mu| + sigma),
# u = 2^-24, so the variance's relative error grows with 1 + |mu| / sigma and
# with the merge depth (log2 C levels).  Bounds:
#   |mean - ref| <= 1e-5 (|mu| + sigma)
#   |var - ref|  <= 1e-5 (1 + |mu| / sigma) var
#   |rstd - ref| <= 1e-5 (1 + |mu| / sigma) rstd
TOL = 1e-5


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    return fa


def _check(mean, var, rstd, x, eps, what):
    rm, rv, rr = wf.row_stats_ref(x, eps)
    sig = np.sqrt(rv)
    k = 1.0 + np.abs(rm) / np.maximum(sig, 1e-30)
    m, v, r = np64(mean), np64(var), np64(rstd)
    assert np.isfinite(m).all() and np.isfinite(v).all()
    assert (np.abs(m - rm) <= TOL * (np.abs(rm) + sig) + 1e-30).all(), f"{what}: mean"
    assert (np.abs(v - rv) <= TOL * k * rv + 1e-30).all(), f"{what}: var"
    assert (np.abs(r - rr) <= TOL * k * rr).all(), f"{what}: rstd"


SHAPES = [(1, 1), (3, 7), (5, 8), (17, 100), (8, 2047), (8, 2048), (64, 4096), (4, 10000),
          (2, 65537)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C", SHAPES)
def test_row_stats(fa, R, C, dtype):
    x = inp.stats_rows(R, C, seed=R * 31 + C, loc=3.0, std=2.0, row_spread=1.0, dtype=dtype)
    mean, var, rstd = fa.fa_row_stats(x.cuda(), eps=1e-5)
    _check(mean, var, rstd, x, 1e-5, f"{R}x{C} {dtype}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_row_stats_unaligned_rows(fa, dtype):
    """Rows that start off a 16-byte boundary take the scalar head path."""
    R, C = 6, 301
    x = inp.stats_rows(R, C, seed=77, loc=-1.0, std=0.5, dtype=dtype)
    buf = torch.empty(R * C + 1, dtype=dtype, device="cuda")
    xv = buf[1:].view(R, C)
    xv.copy_(x.cuda())
    assert xv.data_ptr() % 16 != 0
    mean, var, rstd = fa.fa_row_stats(xv, eps=0.0)
    _check(mean, var, rstd, x, 0.0, "unaligned")


def test_offset_rows_stay_accurate(fa):
    """Mean 100 sigma: the one-pass sum of squares would lose the variance."""
    x = inp.stats_rows(16, 4096, seed=5, loc=100.0, std=1.0, dtype=torch.float32)
    mean, var, rstd = fa.fa_row_stats(x.cuda())
    _check(mean, var, rstd, x, 0.0, "offset")


def test_constant_rows_and_single_column(fa):
    x = torch.full((4, 1000), 2.5, dtype=torch.bfloat16, device="cuda")
    mean, var, rstd = fa.fa_row_stats(x, eps=1e-2)
    assert (mean == 2.5).all() and (var == 0).all()
    assert torch.equal(rstd, torch.full_like(rstd, float(np.float32(1) / np.sqrt(np.float32(1e-2)))))
    y = inp.stats_rows(9, 1, seed=3, dtype=torch.float32)
    mean, var, _ = fa.fa_row_stats(y.cuda())
    assert torch.equal(mean.cpu(), y[:, 0]) and (var == 0).all()


@pytest.mark.parametrize("S", [1, 3, 64, 700])
def test_partials_and_combine(fa, S):
    R, C = 12, 5000
    x = inp.stats_rows(R, C, seed=S, loc=1.0, std=3.0, row_spread=2.0, dtype=torch.bfloat16)
    pn, pm, p2 = fa.fa_row_stats_partials(x.cuda(), S)
    n, mu, m2 = wf.chunk_states_ref(x, S)
    assert np.array_equal(np64(pn), n)
    live = n > 0
    assert np.allclose(np64(pm)[live], mu[live], rtol=0, atol=1e-5 * (1 + np.abs(mu).max()))
    assert np.allclose(np64(p2)[live], m2[live], rtol=1e-4, atol=1e-4)
    assert (np64(pm)[~live] == 0).all() and (np64(p2)[~live] == 0).all()
    mean, var, rstd = fa.fa_row_stats_combine(pn, pm, p2, eps=1e-5)
    _check(mean, var, rstd, x, 1e-5, f"split {S}")


def test_combine_bit_exact_with_c_fold(fa):
    """Seeded chunk states (from the float64 oracle, rounded to fp32; some
    chunks empty): the GPU fold equals the C fp32 fold bit for bit."""
    x = inp.stats_rows(50, 999, seed=8, loc=-2.0, std=1.5, row_spread=3.0, dtype=torch.float32)
    n, mu, m2 = (a.astype(np.float32) for a in wf.chunk_states_ref(x, 1200))
    assert (n == 0).any()
    em, ev, er = cf.welford_combine_f32(n, mu, m2, eps=1e-3)
    t = [torch.from_numpy(a).cuda() for a in (n, mu, m2)]
    gm, gv, gr = fa.fa_row_stats_combine(*t, eps=1e-3)
    assert np.array_equal(gm.cpu().numpy().view(np.uint32), em.view(np.uint32))
    assert np.array_equal(gv.cpu().numpy().view(np.uint32), ev.view(np.uint32))
    assert np.array_equal(gr.cpu().numpy().view(np.uint32), er.view(np.uint32))


def test_deterministic_and_full_size_sampled(fa):
    """LayerNorm statistics of 4 x 16384 tokens at hidden size 4096 (bf16):
    sampled rows against the oracle; two runs give the same bits."""
    R, C = 65536, 4096
    x = inp.stats_rows(R, C, seed=11, loc=0.5, std=1.0, row_spread=1.0, dtype=torch.bfloat16,
                       device="cuda")
    a = fa.fa_row_stats(x, eps=1e-5)
    b = fa.fa_row_stats(x, eps=1e-5)
    for u, w in zip(a, b):
        assert torch.equal(u, w)
    rows = np.random.default_rng(0).choice(R, 300, replace=False)
    rows = np.concatenate([[0, R - 1], rows])
    xs = x[torch.from_numpy(rows).cuda()].cpu()
    _check(a[0][rows], a[1][rows], a[2][rows], xs, 1e-5, "full size")


def test_invalid_args(fa):
    lib = fa.load_library()
    x = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    o = torch.zeros(4, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    p, q = x.data_ptr(), o.data_ptr()
    assert lib.fa_row_stats(p, 4, 0, fa.FA_DTYPE_F32, 0.0, q, q, q, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_row_stats(p, 4, 8, 7, 0.0, q, q, q, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_row_stats(p, 4, 8, fa.FA_DTYPE_F32, -1.0, q, q, q, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_row_stats(p + 2, 4, 8, fa.FA_DTYPE_F32, 0.0, q, q, q, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_row_stats(p, 0, 8, fa.FA_DTYPE_F32, 0.0, None, None, None, s) == fa.FA_OK
    assert lib.fa_row_stats_partials(p, 4, 8, fa.FA_DTYPE_F32, 0, q, q, q, s) == \
        fa.FA_ERR_INVALID_ARG
    assert lib.fa_row_stats_workspace_bytes(3, 5) == 3 * 3 * 5 * 4
