"""Shared helpers of the GPU parity tests: tolerances and error measures.

Tolerances (bf16 inputs, fp32 accumulation), against the float64 oracle:
  * fp32 output of the bf16 kernel: max |O - ref| <= 1e-2, rel-L2 <= 5e-3;
  * bf16 output: max(|O - ref| - 2^-8 |ref|) <= 1e-2 (the 1e-2 bound on top
    of one bf16 rounding of the output, unit roundoff 2^-8), rel-L2 <= 5e-3;
  * LSE: max abs <= 1e-3;
  * fp32 path: max abs <= 1e-5 on O and LSE.
"""
import numpy as np
import torch

BF16_U = 2.0 ** -8
TOL_O = 1e-2
TOL_REL_L2 = 5e-3
TOL_LSE = 1e-3
TOL_F32 = 1e-5


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def rel_l2(a, ref) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def check_o_f32(o, ref, what=""):
    o = np.asarray(o, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref).max() if o.size else 0.0
    r = rel_l2(o, ref)
    assert err <= TOL_O, f"{what}: max abs {err:.3e} > {TOL_O}"
    assert r <= TOL_REL_L2, f"{what}: rel-L2 {r:.3e} > {TOL_REL_L2}"
    return err, r


def check_o_bf16(o, ref, what=""):
    o = np.asarray(o, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    if o.size == 0:
        return 0.0, 0.0
    excess = (np.abs(o - ref) - BF16_U * np.abs(ref)).max()
    r = rel_l2(o, ref)
    assert excess <= TOL_O, f"{what}: max(|err| - u|ref|) {excess:.3e} > {TOL_O}"
    assert r <= TOL_REL_L2, f"{what}: rel-L2 {r:.3e} > {TOL_REL_L2}"
    return float(np.abs(o - ref).max()), r


def check_lse(lse, ref, tol=TOL_LSE, what=""):
    lse = np.asarray(lse, np.float64)
    assert np.isfinite(lse).all(), f"{what}: non-finite LSE"
    err = np.abs(lse - ref).max() if lse.size else 0.0
    assert err <= tol, f"{what}: LSE max abs {err:.3e} > {tol}"
    return err


# Backward (bf16 inputs, P and dS rounded to bf16 before their products, fp32
# accumulation, bf16 gradients), against the float64 oracle on the same
# inputs.  The kernel's Delta uses its own bf16 O, the oracle the exact one.
# Three roundings of relative size up to 2^-9 each (P or dS, the bf16 O in
# Delta, the bf16 gradient) meet in every element.  The rows of dS sum to
# zero (sum_j P_ij (dP_ij - Delta_i) = 0), so dQ = scale dS K is a small
# residual of up to N rounded terms and its relative error grows with N
# (measured: about 2.5e-3 at N <= 1024, 6.3e-3 at N = 16384).  Per gradient
# tensor g with oracle value ref:
#   rel-L2(g, ref) <= 1e-2,
#   max(|g - ref| - 2^-8 |ref|) <= 2e-2 * max|ref|.
TOL_BWD_REL_L2 = 1e-2
TOL_BWD_MAX = 2e-2


def check_grad(g, ref, what=""):
    g = np.asarray(g, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    if g.size == 0:
        return 0.0, 0.0
    scale = float(np.abs(ref).max()) or 1.0
    excess = float((np.abs(g - ref) - BF16_U * np.abs(ref)).max()) / scale
    r = rel_l2(g, ref)
    assert r <= TOL_BWD_REL_L2, f"{what}: rel-L2 {r:.3e} > {TOL_BWD_REL_L2}"
    assert excess <= TOL_BWD_MAX, f"{what}: max excess {excess:.3e} x max|ref| > {TOL_BWD_MAX}"
    return excess, r
