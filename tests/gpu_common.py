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
