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
# tensor g with oracle value ref (the gradient formed with the bf16 O the
# backward call is handed, Delta_i = dO_i . O_i as the call defines it), and
# per row r of it (one query or key position, D values):
#   rel-L2(g, ref) <= 1e-2,
#   max_j(|g_rj - ref_rj| - 2^-8 |ref_rj|) <= 2e-2 max_j|ref_rj| + 1e-3 max|ref|.
# The bound of a row follows that row's own magnitude; the second term is an
# absolute floor of a thousandth of the tensor's largest value, for rows whose
# gradient is nearly zero (a key that no query attends to), where the rounded
# terms of the other rows set the error instead.
TOL_BWD_REL_L2 = 1e-2
TOL_BWD_MAX = 2e-2
TOL_BWD_FLOOR = 1e-3


def check_grad(g, ref, what=""):
    """Checks a gradient tensor (last axis = D) row by row; returns the
    largest row excess relative to its bound and the rel-L2 error."""
    g = np.asarray(g, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    if g.size == 0:
        return 0.0, 0.0
    ref = np.asarray(ref, np.float64)
    D = g.shape[-1]
    g2, r2 = g.reshape(-1, D), ref.reshape(-1, D)
    excess = (np.abs(g2 - r2) - BF16_U * np.abs(r2)).max(axis=1)
    bound = TOL_BWD_MAX * np.abs(r2).max(axis=1) + TOL_BWD_FLOOR * float(np.abs(r2).max())
    ratio = excess / np.where(bound > 0, bound, 1.0)
    worst = int(ratio.argmax())
    r = rel_l2(g, ref)
    assert r <= TOL_BWD_REL_L2, f"{what}: rel-L2 {r:.3e} > {TOL_BWD_REL_L2}"
    assert ratio[worst] <= 1.0, (f"{what}: row {worst} excess {excess[worst]:.3e} over its "
                                 f"bound {bound[worst]:.3e} (row max |ref| "
                                 f"{np.abs(r2[worst]).max():.3e})")
    return float(ratio[worst]), r


def check_grad_exact(g, ref, what=""):
    """A gradient tensor against the exact gradient (Delta from the exact O):
    rel-L2 <= 1e-2 and max(|g - ref| - 2^-8 |ref|) <= 2e-2 max|ref| over the
    tensor.  The rows of a bf16 forward output differ from the exact O by one
    rounding, which moves Delta and so each dQ and dK row by an amount that
    does not follow that row's size; the row-by-row bound applies against
    the gradient formed from the O a call is handed (check_grad)."""
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


def report(name: str, **values) -> None:
    """Appends one JSON line {name, values...} to the file named by the
    FA_PARITY_REPORT environment variable (nothing when it is unset), so a
    run can record the measured errors beside its pass/fail."""
    import json
    import os
    path = os.environ.get("FA_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"test": name, **values}) + "\n")


class ErrorStats:
    """Running error statistics of an output against the oracle, gathered
    piece by piece (a head, a sequence) and checked once at the end with the
    bounds above: max |err|, max(|err| - u|ref|) (one bf16 output rounding),
    and the rel-L2 error over everything seen."""

    def __init__(self):
        self.max_abs = 0.0
        self.max_excess = -np.inf
        self.err2 = 0.0
        self.ref2 = 0.0
        self.count = 0
        self.finite = True
        self.worst = None

    def add(self, got, ref, where=None):
        got = np.asarray(got, np.float64)
        ref = np.asarray(ref, np.float64)
        if got.size == 0:
            return
        self.finite &= bool(np.isfinite(got).all())
        err = np.abs(got - ref)
        m = float(err.max())
        if m > self.max_abs:
            self.max_abs = m
            self.worst = (where, np.unravel_index(int(err.argmax()), err.shape))
        self.max_excess = max(self.max_excess, float((err - BF16_U * np.abs(ref)).max()))
        self.err2 += float((err * err).sum())
        self.ref2 += float((ref * ref).sum())
        self.count += got.size

    @property
    def rel_l2(self) -> float:
        return float(np.sqrt(self.err2 / self.ref2)) if self.ref2 > 0 else 0.0

    def summary(self) -> dict:
        return {"elements": self.count, "max_abs": self.max_abs,
                "max_excess_over_u_ref": self.max_excess, "rel_l2": self.rel_l2,
                "worst": repr(self.worst)}


def check_states(pm, pd, po, M, Dn, Oc, what=""):
    """Split-KV chunk states (base 2) against the oracle's: empty chunks are
    exactly the identity (-inf, 0, 0); otherwise m, d and o within 1e-4
    (relative to the largest magnitude), and d >= 1."""
    pm, pd, po = np64(pm), np64(pd), np64(po)
    empty = ~np.isfinite(M)
    assert (pm[empty] == -np.inf).all() and (pd[empty] == 0).all(), what
    assert not po[empty].any(), what
    full = ~empty
    assert np.abs(pm[full] - M[full]).max() <= 1e-4 * max(1.0, np.abs(M[full]).max()), what
    assert np.abs(pd[full] / Dn[full] - 1).max() <= 1e-4, what
    scale = np.abs(Oc[full]).max()
    assert np.abs(po[full] - Oc[full]).max() <= 1e-4 * scale, what
    assert (pd[full] >= 1.0 - 1e-6).all(), what
