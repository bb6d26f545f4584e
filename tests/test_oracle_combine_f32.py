"""Pins of the plain C fp32 combine (the bit-exact reference of the split-KV
state fold).

Its two textbook kernels are checked against the correctly rounded values of
2^x and ln x (Python's math library in double, rounded once), and its fold
against the float64 fold of the same fp32 states, against the hand-worked
base-2 example, and against exact properties (identity law, one chunk).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as ora
from oracle import combine_f32 as cf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def ulp_diff(a: float, b: float) -> int:
    ia = np.array([a], np.float32).view(np.int32)[0]
    ib = np.array([b], np.float32).view(np.int32)[0]
    return abs(int(ia) - int(ib))


def test_exp2_exact_points():
    for n in range(-126, 1):
        assert cf.exp2f(float(n)) == 2.0 ** n
    assert cf.exp2f(-200.0) == 0.0
    assert cf.exp2f(-126.5) == 0.0


def test_exp2_accuracy_sweep():
    xs = np.concatenate([np.linspace(-126, 0, 20001, dtype=np.float32),
                         -np.abs(np.random.default_rng(0).standard_normal(5000)
                                 .astype(np.float32)) * 30])
    worst = 0
    for x in xs.tolist():
        x32 = float(np.float32(x))
        ref = float(np.float32(2.0 ** x32))
        if ref < 2.0 ** -126:
            continue  # subnormal results are outside the stated range
        worst = max(worst, ulp_diff(cf.exp2f(x32), ref))
    assert worst <= 2, worst


def test_ln_accuracy_sweep():
    rng = np.random.default_rng(1)
    xs = np.concatenate([np.float32(1.0) + np.arange(2000, dtype=np.float32) * np.float32(1e-3),
                         np.exp(rng.uniform(0, 20, 5000)).astype(np.float32)])
    assert cf.lnf(1.0) == 0.0
    worst = 0
    for x in xs.tolist():
        x32 = float(np.float32(x))
        ref = math.log(x32)
        got = cf.lnf(x32)
        # relative error against the double value, in fp32 ulps of the result
        if abs(ref) < 1e-6:
            assert abs(got - ref) < 1e-7
            continue
        worst = max(worst, ulp_diff(got, float(np.float32(ref))))
    assert worst <= 3, worst


def _random_states(rows, S, D, seed, empty_frac=0.2):
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal((rows, S)) * 20).astype(np.float32)
    d = rng.uniform(1.0, 500.0, (rows, S)).astype(np.float32)
    o = (rng.standard_normal((rows, S, D)) * 30).astype(np.float32)
    empty = rng.uniform(size=(rows, S)) < empty_frac
    m[empty] = -np.inf
    d[empty] = 0.0
    o[empty] = 0.0
    return m, d, o


@pytest.mark.parametrize("S", [1, 2, 16, 37])
def test_combine_against_float64_fold(S):
    m, d, o = _random_states(64, S, 128, S)
    O, Ob, L = cf.combine_f32(m, d, o)
    Or, Lr = ora.combine_ref(m.astype(np.float64), d.astype(np.float64),
                             o.astype(np.float64))
    full = np.isfinite(Lr)
    np.testing.assert_allclose(O[full], Or[full], rtol=2e-5, atol=1e-5)
    np.testing.assert_allclose(L[full], Lr[full], rtol=1e-6, atol=1e-5)
    assert (L[~full] == -np.inf).all() and not O[~full].any()
    # bf16 output is the round-to-nearest-even of the fp32 output
    bf = (Ob.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_allclose(bf, O, rtol=2.0 ** -8, atol=0)


def test_combine_hand_example():
    with open(GOLDEN) as f:
        g = json.load(f)["base2_states"]
    st = g["states"]
    m = np.array([[float(Fraction(s["m"])) for s in st]], np.float32)
    d = np.array([[float(Fraction(s["d"])) for s in st]], np.float32)
    o = np.array([[[float(Fraction(x)) for x in s["o"]] for s in st]], np.float32)
    O, _, L = cf.combine_f32(m, d, o)
    exp_O = [float(Fraction(x)) for x in g["O"]]
    np.testing.assert_allclose(O[0], exp_O, rtol=2e-7)
    assert abs(L[0] - math.log(11.0)) < 4e-7


def test_identity_chunks_change_no_bit():
    """Interleaving empty chunks (the identity) anywhere leaves every output
    bit unchanged, and chunk order among non-empty chunks is fixed."""
    m, d, o = _random_states(32, 8, 64, 5, empty_frac=0.0)
    O1, B1, L1 = cf.combine_f32(m, d, o)
    S2 = 13
    m2 = np.full((32, S2), -np.inf, np.float32)
    d2 = np.zeros((32, S2), np.float32)
    o2 = np.zeros((32, S2, 64), np.float32)
    pos = [0, 2, 3, 5, 8, 9, 11, 12]
    m2[:, pos], d2[:, pos], o2[:, pos] = m, d, o
    O2, B2, L2 = cf.combine_f32(m2, d2, o2)
    assert (O1.view(np.int32) == O2.view(np.int32)).all()
    assert (B1 == B2).all() and (L1.view(np.int32) == L2.view(np.int32)).all()


def test_one_chunk_is_a_single_division():
    m, d, o = _random_states(16, 1, 32, 9, empty_frac=0.0)
    O, _, _ = cf.combine_f32(m, d, o)
    exp = o[:, 0, :] / d[:, 0:1]  # numpy float32 division is correctly rounded
    assert (O.view(np.int32) == exp.view(np.int32)).all()
