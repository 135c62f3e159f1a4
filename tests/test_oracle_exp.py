"""Pins of the oracle's own fp32 exp against libm and its stated special values.

The bound is one ulp (faithful rounding): the polynomial truncation error is
about 0.12 ulp and Horner evaluation adds well under one more.

The oracle computes softmax weights with csa_oracle_exp_f32 (Cody-Waite reduction
plus a degree-7 Taylor polynomial), so that the CUDA library can evaluate the
same function bit for bit.  Here it is checked against the platform exp in fp64.
"""
import math

import numpy as np
import pytest

import oracle


def ulps(got, ref):
    ref32 = ref.astype(np.float32)
    return np.abs(got.astype(np.float64) - ref) / np.spacing(np.abs(ref32)).astype(np.float64)


def test_exp_accuracy_dense_sweep():
    # 40001 points over the range where the result is a normal float.
    xs = np.linspace(-87.0, 0.0, 40001).astype(np.float32)
    got = oracle.exp_f32(xs)
    ref = np.exp(xs.astype(np.float64))
    assert ulps(got, ref).max() <= 1.0  # faithful: within one ulp of the true value


def test_exp_accuracy_near_zero_and_at_integers_of_ln2():
    xs = np.concatenate([
        -np.logspace(-12, 0, 2000),
        -np.arange(1, 126) * math.log(2.0),
        -(np.arange(1, 126) + 0.5) * math.log(2.0),
    ]).astype(np.float32)
    got = oracle.exp_f32(xs)
    ref = np.exp(xs.astype(np.float64))
    assert ulps(got, ref).max() <= 1.0  # faithful: within one ulp of the true value


def test_exp_special_values():
    got = oracle.exp_f32(np.array([0.0, -0.0, -np.inf, np.nan, -88.0, -100.0, -1e30], np.float32))
    assert got[0] == 1.0 and got[1] == 1.0
    assert got[2] == 0.0 and not np.signbit(got[2])
    assert np.isnan(got[3])
    assert got[4] == 0.0 and got[5] == 0.0 and got[6] == 0.0


def test_exp_subnormal_edge_is_tiny_and_nonnegative():
    # Between -87.68 and -87 results fall near 2^-126; they must be within a few
    # subnormal steps of the true value, and never negative.
    xs = np.linspace(-87.9, -86.9, 2001).astype(np.float32)
    got = oracle.exp_f32(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    assert (got >= 0).all()
    flushed = xs < -87.6
    assert np.all(np.abs(got[~flushed] - ref[~flushed]) <= 2 * np.spacing(np.float32(ref[~flushed].max())))
    assert np.all(got[flushed] <= 2.0 ** -126)


def test_exp_monotone_on_sweep():
    xs = np.linspace(-20.0, 0.0, 20001).astype(np.float32)
    got = oracle.exp_f32(xs)
    assert np.all(np.diff(got.astype(np.float64)) >= 0)


@pytest.mark.parametrize("x", [-1e-7, -0.5, -0.3465736, -0.3465737, -1.0, -10.0, -50.0, -86.0])
def test_exp_points(x):
    got = float(oracle.exp_f32(np.array([x], np.float32))[0])
    ref = math.exp(float(np.float32(x)))
    assert abs(got - ref) <= 2 * float(np.spacing(np.float32(ref)))
