"""Pins for the oracle's elementary functions (Stage 2 scoring functions).

Each pinned function is checked against the library's double-precision
routine (numpy / math) within a stated ulp bound, plus the special values the
mathematics fixes.  A wrong Taylor coefficient, a missing reduction term or a
sign error fails these by many ulps.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _ulp_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    sp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.abs(got - ref) / sp


def _vec(f, xs):
    return np.array([f(float(v)) for v in xs], dtype=np.float32)


def _sweep(lo, hi, n, rng):
    xs = np.concatenate([np.linspace(lo, hi, n // 2), rng.uniform(lo, hi, n // 2)])
    return xs.astype(np.float32)


def test_exp_within_2ulp(rng):
    xs = _sweep(-87.0, 88.5, 40000, rng)
    got = _vec(oracle.exp, xs)
    ref = np.exp(xs.astype(np.float64))
    assert _ulp_err(got, ref).max() <= 2.0


def test_exp_special_values():
    assert oracle.exp(0.0) == 1.0
    assert oracle.exp(89.0) == math.inf
    assert oracle.exp(-100.0) == 0.0
    assert math.isnan(oracle.exp(math.nan))
    # e^1 and e^-1 to within an ulp of the correctly rounded value
    assert _ulp_err([oracle.exp(1.0)], [math.e])[0] <= 1.0
    assert _ulp_err([oracle.exp(-1.0)], [1 / math.e])[0] <= 1.0


def test_exp_is_monotone_on_a_dense_grid():
    xs = np.linspace(-20.0, 20.0, 200001).astype(np.float32)
    ys = _vec(oracle.exp, xs)
    assert np.all(np.diff(ys.astype(np.float64)) >= 0)


def test_log1p_within_2ulp(rng):
    ys = np.concatenate([_sweep(0.0, 1.0, 20000, rng), np.float32([1e-30, 1e-8, 1e-3])])
    got = _vec(oracle.log1p, ys)
    ref = np.log1p(ys.astype(np.float64))
    ok = ref > 0
    assert _ulp_err(got[ok], ref[ok]).max() <= 2.0
    assert oracle.log1p(0.0) == 0.0


def test_sigmoid_within_3ulp_and_symmetry(rng):
    xs = _sweep(-80.0, 80.0, 40000, rng)
    got = _vec(oracle.sigmoid, xs)
    ref = 1.0 / (1.0 + np.exp(-xs.astype(np.float64)))
    assert _ulp_err(got, ref).max() <= 3.0
    assert oracle.sigmoid(0.0) == 0.5
    # sigma(x) + sigma(-x) = 1
    s = got.astype(np.float64) + _vec(oracle.sigmoid, -xs).astype(np.float64)
    assert np.abs(s - 1.0).max() <= 2.5e-7


def test_sqrtsoftplus_within_3ulp(rng):
    ls = _sweep(-60.0, 60.0, 40000, rng)
    got = _vec(oracle.sqrtsoftplus, ls)
    l64 = ls.astype(np.float64)
    ref = np.sqrt(np.maximum(l64, 0) + np.log1p(np.exp(-np.abs(l64))))
    assert _ulp_err(got, ref).max() <= 3.0
    assert _ulp_err([oracle.sqrtsoftplus(0.0)], [math.sqrt(math.log(2.0))])[0] <= 1.0


def test_bf16_rounding_matches_torch(rng):
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 3,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 3.4e38,
                                    1e-40, -2.5])])
    # exact ties: the halfway points between adjacent bf16 values
    ties = ((np.arange(1, 200, dtype=np.uint32) << 16) | 0x3F808000).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    got = np.array([oracle.f32_to_bf16(float(a)) for a in v], dtype=np.uint16)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
