"""Pins for the oracle's latent-MoE tail (NVIDIA LatentMoERunner page, tier 1
"_overlap_allreduce_tail" with one rank: RMSNorm of the routed latent output,
up-projection to the hidden size, shared-expert output added; reading R16).

RMSNorm is pinned by exact power-of-two scale invariance (every step of the
pinned fp32 order scales exactly), by constant rows (the output is the weight
itself), by unit RMS of the output and by a float64 restatement within bf16
rounding; the tail by the identity norm reducing it to a library matmul and by
the shared term entering additively.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.test_oracle_mlp import _bf16_bits, _f


def test_rmsnorm_power_of_two_scale_invariance(rng):
    L = 384
    v = _bf16_bits(rng.standard_normal(L))
    w = _bf16_bits(rng.standard_normal(L))
    z1 = oracle.rmsnorm_row(v, w, 0.0)
    for c in (4.0, 0.25, 1024.0):
        vc = _bf16_bits(_f(v) * c)  # exact: a power of two moves the exponent only
        assert np.array_equal(oracle.rmsnorm_row(vc, w, 0.0), z1)


def test_rmsnorm_constant_row_returns_the_weight(rng):
    L = 256
    w = _bf16_bits(rng.standard_normal(L))
    for c in (1.0, -3.0, 0.5):
        v = _bf16_bits(np.full(L, c))
        z = oracle.rmsnorm_row(v, w, 0.0)
        assert np.array_equal(z, _bf16_bits(np.sign(c) * _f(w)))


def test_rmsnorm_unit_rms_and_float64_restatement(rng):
    L = 1024
    v = _bf16_bits(rng.standard_normal(L) * 3)
    ones = _bf16_bits(np.ones(L))
    z = _f(oracle.rmsnorm_row(v, ones, 1e-6))
    assert abs(np.sqrt(np.mean(z ** 2)) - 1.0) < 4e-3
    w = _bf16_bits(rng.standard_normal(L))
    zr = _f(v) / np.sqrt(np.mean(_f(v) ** 2) + 1e-6) * _f(w)
    z2 = _f(oracle.rmsnorm_row(v, w, 1e-6))
    assert np.all(np.abs(z2 - zr) <= 2.0 ** -8 * np.abs(zr) + 1e-30)


def test_tail_without_norm_is_matmul_plus_shared(rng):
    T, L, Hm = 7, 256, 128
    lat = _bf16_bits(rng.standard_normal((T, L)))
    up = _bf16_bits(rng.standard_normal((Hm, L)) * 0.05)
    sh = _bf16_bits(rng.standard_normal((T, Hm)))
    out = oracle.latent_tail(lat, up, None, shared=sh, nthreads=2)
    ref = _bf16_bits((_f(lat) @ _f(up).T).astype(np.float32).astype(np.float64) + _f(sh))
    d = np.abs(out.astype(np.int32) - ref.astype(np.int32))
    assert d.max() <= 1 and np.mean(d == 0) > 0.99
    # the shared term enters additively
    out0 = oracle.latent_tail(lat, up, None, shared=None, nthreads=2)
    assert np.allclose(_f(out) - _f(out0), _f(sh), atol=2.0 ** -6 * np.abs(_f(out)).max())


def test_tail_uses_the_normalised_rows(rng):
    T, L, Hm = 5, 256, 64
    lat = _bf16_bits(rng.standard_normal((T, L)) * 5)
    w = _bf16_bits(1.0 + 0.1 * rng.standard_normal(L))
    up = _bf16_bits(rng.standard_normal((Hm, L)) * 0.05)
    out = oracle.latent_tail(lat, up, w, eps=1e-6, nthreads=2)
    z = np.stack([oracle.rmsnorm_row(lat[t], w, 1e-6) for t in range(T)])
    ref = oracle.latent_tail(z, up, None, nthreads=2)
    assert np.array_equal(out, ref)
