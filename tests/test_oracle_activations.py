"""Pins for the oracle's gated activations of the expert MLP (Stage 4
activation branches: SwiGLU, clipped SwiGLU-OAI, GeGLU with erf and with the
tanh approximation; reading R15).

Each is pinned by identities the definitions imply (odd symmetry of
x * sigmoid(a x) and of x * Phi(x), zeros, limits, the clipping plateaus) and
by textbook values (the standard normal CDF at 1), none of which restates the
oracle's formula; the grouped MLP is then checked to route the activation
through (dense library matmuls on the same rows).
"""
import math

import numpy as np
import pytest

import oracle
import synth

ACTS = ["swiglu", "swiglu_oai", "geglu", "geglu_tanh"]


def f(act, g, u=1.0):
    return oracle.act_value(act, g, u)


@pytest.mark.parametrize("act", ACTS)
def test_zero_gate_and_zero_up(act):
    for g in (0.0, -0.0):
        assert f(act, g, 3.0) == 0.0
    if act != "swiglu_oai":  # the OAI branch multiplies by (u + 1)
        for g in (-2.0, 0.5, 3.0):
            assert f(act, g, 0.0) == 0.0


@pytest.mark.parametrize("act", ["swiglu", "geglu", "geglu_tanh"])
def test_odd_part_is_identity(act):
    # g*s(g) - (-g)*s(-g) = g when s(g) + s(-g) = 1 (sigmoid, Phi, tanh form)
    for g in np.linspace(-6, 6, 61):
        assert abs(f(act, g) - f(act, -g) - g) <= 1e-12 * max(1.0, abs(g))


def test_oai_odd_part_inside_clip():
    # u = 0 inside the clip: g*sigmoid(1.702 g) - (-g)*sigmoid(-1.702 g) = g
    for g in np.linspace(-6.9, 6.9, 47):
        assert abs(f("swiglu_oai", g, 0.0) - f("swiglu_oai", -g, 0.0) - g) <= 1e-12 * max(1, abs(g))


def test_oai_clipping_plateaus_and_up_offset():
    for u in (-3.0, 0.0, 2.5):
        assert f("swiglu_oai", 9.0, u) == f("swiglu_oai", 7.0, u)   # gate capped at 7
        assert f("swiglu_oai", 50.0, u) == f("swiglu_oai", 7.0, u)
    for g in (-1.0, 0.3, 4.0):
        assert f("swiglu_oai", g, 11.0) == f("swiglu_oai", g, 7.0)  # up clamped to [-7, 7]
        assert f("swiglu_oai", g, -11.0) == f("swiglu_oai", g, -7.0)
        assert f("swiglu_oai", g, -1.0) == 0.0                       # (u + 1) = 0
    # the gate is not clamped from below: large negative gates vanish
    assert abs(f("swiglu_oai", -40.0, 3.0)) < 1e-20


@pytest.mark.parametrize("act", ["geglu", "geglu_tanh"])
def test_gelu_limits_and_slope(act):
    assert abs(f(act, 12.0) - 12.0) < 1e-12
    assert abs(f(act, -12.0)) < 1e-12
    h = 1e-7
    assert abs(f(act, h) / h - 0.5) < 1e-6   # GELU'(0) = Phi(0) = 1/2


def test_gelu_textbook_values():
    # GELU(1) = Phi(1), the standard normal CDF at 1
    assert abs(f("geglu", 1.0) - 0.8413447460685429) < 1e-15
    assert abs(f("geglu", -1.0) - (0.8413447460685429 - 1.0)) < 1e-15
    # the tanh approximation stays within 1e-3 of the exact GELU
    gs = np.linspace(-8, 8, 801)
    d = max(abs(f("geglu_tanh", g) - f("geglu", g)) for g in gs)
    assert 1e-5 < d < 1e-3


def test_silu_textbook_value():
    # silu(1) = 1 / (1 + 1/e)
    assert abs(f("swiglu", 1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


@pytest.mark.parametrize("act", ACTS)
def test_grouped_mlp_applies_the_activation(act, rng):
    H, I, n = 128, 64, 9
    from tests.test_oracle_mlp import _bf16_bits, _f
    x = _bf16_bits(rng.standard_normal((n, H)))
    wg, wu = (_bf16_bits(rng.standard_normal((I, H)) * 0.3) for _ in range(2))
    wd = _bf16_bits(rng.standard_normal((H, I)) * 0.1)
    a, y = oracle.expert_ffn_rows(x, wg, wu, wd, nthreads=2, activation=act)
    g = (_f(x) @ _f(wg).T).astype(np.float32).astype(np.float64)
    u = (_f(x) @ _f(wu).T).astype(np.float32).astype(np.float64)
    ref = np.vectorize(lambda gg, uu: f(act, gg, uu))(g, u)
    a_ref = _bf16_bits(ref)
    d = np.abs(a.astype(np.int32) - a_ref.astype(np.int32))
    assert d.max() <= 1 and np.mean(d == 0) > 0.99
    # the clipped branch really clips on these inputs (|g|, |u| reach > 7)
    if act == "swiglu_oai":
        assert np.abs(g).max() > 7 and np.abs(u).max() > 7
    y_ref = (_f(a) @ _f(wd).T).astype(np.float32)
    assert np.allclose(y, y_ref, rtol=1e-6, atol=1e-6)
