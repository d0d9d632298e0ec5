"""Pins for the oracle's MX block-scaled expert path (Stage 4 quantized
paths, MXFP and W4A8; reading R18: OCP Microscaling blocks of 32 elements
with a power-of-two UE8M0 scale, E4M3 or E2M1 elements).

Pinned against facts fixed by the format definitions, not by restating the
oracle: the E2M1 value set and its ties, the block exponent on worked blocks
(largest magnitude at and around the top of the element range), the
quantization error bound on random blocks, the nibble packing order, and the
grouped MLP against dense library matmuls of the dequantized operands.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_mlp import _bf16_bits, _f

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def deq(q, sc, fmt):
    """Dequantize MX codes with numpy (independent of the oracle's C path)."""
    q = np.asarray(q)
    if fmt == "e2m1":
        lo, hi = q & 15, q >> 4
        codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
        mag = np.array(E2M1)[codes & 7]
        v = np.where(codes & 8, -mag, mag)
    else:
        v = np.vectorize(oracle.e4m3_to_f32)(q).astype(np.float64)
    scale = np.exp2(np.asarray(sc, np.float64) - 127.0)
    return v * np.repeat(scale, 32, axis=1)


def test_e2m1_values():
    for c in range(16):
        want = E2M1[c & 7] * (-1 if c & 8 else 1)
        assert oracle.e2m1_to_f32(c) == want
        assert oracle.f32_to_e2m1(want) == (c if c != 8 else 8)


@pytest.mark.parametrize("x, code", [
    (0.25, 0), (0.2500001, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6),
    (5.0, 6), (5.0001, 7), (6.5, 7), (1e30, 7), (0.1, 0), (-0.75, 10), (-5.0, 14), (-0.0, 8),
])
def test_e2m1_rounding_ties_to_even(x, code):
    assert oracle.f32_to_e2m1(x) == code


def test_block_exponent_worked_blocks():
    # E4M3: largest binade 2^8 (448 = 1.75 * 2^8); E2M1: 2^2 (6 = 1.5 * 2^2)
    assert oracle.mx_block_exp(1.0, "e4m3") == -8
    assert oracle.mx_block_exp(448.0, "e4m3") == 0
    assert oracle.mx_block_exp(511.0, "e4m3") == 0
    assert oracle.mx_block_exp(512.0, "e4m3") == 1
    assert oracle.mx_block_exp(6.0, "e2m1") == 0
    assert oracle.mx_block_exp(7.9, "e2m1") == 0
    assert oracle.mx_block_exp(1.0, "e2m1") == -2
    assert oracle.mx_block_exp(0.0, "e4m3") == 0
    assert oracle.mx_block_exp(2.0 ** -130, "e4m3") == -127       # clamped


def test_worked_rows():
    row = np.zeros((1, 64), np.float64)
    row[0, 0], row[0, 1], row[0, 2] = 1.0, -0.5, 2.0 ** -9   # block 0: amax 1
    row[0, 32], row[0, 33] = 480.0, 3.0                       # block 1: amax 480
    q, sc = oracle.mx_quantize_rows(_bf16_bits(row), "e4m3")
    assert list(sc[0]) == [127 - 8, 127]
    # 1 / 2^-8 = 256 = 2^8 (exponent field 15, mantissa 0); -0.5 -> -128;
    # 2^-9 -> 2^-1 (exponent field 6); 480 saturates to 448 (0x7e); 3 -> 0x44
    assert q[0, 0] == 0x78 and q[0, 1] == 0xF0 and q[0, 2] == 0x30
    assert q[0, 32] == 0x7E and q[0, 33] == 0x44
    assert np.all(q[0, 3:32] == 0) and np.all(sc[0] <= 127)
    z, zs = oracle.mx_quantize_rows(np.zeros((2, 32), np.uint16), "e2m1")
    assert np.all(z == 0) and np.all(zs == 127)               # all-zero blocks: scale 1


def test_e2m1_packing_order():
    row = np.zeros((1, 32))
    row[0, :4] = [6.0, 1.0, -0.5, 4.0]                        # amax 6: scale 1
    q, sc = oracle.mx_quantize_rows(_bf16_bits(row), "e2m1")
    assert sc[0, 0] == 127
    assert q[0, 0] == (7 | (2 << 4)) and q[0, 1] == (9 | (6 << 4))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_quantization_error_bound(fmt, rng):
    x = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, (64, 1)))
    xb = _bf16_bits(x)
    v = _f(xb)
    q, sc = oracle.mx_quantize_rows(xb, fmt)
    d = deq(q, sc, fmt)
    # largest binade, mantissa bits, smallest normal binade of the element format
    top, mbits, emin = (8, 3, -6) if fmt == "e4m3" else (2, 1, 0)
    for b in range(v.shape[1] // 32):
        blk = v[:, 32 * b:32 * (b + 1)]
        amax = np.abs(blk).max(axis=1)
        e = np.floor(np.log2(amax)) - top
        assert np.array_equal(sc[:, b].astype(int) - 127, e.astype(int))
        # |v - deq| <= half the element spacing at |v| (after scaling), or
        # the value saturated at the format maximum
        X = np.exp2(e)[:, None]
        r = np.abs(blk) / X
        binade = np.floor(np.log2(np.maximum(r, 1e-300)))
        spacing = np.exp2(np.maximum(binade, emin) - mbits)
        err = np.abs(blk - d[:, 32 * b:32 * (b + 1)]) / X
        vmax = 448.0 if fmt == "e4m3" else 6.0
        ok = (err <= 0.5 * spacing + 1e-12) | (r > vmax)
        assert ok.all()


@pytest.mark.parametrize("wfmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_grouped_mlp_matches_dense_matmuls(wfmt, act, rng):
    H, I, P = 128, 64, 3
    rows = [5, 0, 7]
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N, T = int(offs[-1]), 9
    x = _bf16_bits(rng.standard_normal((T, H)))
    r2t = rng.integers(0, T, N).astype(np.int32)
    W = [[_bf16_bits(rng.standard_normal(sh) * 0.1) for sh in ((I, H), (I, H), (H, I))]
         for _ in range(P)]
    xq, xs = oracle.mx_quantize_rows(x, "e4m3")
    qw = [[oracle.mx_quantize_rows(w, wfmt) for w in ws] for ws in W]
    st = lambda j, k: np.stack([q[j][k] for q in qw])  # noqa: E731
    a, aq, as_, y = oracle.ffn_grouped_mx(xq, xs, r2t, offs, st(0, 0), st(0, 1), st(1, 0),
                                          st(1, 1), st(2, 0), st(2, 1), wfmt=wfmt, nthreads=2,
                                          activation=act)
    xd = deq(xq, xs, "e4m3")
    for p in range(P):
        r0, r1 = offs[p], offs[p + 1]
        if r0 == r1:
            continue
        wgd, wud, wdd = (deq(qw[p][j][0], qw[p][j][1], wfmt) for j in range(3))
        g = (xd[r2t[r0:r1]] @ wgd.T).astype(np.float32).astype(np.float64)
        u = (xd[r2t[r0:r1]] @ wud.T).astype(np.float32).astype(np.float64)
        ref = _bf16_bits(np.vectorize(lambda gg, uu: oracle.act_value(act, gg, uu))(g, u))
        dd = np.abs(a[r0:r1].astype(np.int32) - ref.astype(np.int32))
        assert dd.max() <= 1 and np.mean(dd == 0) > 0.99
        # the activation codes are the MX E4M3 quantization of the bf16 activation
        q2, s2 = oracle.mx_quantize_rows(a[r0:r1], "e4m3")
        assert np.array_equal(aq[r0:r1], q2) and np.array_equal(as_[r0:r1], s2)
        y_ref = deq(aq[r0:r1], as_[r0:r1], "e4m3") @ wdd.T
        assert np.allclose(y[r0:r1], y_ref, rtol=1e-6, atol=1e-30)


def test_e2m1_matches_brute_force_nearest(rng):
    """Every value against a search over the eight magnitudes: the nearest,
    ties to the even code, beyond 6 saturated; the sign kept (also on zero)."""
    mids = [0.5 * (a + b) for a, b in zip(E2M1[:-1], E2M1[1:])]
    vals = np.concatenate([rng.uniform(-8, 8, 3000), mids, [-m for m in mids], E2M1,
                           [6.0001, 7.999, -1e-7]]).astype(np.float32)
    mags = np.array(E2M1)
    for v in vals:
        a = abs(float(v))
        if a >= 6.0:
            k = 7
        else:
            dist = np.abs(mags - a)
            cand = np.flatnonzero(dist == dist.min())
            k = int(cand[0]) if len(cand) == 1 else int(cand[cand % 2 == 0][0])
        want = k | (8 if np.signbit(v) else 0)
        assert oracle.f32_to_e2m1(float(v)) == want, v
