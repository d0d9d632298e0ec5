"""Pins for the oracle's FP8 (OCP E4M3) quantization and FP8 expert MLP
(Stage 4 quantized paths, W8A8FP; reading R17).

The E4M3 encoder is pinned by the format itself: every finite code decodes
and re-encodes to itself, decoded codes are strictly increasing, textbook
values (1.0, 448, the smallest subnormal, ties between subnormals), saturation,
and agreement with a brute-force nearest-value search (ties to the even code)
over all finite codes.  Row quantization maps the row's largest magnitude to
+-448 exactly.  The FP8 MLP is checked against dequantized library matmuls.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.test_oracle_mlp import _bf16_bits, _f


def _codes_finite():
    return [c for c in range(256) if (c & 0x7f) != 0x7f]


def test_e4m3_round_trip_and_order():
    vals = {c: oracle.e4m3_to_f32(c) for c in _codes_finite()}
    for c, v in vals.items():
        assert oracle.f32_to_e4m3(v) == c
    pos = [vals[c] for c in range(0, 0x7f)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    assert oracle.e4m3_to_f32(0x7e) == 448.0


def test_e4m3_textbook_values():
    f = oracle.f32_to_e4m3
    assert f(1.0) == 0x38 and f(-1.0) == 0xb8
    assert f(448.0) == 0x7e and f(1e6) == 0x7e and f(-1e6) == 0xfe and f(464.0) == 0x7e
    assert f(2.0 ** -9) == 0x01          # smallest subnormal
    assert f(2.0 ** -10) == 0x00         # tie between 0 and 2^-9: the even code
    assert f(3 * 2.0 ** -10) == 0x02     # tie between codes 1 and 2: the even one
    assert f(1.0625) == 0x38             # tie between 1 and 1.125: even mantissa
    assert f(1.1875) == 0x3a             # tie between 1.125 and 1.25: even mantissa (1.25)
    assert f(0.0) == 0x00 and f(-0.0) == 0x80


def test_e4m3_matches_brute_force_nearest(rng):
    codes = list(range(0, 0x7f))
    grid = np.array([oracle.e4m3_to_f32(c) for c in codes])
    xs = np.concatenate([rng.uniform(0, 460, 3000), np.exp(rng.uniform(-12, 6, 3000))])
    for x in xs.astype(np.float32):
        x = float(x)
        d = np.abs(grid - x)
        best = np.flatnonzero(d == d.min())
        want = codes[best[0]] if len(best) == 1 else [codes[b] for b in best if codes[b] % 2 == 0][0]
        if x >= 448.0:
            want = 0x7e
        assert oracle.f32_to_e4m3(x) == want, x


def test_quantize_rows_scale_and_extremes(rng):
    x = _bf16_bits(rng.standard_normal((6, 96)) * 3)
    x[5] = 0
    q, s = oracle.quantize_rows(x)
    for r in range(5):
        a = np.abs(_f(x[r]))
        assert s[r] == np.float32(a.max()) / np.float32(448.0)
        i = int(np.argmax(a))
        assert (q[r, i] & 0x7f) == 0x7e
        deq = np.array([oracle.e4m3_to_f32(c) for c in q[r]]) * s[r]
        assert np.all(np.abs(deq - _f(x[r])) <= a.max() / 448 * 2 ** -3 * np.maximum(1, np.abs(_f(x[r])) / (a.max() / 448)) + 1e-30)
    assert s[5] == 1.0 and np.all(q[5] == 0)


def test_fp8_grouped_mlp_matches_dequantized_matmuls(rng):
    H, I, T = 128, 64, 10
    x = _bf16_bits(rng.standard_normal((T, H)))
    rows = [4, 0, 6]
    P = len(rows)
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    r2t = rng.permutation(T).astype(np.int32)
    W = [[_bf16_bits(rng.standard_normal(sh) * 0.1) for sh in ((I, H), (I, H), (H, I))]
         for _ in range(P)]
    xq, sx = oracle.quantize_rows(x)
    qs = [[oracle.quantize_rows(w) for w in ws] for ws in W]
    wg = np.stack([q[0][0] for q in qs]); sg = np.stack([q[0][1] for q in qs])
    wu = np.stack([q[1][0] for q in qs]); su = np.stack([q[1][1] for q in qs])
    wd = np.stack([q[2][0] for q in qs]); sd = np.stack([q[2][1] for q in qs])
    act, y = oracle.ffn_grouped_fp8(xq, sx, r2t, offs, wg, sg, wu, su, wd, sd, nthreads=2)
    dq = np.vectorize(oracle.e4m3_to_f32)
    for p in range(P):
        for r in range(offs[p], offs[p + 1]):
            t = r2t[r]
            xd = dq(xq[t]).astype(np.float64) * sx[t]
            g = (xd @ (dq(wg[p]).T * sg[p])).astype(np.float32)
            u = (xd @ (dq(wu[p]).T * su[p])).astype(np.float32)
            a_ref = _bf16_bits(g / (1 + np.exp(-g.astype(np.float64))) * u)
            assert np.abs(act[r].astype(np.int32) - a_ref.astype(np.int32)).max() <= 1
            aq, sa = oracle.quantize_rows(act[r][None])
            yr = (dq(aq[0]).astype(np.float64) * sa[0]) @ (dq(wd[p]).T * sd[p])
            assert np.allclose(y[r], yr, rtol=1e-5, atol=1e-6 * np.abs(yr).max())
