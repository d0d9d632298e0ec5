"""The seeded input generator: determinism, moments, table validity."""
import numpy as np

import synth


def test_deterministic_and_distinct_streams():
    a = synth.normal_bf16(3, synth.TAG_WG, 5, 1000, 0.02)
    b = synth.normal_bf16(3, synth.TAG_WG, 5, 1000, 0.02)
    c = synth.normal_bf16(3, synth.TAG_WG, 6, 1000, 0.02)
    d = synth.normal_bf16(3, synth.TAG_WU, 5, 1000, 0.02)
    assert np.array_equal(a, b) and not np.array_equal(a, c) and not np.array_equal(a, d)


def test_normal_moments():
    v = synth.normal_f32(1, synth.TAG_X, 0, 1 << 20, 1.0).astype(np.float64)
    assert abs(v.mean()) < 5e-3 and abs(v.std() - 1.0) < 5e-3
    w = synth.bf16_to_f32(synth.normal_bf16(1, synth.TAG_WG, 0, 1 << 20, 0.02))
    assert abs(w.std() - 0.02) < 2e-4
    # an Irwin-Hall sum of four uniforms has excess kurtosis -0.3
    kurt = ((v - v.mean()) ** 4).mean() / v.var() ** 2 - 3
    assert abs(kurt + 0.3) < 0.02


def test_slices_match_whole():
    whole = synth.normal_bf16(9, synth.TAG_X, 0, 5000, 1.0)
    k = synth.key(9, synth.TAG_X, 0)
    part = np.empty(100, np.uint16)
    synth._L().synth_normal_bf16(k, 1234, 100, float(synth.normal_scale(1.0)), part.ctypes.data)
    assert np.array_equal(part, whole[1234:1334])


def test_uniform_ids_and_rows():
    ids = synth.uniform_i32(3, synth.TAG_IDS, 0, 100000, 163840)
    assert ids.min() >= 0 and ids.max() < 163840 and abs(ids.mean() / 163840 - 0.5) < 0.01
    rows = synth.distinct_rows(3, synth.TAG_TID, 20000, 384, 8)
    assert rows.min() >= 0 and rows.max() < 384
    assert all(len(set(r)) == 8 for r in rows)
    counts = np.bincount(rows.ravel(), minlength=384)
    assert counts.min() > 0.8 * counts.mean()


def test_torch_restatement_matches_c_generator():
    import torch
    n = 3 * 4096 + 17
    d = synth.normal_bf16_device(5, synth.TAG_WU, 9, n, 0.02, "cpu")
    h = synth.normal_bf16(5, synth.TAG_WU, 9, n, 0.02)
    assert np.array_equal(d.view(torch.int16).numpy().view(np.uint16), h)
