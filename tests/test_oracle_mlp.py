"""Pins for the oracle's expert MLP and combine (Stage 4: grouped gate/up ->
SwiGLU -> grouped down; AllGather combine restores token order and applies
the probabilities; shared experts added to the routed output).

The expert MLP is pinned by a dense brute force written with library
matmuls (every expert on every token, then masked by the routing weights),
by the E=1 case reducing to a plain SwiGLU MLP, by k=E softmax reducing to a
dense softmax-weighted mixture, and by replicated placements giving the same
output as the identity placement.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _bf16_bits(a64):
    """fp64 -> fp32 -> bf16 (round to nearest even) via torch, as raw bits."""
    t = torch.from_numpy(np.asarray(a64, dtype=np.float64).astype(np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return synth.bf16_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def _ffn_dense(x_bits, wg, wu, wd):
    """SwiGLU expert by library matmuls: act = bf16(silu(g) u), y = fp32(act Wd^T)."""
    x = _f(x_bits)
    g = (x @ _f(wg).T).astype(np.float32).astype(np.float64)
    u = (x @ _f(wu).T).astype(np.float32).astype(np.float64)
    act = _bf16_bits(g / (1 + np.exp(-g)) * u)
    y = (_f(act) @ _f(wd).T).astype(np.float32)
    return act, y


def _close_f32(a, b, ulps=2):
    """fp32 arrays equal to within a couple of ulps (double sums in other orders)."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    sp = np.spacing(np.abs(b).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(a - b) <= ulps * sp + 1e-30)


def _close_bf16(a_bits, b_bits, max_ulps=1, frac=0.999):
    """bf16 arrays equal except for at most one-ulp flips on a tiny fraction
    (the two sides sum the same exact products in different double orders)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    d = np.abs(a - b)
    assert d.max() <= max_ulps
    assert np.mean(d == 0) >= frac


def test_expert_rows_match_library_matmul(rng):
    cfg = synth.MINI["mini_decode"]
    d = synth.make_inputs(cfg)
    wg, wu, wd = synth.expert_weights_host(cfg, 5)
    act, y = oracle.expert_ffn_rows(d["x"][:40], wg, wu, wd, nthreads=4)
    act_r, y_r = _ffn_dense(d["x"][:40], wg, wu, wd)
    _close_bf16(act, act_r)
    _close_f32(y, y_r)


@pytest.mark.parametrize("name", ["tiny", "mini_decode", "mini_hash", "mini_skew"])
def test_routed_output_matches_dense_brute_force(name):
    cfg = synth.MINI[name]
    d = synth.make_inputs(cfg)
    W = synth.all_expert_weights_host(cfg)
    o = oracle.run_config(cfg, inputs=d, weights=W, nthreads=4)
    T, H = cfg.T, cfg.H
    # every physical expert on every token, then masked by the routing weights
    dense = np.zeros((T, H))
    mask = np.zeros((T, cfg.P))
    for t in range(T):
        for j in range(cfg.k):
            mask[t, o["ids_phys"][t, j]] += o["weights"][t, j]
    for p in range(cfg.P):
        _, y = _ffn_dense(d["x"], W[0][p], W[1][p], W[2][p])
        dense += mask[:, p:p + 1] * y.astype(np.float64)
    sw = synth.shared_weights_host(cfg)
    if sw is not None:
        dense += _ffn_dense(d["x"], *sw)[1].astype(np.float64)
    _close_bf16(o["out"], _bf16_bits(dense), frac=0.995)
    # stage outputs are consistent with the permutation
    assert np.array_equal(o["counts"], np.bincount(o["ids_phys"].ravel(),
                                                   minlength=cfg.P).astype(np.int32))


def test_single_expert_is_plain_swiglu_mlp(rng):
    H, I, T = 128, 64, 9
    x = _bf16_bits(rng.standard_normal((T, H)))
    wg, wu = (_bf16_bits(rng.standard_normal((I, H)) * 0.1) for _ in range(2))
    wd = _bf16_bits(rng.standard_normal((H, I)) * 0.1)
    cfg = oracle.route_cfg(1, 1, "softmax", routed_scaling=1.0)
    o = oracle.moe_forward(cfg, x, H, I, logits=rng.standard_normal((T, 1)).astype(np.float32),
                           wg=wg[None], wu=wu[None], wd=wd[None], nthreads=2)
    assert np.all(o["weights"] == 1.0)
    _, y = _ffn_dense(x, wg, wu, wd)
    _close_bf16(o["out"], _bf16_bits(y))


def test_all_experts_softmax_is_dense_softmax_mixture(rng):
    E, H, I, T = 6, 64, 32, 11
    x = _bf16_bits(rng.standard_normal((T, H)))
    wg = _bf16_bits(rng.standard_normal((E, I, H)) * 0.1)
    wu = _bf16_bits(rng.standard_normal((E, I, H)) * 0.1)
    wd = _bf16_bits(rng.standard_normal((E, H, I)) * 0.1)
    l = rng.standard_normal((T, E)).astype(np.float32)
    o = oracle.moe_forward(oracle.route_cfg(E, E, "softmax"), x, H, I, logits=l,
                           wg=wg, wu=wu, wd=wd, nthreads=2)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    dense = sum(p[:, e:e + 1] * _ffn_dense(x, wg[e], wu[e], wd[e])[1] for e in range(E))
    _close_bf16(o["out"], _bf16_bits(dense), frac=0.99)


def test_replicated_placement_equals_identity_placement():
    cfg = synth.MINI["mini_skew"]
    d = synth.make_inputs(cfg)
    o_rep = oracle.run_config(cfg, inputs=d, nthreads=4)
    # the same layer with one slot per logical expert
    ident = synth.MoEConfig(**{**cfg.__dict__, "n_hot_replicas": 0, "name": "ident"})
    d_id = dict(d)
    d_id["placement"] = synth.placement(ident)
    W = [np.stack([synth.expert_weights_host(cfg, e)[i] for e in range(cfg.E)]) for i in range(3)]
    o_id = oracle.run_config(ident, inputs=d_id, weights=W, nthreads=4)
    assert np.array_equal(o_rep["ids_log"], o_id["ids_log"])
    assert np.array_equal(o_rep["weights"], o_id["weights"])
    assert np.array_equal(o_rep["out"], o_id["out"])
    assert not np.array_equal(o_rep["ids_phys"], o_id["ids_phys"])
    # per-logical counts equal the sum over that expert's replicas
    pl = d["placement"]
    per_log = np.zeros(cfg.E, np.int64)
    np.add.at(per_log, pl.phys_to_log, o_rep["counts"])
    assert np.array_equal(per_log, o_id["counts"])


def test_combine_restores_token_order(rng):
    T, k, H = 7, 3, 16
    N = T * k
    y = rng.standard_normal((N, H)).astype(np.float32)
    f2r = rng.permutation(N).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    ys = rng.standard_normal((T, H)).astype(np.float32)
    out = oracle.combine(y, f2r, w, ys)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            ref[t] += float(w[t, j]) * y[f2r[t * k + j]].astype(np.float64)
    ref += ys
    _close_bf16(out, _bf16_bits(ref), frac=1.0)
