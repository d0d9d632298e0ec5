"""Pins for the oracle's routing (Runner Initialization settings; Stage 2
Select Experts; Stage 4 step 2 log2phy mapping).

Router logits are pinned by exact integer arithmetic and by the fp32 error
bound of the pinned summation; selection by a brute-force lexicographic sort
(numpy) including deliberate ties; weights by the renormalisation invariants
and by the closed forms of each scoring function.
"""
import math

import numpy as np
import pytest

import oracle
import synth

U = 2.0 ** -24


def _bf16(a):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_logits_exact_on_integer_inputs(rng):
    # small integers: every product and partial sum is exact in fp32, so the
    # logits must equal the integer dot product whatever the summation order
    T, E, H = 5, 7, 100
    xi = rng.integers(-8, 9, size=(T, H))
    wi = rng.integers(-8, 9, size=(E, H))
    lg = oracle.router_logits(_bf16(xi), wi.astype(np.float32))
    assert np.array_equal(lg.astype(np.int64), xi @ wi.T)
    assert lg.shape == (T, E)


def test_logits_within_pinned_order_error_bound(rng):
    T, E, H = 4, 6, 7168
    x = _bf16(rng.standard_normal((T, H)))
    w = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    lg = oracle.router_logits(x, w)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    for t in range(T):
        for e in range(E):
            terms = xf[t] * w[e].astype(np.float64)
            exact = math.fsum(terms)
            bound = (H / 32 + 5 + 1) * U * np.abs(terms).sum()
            assert abs(float(lg[t, e]) - exact) <= bound


def test_router_bias_added_last(rng):
    x = _bf16(rng.standard_normal((3, 64)))
    w = rng.standard_normal((5, 64)).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    l0 = oracle.router_logits(x, w)
    l1 = oracle.router_logits(x, w, router_bias=b)
    assert np.array_equal(l1, (l0 + b).astype(np.float32))


def test_softmax_scores(rng):
    l = (rng.standard_normal(37) * 3).astype(np.float32)
    s = oracle.scores(l, "softmax").astype(np.float64)
    ref = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
    assert abs(s.sum() - 1.0) < 37 * 4 * U
    assert np.max(np.abs(s - ref) / ref) < 8 * U
    eq = oracle.scores(np.zeros(16, np.float32), "softmax")
    assert np.all(eq == np.float32(1 / 16))


def test_sigmoid_and_sqrtsoftplus_scores(rng):
    l = (rng.standard_normal(50) * 4).astype(np.float32)
    s = oracle.scores(l, "sigmoid").astype(np.float64)
    assert np.max(np.abs(s - 1 / (1 + np.exp(-l.astype(np.float64))))) < 4e-7
    q = oracle.scores(l, "sqrtsoftplus").astype(np.float64)
    ref = np.sqrt(np.log1p(np.exp(l.astype(np.float64))))
    assert np.max(np.abs(q - ref) / ref) < 4e-7


def _brute_select(sel, E, k, G, kg, mode):
    """Grouped top-k by lexicographic sorting (numpy), ties to lower index."""
    if G > 1:
        gs = E // G
        gsc = []
        for g in range(G):
            v = np.sort(sel[g * gs:(g + 1) * gs])[::-1]
            gsc.append(np.float32(v[0] + v[1]) if (mode == "top2sum" and gs > 1) else v[0])
        gsc = np.array(gsc, dtype=np.float32)
        keep = np.lexsort((np.arange(G), -gsc.astype(np.float64)))[:kg]
        allowed = np.zeros(E, bool)
        for g in keep:
            allowed[g * gs:(g + 1) * gs] = True
    else:
        allowed = np.ones(E, bool)
    cand = np.nonzero(allowed)[0]
    order = np.lexsort((cand, -sel[cand].astype(np.float64)))
    return cand[order[:k]]


CASES = [  # (E, k, n_group, topk_group, group_score, scoring, bias)
    (8, 2, 1, 1, "max", "softmax", False),
    (16, 4, 4, 2, "top2sum", "sigmoid", True),
    (16, 4, 4, 2, "max", "sigmoid", False),
    (32, 8, 8, 4, "top2sum", "sigmoid", True),
    (12, 3, 3, 1, "max", "sqrtsoftplus", False),
    (10, 10, 1, 1, "max", "softmax", False),
    (24, 5, 6, 3, "top2sum", "softmax", True),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("quantised", [False, True])
def test_selection_matches_brute_force(case, quantised, rng):
    E, k, G, kg, mode, scoring, bias = case
    T = 64
    l = rng.standard_normal((T, E)).astype(np.float32)
    cb = (rng.standard_normal(E) * 0.1).astype(np.float32) if bias else None
    if quantised:  # force many exact ties
        l = np.round(l * 2) / 2
        if cb is not None:
            cb = np.round(cb * 8) / 8
    cfg = oracle.route_cfg(E, k, scoring, n_group=G, topk_group=kg, group_score=mode,
                           routed_scaling=1.0)
    ids, ids_p, w = oracle.route(cfg, l, corr_bias=cb)
    assert np.array_equal(ids, ids_p)  # identity placement
    for t in range(T):
        s = oracle.scores(l[t], scoring)
        sel = (s + cb).astype(np.float32) if cb is not None else s
        assert list(ids[t]) == list(_brute_select(sel, E, k, G, kg, mode))


def test_flat_topk_special_cases(rng):
    E, k, T = 32, 8, 50
    l = rng.standard_normal((T, E)).astype(np.float32)
    cb = (rng.standard_normal(E) * 0.1).astype(np.float32)
    flat = oracle.route(oracle.route_cfg(E, k, "sigmoid"), l, corr_bias=cb)[0]
    all_groups = oracle.route(oracle.route_cfg(E, k, "sigmoid", n_group=8, topk_group=8,
                                               group_score="top2sum"), l, corr_bias=cb)[0]
    assert np.array_equal(flat, all_groups)
    # k = E: every expert, in descending selection order
    ids = oracle.route(oracle.route_cfg(E, E, "softmax"), l)[0]
    for t in range(T):
        assert list(ids[t]) == list(np.lexsort((np.arange(E), -l[t].astype(np.float64))))


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid", "sqrtsoftplus"])
def test_weights_renormalised_and_scaled_from_unbiased_scores(scoring, rng):
    E, k, T, scale = 16, 4, 40, 2.5
    l = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    cb = (rng.standard_normal(E) * 5.0).astype(np.float32)  # large: changes the picks
    cfg = oracle.route_cfg(E, k, scoring, routed_scaling=scale)
    ids, _, w = oracle.route(cfg, l, corr_bias=cb)
    for t in range(T):
        s = oracle.scores(l[t], scoring).astype(np.float64)[ids[t]]
        assert abs(w[t].astype(np.float64).sum() - scale) <= 4 * k * U * scale
        np.testing.assert_allclose(w[t], s / s.sum() * scale, rtol=4e-7)
    cfg0 = oracle.route_cfg(E, k, scoring, renormalize=False, routed_scaling=scale)
    ids0, _, w0 = oracle.route(cfg0, l, corr_bias=cb)
    assert np.array_equal(ids0, ids)
    for t in range(T):
        s = oracle.scores(l[t], scoring)[ids[t]]
        assert np.array_equal(w0[t], (s * np.float32(scale)).astype(np.float32))


def test_softmax_renorm_equals_softmax_over_chosen(rng):
    E, k, T = 24, 6, 30
    l = rng.standard_normal((T, E)).astype(np.float32)
    ids, _, w = oracle.route(oracle.route_cfg(E, k, "softmax"), l)
    for t in range(T):
        c = l[t, ids[t]].astype(np.float64)
        ref = np.exp(c - c.max()) / np.exp(c - c.max()).sum()
        np.testing.assert_allclose(w[t], ref, rtol=2e-6)


def test_hash_routing(rng):
    E, k, T, V = 48, 8, 60, 500
    tbl = synth.distinct_rows(7, synth.TAG_TID, V, E, k)
    assert all(len(set(r)) == k for r in tbl) and tbl.min() >= 0 and tbl.max() < E
    ids_in = rng.integers(0, V, T).astype(np.int32)
    l = rng.standard_normal((T, E)).astype(np.float32)
    cfg = oracle.route_cfg(E, k, "sqrtsoftplus", routed_scaling=2.5, use_hash=True)
    ids, ids_p, w = oracle.route(cfg, l, input_ids=ids_in, tid2eid=tbl)
    assert np.array_equal(ids, tbl[ids_in]) and np.array_equal(ids_p, ids)
    for t in range(T):
        s = np.sqrt(np.log1p(np.exp(l[t, ids[t]].astype(np.float64))))
        np.testing.assert_allclose(w[t], s / s.sum() * 2.5, rtol=1e-6)
    bad = ids_in.copy()
    bad[3] = V
    with pytest.raises(ValueError):
        oracle.route(cfg, l, input_ids=bad, tid2eid=tbl)
    tbl2 = tbl.copy()
    tbl2[ids_in[0], 2] = E
    with pytest.raises(ValueError):
        oracle.route(cfg, l, input_ids=ids_in, tid2eid=tbl2)


def test_log2phy_replica_by_token_position(rng):
    E, k, T = 16, 4, 33
    P = 21
    l2p = np.zeros((E, 3), np.int32)
    cnt = np.ones(E, np.int32)
    slots = rng.permutation(P).astype(np.int32)
    nxt = 0
    for e in range(E):
        l2p[e, 0] = slots[nxt]; nxt += 1
    for e in (1, 5, 9):          # 2 replicas
        cnt[e] = 2; l2p[e, 1] = slots[nxt]; nxt += 1
    cnt[12] = 3                  # 3 replicas
    l2p[12, 1] = slots[nxt]; l2p[12, 2] = slots[nxt + 1]
    l = rng.standard_normal((T, E)).astype(np.float32)
    cfg = oracle.route_cfg(E, k, "sigmoid", P=P)
    ids, ids_p, _ = oracle.route(cfg, l, log2phy=l2p, replica_cnt=cnt)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            assert ids_p[t, j] == l2p[e, t % cnt[e]]
    # logical ids do not depend on the placement
    assert np.array_equal(ids, oracle.route(oracle.route_cfg(E, k, "sigmoid"), l)[0])
    bad = l2p.copy()
    bad[3, 0] = P
    with pytest.raises(ValueError):
        oracle.route(cfg, l, log2phy=bad, replica_cnt=cnt)


def test_skew_placement_table_is_valid():
    for cfg in (synth.CONFIGS["skew"], synth.MINI["mini_skew"]):
        pl = synth.placement(cfg)
        used = []
        for e in range(cfg.E):
            used += [int(pl.log2phy[e, r]) for r in range(pl.replica_cnt[e])]
            assert all(pl.phys_to_log[pl.log2phy[e, r]] == e for r in range(pl.replica_cnt[e]))
        assert sorted(used) == list(range(cfg.P))
        b = synth.zipf_router_bias(cfg)
        hot = np.nonzero(pl.replica_cnt == 2)[0]
        assert len(hot) == cfg.n_hot_replicas
        assert b[hot].min() > np.delete(b, hot).max()   # the hottest get the replicas
