"""Property-based pins of the oracle (hypothesis): randomized shapes, groupings,
scorings, ties, empty experts and replica maps, each example checked against
an independent brute force or an invariant.

- selection: grouped top-k of the vLLM-Ascend "Kimi K3 MoE Forward Insight"
  page, section "Stage 2: Select Experts" (with the readings R3-R6) against a
  lexicographic sort in numpy; weights against the renormalisation identity;
- logical-to-physical mapping ("Stage 4", step 2; reading R8) against the
  table lookup, logical ids independent of the placement;
- permutation ("Stage 4" AllGather row; reading R9): bincount, bijection,
  stability, permute-then-unpermute identity, on any T including 0;
- the routed layer against every expert run on every token and masked by
  the routing weights.

The GPU machine has no hypothesis; these run with the CPU suite.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from tests.test_oracle_mlp import _bf16_bits, _close_bf16, _ffn_dense  # noqa: E402
from tests.test_oracle_permute import _check  # noqa: E402
from tests.test_oracle_route import _brute_select  # noqa: E402

U = 2.0 ** -24
SETTINGS = settings(max_examples=60, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.too_slow, HealthCheck.data_too_large])


@st.composite
def routing_case(draw):
    G = draw(st.integers(1, 8))
    gs = draw(st.integers(1, 8))
    E = G * gs
    kg = draw(st.integers(1, G))
    k = draw(st.integers(1, min(kg * gs, 16)))
    return {
        "E": E, "G": G, "kg": kg, "k": k,
        "mode": draw(st.sampled_from(["max", "top2sum"])),
        "scoring": draw(st.sampled_from(["softmax", "sigmoid", "sqrtsoftplus"])),
        "bias": draw(st.booleans()),
        "grid": draw(st.sampled_from([0, 1, 4])),       # 0: continuous logits; else ties
        "renorm": draw(st.booleans()),
        "scale": draw(st.sampled_from([1.0, 2.5, 0.75])),
        "T": draw(st.integers(1, 40)),
        "seed": draw(st.integers(0, 2 ** 31 - 1)),
    }


@SETTINGS
@given(routing_case())
def test_selection_and_weights_on_random_configurations(c):
    rng = np.random.default_rng(c["seed"])
    E, T = c["E"], c["T"]
    l = (rng.standard_normal((T, E)) * 3).astype(np.float32)
    cb = (rng.standard_normal(E) * 0.5).astype(np.float32) if c["bias"] else None
    if c["grid"]:  # logits and bias on a coarse grid: many exact ties
        l = (np.round(l * c["grid"]) / c["grid"]).astype(np.float32)
        if cb is not None:
            cb = (np.round(cb * 8) / 8).astype(np.float32)
    cfg = oracle.route_cfg(E, c["k"], c["scoring"], n_group=c["G"], topk_group=c["kg"],
                           group_score=c["mode"], renormalize=c["renorm"],
                           routed_scaling=c["scale"])
    ids, ids_p, w = oracle.route(cfg, l, corr_bias=cb)
    assert np.array_equal(ids, ids_p)
    for t in range(T):
        s = oracle.scores(l[t], c["scoring"])
        sel = (s + cb).astype(np.float32) if cb is not None else s
        assert list(ids[t]) == list(_brute_select(sel, E, c["k"], c["G"], c["kg"], c["mode"]))
        assert len(set(ids[t].tolist())) == c["k"]
        chosen = s.astype(np.float64)[ids[t]]
        if c["renorm"]:
            assert abs(w[t].astype(np.float64).sum() - c["scale"]) <= 4 * c["k"] * U * c["scale"]
            np.testing.assert_allclose(w[t], chosen / chosen.sum() * c["scale"], rtol=4e-7)
        else:
            assert np.array_equal(w[t], (s[ids[t]] * np.float32(c["scale"])).astype(np.float32))


@st.composite
def placement_case(draw):
    E = draw(st.integers(2, 24))
    k = draw(st.integers(1, min(E, 8)))
    R = draw(st.integers(1, 3))
    cnt = draw(st.lists(st.integers(1, R), min_size=E, max_size=E))
    return {"E": E, "k": k, "R": R, "cnt": cnt, "T": draw(st.integers(1, 50)),
            "seed": draw(st.integers(0, 2 ** 31 - 1))}


@SETTINGS
@given(placement_case())
def test_replica_choice_on_random_placements(c):
    rng = np.random.default_rng(c["seed"])
    E, k, R, T = c["E"], c["k"], c["R"], c["T"]
    cnt = np.array(c["cnt"], np.int32)
    P = int(cnt.sum())
    slots = rng.permutation(P).astype(np.int32)
    l2p = np.full((E, R), 0, np.int32)
    nxt = 0
    for e in range(E):
        for r in range(cnt[e]):
            l2p[e, r] = slots[nxt]
            nxt += 1
    l = rng.standard_normal((T, E)).astype(np.float32)
    ids, ids_p, w = oracle.route(oracle.route_cfg(E, k, "sigmoid", P=P), l, log2phy=l2p,
                                 replica_cnt=cnt)
    ids0, _, w0 = oracle.route(oracle.route_cfg(E, k, "sigmoid"), l)
    assert np.array_equal(ids, ids0) and np.array_equal(w, w0)
    for t in range(T):
        for j in range(k):
            assert ids_p[t, j] == l2p[ids[t, j], t % cnt[ids[t, j]]]
    # every physical slot's count is its share of its logical expert's picks
    counts = oracle.permute(ids_p, P)[0]
    per_log = np.zeros(E, np.int64)
    for e in range(E):
        per_log[e] = sum(int(counts[l2p[e, r]]) for r in range(cnt[e]))
    assert np.array_equal(per_log, np.bincount(ids.ravel(), minlength=E))


@SETTINGS
@given(st.integers(0, 300), st.integers(1, 8), st.integers(1, 64), st.integers(0, 3),
       st.integers(0, 2 ** 31 - 1))
def test_permutation_on_random_ids(T, k, P, skew, seed):
    rng = np.random.default_rng(seed)
    # skew > 0 piles the picks onto the first experts (others stay empty)
    w = 1.0 / np.arange(1, P + 1) ** skew
    ids = rng.choice(P, size=(T, k), p=w / w.sum()).astype(np.int32)
    counts, offsets, r2t, f2r = _check(ids, P)
    assert counts.sum() == T * k


@st.composite
def layer_case(draw):
    E = draw(st.integers(1, 5))
    return {"E": E, "k": draw(st.integers(1, E)), "H": 8 * draw(st.integers(2, 8)),
            "I": 8 * draw(st.integers(1, 6)), "T": draw(st.integers(1, 12)),
            "scoring": draw(st.sampled_from(["softmax", "sigmoid"])),
            "seed": draw(st.integers(0, 2 ** 31 - 1))}


@settings(max_examples=25, deadline=None, derandomize=True,
          suppress_health_check=[HealthCheck.too_slow])
@given(layer_case())
def test_routed_layer_equals_masked_dense_experts(c):
    rng = np.random.default_rng(c["seed"])
    E, k, H, I, T = c["E"], c["k"], c["H"], c["I"], c["T"]
    x = _bf16_bits(rng.standard_normal((T, H)))
    wg = _bf16_bits(rng.standard_normal((E, I, H)) * 0.1)
    wu = _bf16_bits(rng.standard_normal((E, I, H)) * 0.1)
    wd = _bf16_bits(rng.standard_normal((E, H, I)) * 0.1)
    l = rng.standard_normal((T, E)).astype(np.float32)
    o = oracle.moe_forward(oracle.route_cfg(E, k, c["scoring"], routed_scaling=1.5), x, H, I,
                           logits=l, wg=wg, wu=wu, wd=wd, nthreads=2)
    mask = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            mask[t, o["ids_log"][t, j]] += o["weights"][t, j]
    dense = sum(mask[:, e:e + 1] * _ffn_dense(x, wg[e], wu[e], wd[e])[1].astype(np.float64)
                for e in range(E))
    _close_bf16(o["out"], _bf16_bits(dense), frac=0.98)
