"""GPU parity: every stage and the whole layer, through the C ABI, against the
CPU oracle on the same seeded inputs, element by element.

Bars: expert ids, permutation indices and counts bit-exact; routing weights
and logits bit-exact (both sides follow the same pinned fp32 definitions);
activations and outputs within |gpu - oracle| <= 1e-2 + 1e-2 |oracle| per
element, plus a tighter diagnostic (max error <= 2 bf16 ulps of the output
scale) because the small workloads' outputs are ~1e-2 in magnitude.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import bf16_dev, device_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SMALL = list(synth.MINI)


def _gb():
    import routed_mixture_experts_gemm_gb300 as gb
    return gb


def _np(t):
    return t.cpu().numpy()


def _bf(t):
    return _np(t.float())


def assert_within_tol(got, exp, what):
    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    err = np.abs(got - exp)
    bad = err > 1e-2 + 1e-2 * np.abs(exp)
    assert not bad.any(), f"{what}: {bad.sum()} elements outside tolerance, max err {err.max()}"
    scale = max(np.abs(exp).max(), 1e-30)
    assert err.max() <= 2 * 2.0 ** -8 * scale, f"{what}: max err {err.max()} vs scale {scale}"


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()
    return _gb()


_cache = {}


def case_and_ref(name):
    if name not in _cache:
        cfg = synth.MINI[name]
        case = device_case(cfg, DEV, host_weights=True)
        ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
        _cache[name] = (case, ref)
    return _cache[name]


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid", "sqrtsoftplus"])
def test_scoring_functions_bit_exact(built, scoring):
    gb = built
    # k = E, no renormalisation: the weights are the scores, sorted descending
    E, T = 64, 96
    rng = np.random.default_rng(5)
    l = np.concatenate([rng.standard_normal((T - 4, E)) * 6,
                        np.linspace(-95, 95, 4 * E).reshape(4, E)]).astype(np.float32)
    cfg = gb.route_cfg(E, 32, scoring, renormalize=False, routed_scaling=1.0)
    o = gb.moe_route(cfg, logits=torch.from_numpy(l).to(DEV))
    ocfg = oracle.route_cfg(E, 32, scoring, renormalize=False, routed_scaling=1.0)
    ids, _, w = oracle.route(ocfg, l)
    assert np.array_equal(_np(o["ids_log"]), ids)
    assert np.array_equal(_np(o["weights"]).view(np.uint32), w.view(np.uint32))


# router-logit paths: TMA tiles of 32 tokens x 32 experts (many tokens), of
# 16 x 16 (few tokens, ragged token and expert tails), each with 256- and
# 128-wide chunks (H % 256 == 0 or not), and the generic kernel for H not a
# multiple of 128
LOGIT_SHAPES = [(1024, 320, 256), (1024, 320, 384), (37, 40, 384), (1, 256, 7168),
                (128, 256, 1024), (9, 8, 200), (300, 64, 96)]


@pytest.mark.parametrize("shape", LOGIT_SHAPES)
def test_router_logit_paths_bit_exact(built, shape):
    gb = built
    T, E, H = shape
    rng = np.random.default_rng(T * 7 + E + H)
    from tests.test_oracle_mlp import _bf16_bits
    x = _bf16_bits(rng.standard_normal((T, H)))
    w = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    b = rng.standard_normal(E).astype(np.float32)
    cfg = gb.route_cfg(E, min(4, E), "sigmoid")
    o = gb.moe_route(cfg, x=bf16_dev(x, DEV), w_router=torch.from_numpy(w).to(DEV),
                     router_bias=torch.from_numpy(b).to(DEV))
    assert gb.check_device_status() == 0
    ref = oracle.router_logits(x, w, router_bias=b, nthreads=8)
    assert np.array_equal(_np(o["logits"]).view(np.uint32), ref.view(np.uint32))


# grouped top-k: lane-aligned groups (E=256/8, 384/8, 96/6) and the general
# group loop (E=60/5, 40/4, 200/8); logits on a coarse grid so that scores,
# group scores and selections tie often
SELECT_CASES = [(256, 8, 4, 8, "top2sum"), (384, 8, 4, 8, "max"), (96, 6, 3, 6, "top2sum"),
                (60, 5, 2, 7, "top2sum"), (40, 4, 2, 5, "max"), (200, 8, 3, 8, "top2sum")]


@pytest.mark.parametrize("case", SELECT_CASES)
@pytest.mark.parametrize("scoring", ["sigmoid", "softmax"])
def test_grouped_selection_paths_bit_exact(built, case, scoring):
    gb = built
    E, G, kg, k, mode = case
    T = 257
    rng = np.random.default_rng(E + G + k)
    l = (np.round(rng.standard_normal((T, E)) * 4) / 4).astype(np.float32)
    cb = (np.round(rng.standard_normal(E) * 8) / 64).astype(np.float32)
    cfg = gb.route_cfg(E, k, scoring, n_group=G, topk_group=kg, group_score=mode,
                       routed_scaling=2.5)
    o = gb.moe_route(cfg, logits=torch.from_numpy(l).to(DEV),
                     corr_bias=torch.from_numpy(cb).to(DEV))
    assert gb.check_device_status() == 0
    ocfg = oracle.route_cfg(E, k, scoring, n_group=G, topk_group=kg, group_score=mode,
                            routed_scaling=2.5)
    ids, _, w = oracle.route(ocfg, l, corr_bias=cb)
    assert np.array_equal(_np(o["ids_log"]), ids)
    assert np.array_equal(_np(o["weights"]).view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("name", SMALL)
def test_route_bit_exact(built, name):
    gb = built
    case, ref = case_and_ref(name)
    cfg = case.cfg
    o = gb.moe_route(case.layer.cfg, x=case.x, w_router=case.dev["w_router"],
                     router_bias=case.dev["router_bias"], corr_bias=case.dev["corr_bias"],
                     input_ids=case.input_ids, tid2eid=case.dev["tid2eid"],
                     log2phy=case.dev["log2phy"], replica_cnt=case.dev["replica_cnt"])
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(o["logits"]).view(np.uint32), ref["logits"].view(np.uint32))
    assert np.array_equal(_np(o["ids_log"]), ref["ids_log"])
    assert np.array_equal(_np(o["ids_phys"]), ref["ids_phys"])
    assert np.array_equal(_np(o["weights"]).view(np.uint32), ref["weights"].view(np.uint32))
    assert np.array_equal(_np(o["counts"]), ref["counts"])
    # load tracking: counts accumulate across calls like moe_load
    load = gb.moe_expert_counts(o["ids_phys"], cfg.P)
    gb.moe_expert_counts(o["ids_phys"], cfg.P, counts=load, accumulate=True)
    assert np.array_equal(_np(load), 2 * ref["counts"])


@pytest.mark.parametrize("name", SMALL)
def test_permute_bit_exact(built, name):
    gb = built
    case, ref = case_and_ref(name)
    ids = torch.from_numpy(ref["ids_phys"]).to(DEV)
    o = gb.moe_permute(ids, case.cfg.P, x=case.x)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(o["counts"]), ref["counts"])
    assert np.array_equal(_np(o["offsets"]), ref["offsets"])
    assert np.array_equal(_np(o["row_to_token"]), ref["row_to_token"])
    assert np.array_equal(_np(o["flat_to_row"]), ref["flat_to_row"])
    xp = _np(o["x_perm"].view(torch.int16)).view(np.uint16)
    assert np.array_equal(xp, case.inputs["x"][ref["row_to_token"]])


# both permutation paths: one block for N = T*k <= 4096 (and P <= 1024), the
# histogram / column-scan / scatter kernels above; skewed ids leave experts
# empty and pile rows onto a few
PERM_SHAPES = [(1, 1, 5), (3, 8, 1024), (512, 8, 256), (513, 8, 256), (1000, 8, 300),
               (2048, 6, 1000), (4096, 8, 288)]


@pytest.mark.parametrize("shape", PERM_SHAPES)
def test_permute_paths_bit_exact(built, shape):
    gb = built
    T, k, P = shape
    rng = np.random.default_rng(T + k + P)
    # Zipf-like skew over experts, k distinct experts per token when possible
    wts = 1.0 / np.arange(1, P + 1) ** 1.1
    wts /= wts.sum()
    ids = np.stack([rng.choice(P, size=k, replace=k > P, p=wts) for _ in range(T)]).astype(np.int32)
    H = 64
    from tests.test_oracle_mlp import _bf16_bits
    x = _bf16_bits(rng.standard_normal((T, H)))
    o = gb.moe_permute(torch.from_numpy(ids).to(DEV), P, x=bf16_dev(x, DEV))
    assert gb.check_device_status() == 0
    counts, offsets, r2t, f2r = oracle.permute(ids, P)
    assert np.array_equal(_np(o["counts"]), counts)
    assert np.array_equal(_np(o["offsets"]), offsets)
    assert np.array_equal(_np(o["row_to_token"]), r2t)
    assert np.array_equal(_np(o["flat_to_row"]), f2r)
    xp = _np(o["x_perm"].view(torch.int16)).view(np.uint16)
    assert np.array_equal(xp, x[r2t])


@pytest.mark.parametrize("name", SMALL)
def test_grouped_gemms(built, name):
    gb = built
    case, ref = case_and_ref(name)
    x_perm = bf16_dev(case.inputs["x"][ref["row_to_token"]], DEV)
    offs = torch.from_numpy(ref["offsets"]).to(DEV)
    act = gb.moe_gemm_gateup_act(x_perm, offs, case.dev["w_gate"], case.dev["w_up"])
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(act), synth.bf16_to_f32(ref["act"]), "act")
    # the down GEMM on the oracle's activations isolates GEMM2
    y = gb.moe_gemm_down(bf16_dev(ref["act"], DEV), offs, case.dev["w_down"])
    assert gb.check_device_status() == 0
    assert_within_tol(_np(y), ref["y"], "y")


@pytest.mark.parametrize("name", SMALL)
def test_combine(built, name):
    gb = built
    case, ref = case_and_ref(name)
    ys = torch.from_numpy(ref["ys"]).to(DEV) if "ys" in ref else None
    out = gb.moe_combine(torch.from_numpy(ref["y"]).to(DEV),
                         torch.from_numpy(ref["flat_to_row"]).to(DEV),
                         torch.from_numpy(ref["weights"]).to(DEV), shared_y=ys)
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), "combine")


@pytest.mark.parametrize("name", SMALL)
def test_forward_end_to_end(built, name):
    gb = built
    case, ref = case_and_ref(name)
    cfg = case.cfg
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    idp = torch.empty_like(ids)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.P, dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids, ids_log=ids,
                         ids_phys=idp, weights=w, counts=cnt)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(ids), ref["ids_log"])
    assert np.array_equal(_np(idp), ref["ids_phys"])
    assert np.array_equal(_np(w).view(np.uint32), ref["weights"].view(np.uint32))
    assert np.array_equal(_np(cnt), ref["counts"])
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), "out")
    # run-to-run determinism (bitwise)
    out2 = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


# the gated activation branches: each GEMM tile variant (128- and 256-token
# gate/up tiles, contiguous and gathered operands) and the whole layer (fused
# decode-sized and two-launch prefill-sized expert MLPs, shared expert)
ACTS = ["swiglu_oai", "geglu", "geglu_tanh", "swiglu"]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("rows", [[40, 3, 17, 0, 90], [150, 200, 300, 1, 0]])
def test_gateup_activations(built, act, rows):
    gb = built
    H, I = 256, 256
    rng = np.random.default_rng(len(rows) + sum(rows))
    from tests.test_oracle_mlp import _bf16_bits
    P = len(rows)
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(offs[-1])
    x = _bf16_bits(rng.standard_normal((N, H)))
    # gate/up projections ~ N(0, 4^2): the clipped branch's caps at +-7 engage
    wg = _bf16_bits(rng.standard_normal((P, I, H)) * 0.25)
    wu = _bf16_bits(rng.standard_normal((P, I, H)) * 0.25)
    wd = _bf16_bits(rng.standard_normal((P, H, I)) * 0.05)
    act_o = np.zeros((N, I), np.uint16)
    for p in range(P):
        if rows[p]:
            a, _ = oracle.expert_ffn_rows(x[offs[p]:offs[p + 1]], wg[p], wu[p], wd[p],
                                          nthreads=4, activation=act)
            act_o[offs[p]:offs[p + 1]] = a
    d_offs = torch.from_numpy(offs).to(DEV)
    dwg, dwu = bf16_dev(wg, DEV), bf16_dev(wu, DEV)
    a1 = gb.moe_gemm_gateup_act(bf16_dev(x, DEV), d_offs, dwg, dwu, activation=act)
    # gathered: the same rows from a reversed source
    src = bf16_dev(x[::-1].copy(), DEV)
    r2t = torch.arange(N - 1, -1, -1, dtype=torch.int32, device=DEV)
    a2 = gb.moe_gemm_gateup_act_rows(src, r2t, d_offs, dwg, dwu, activation=act)
    assert gb.check_device_status() == 0
    ref = synth.bf16_to_f32(act_o)
    assert_within_tol(_bf(a1), ref, f"act {act} {rows}")
    assert_within_tol(_bf(a2), ref, f"act (gathered) {act} {rows}")


@pytest.mark.parametrize("act", ["swiglu_oai", "geglu", "geglu_tanh"])
@pytest.mark.parametrize("name", ["mini_decode", "mini_prefill", "mini_skew"])
def test_forward_activations(built, act, name):
    gb = built
    cfg = synth.MINI[name]
    case = device_case(cfg, DEV, host_weights=True, activation=act)
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host, activation=act)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids)
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), f"out {act} {name}")


def test_unknown_activation_is_rejected(built):
    gb = built
    x = torch.zeros((16, 128), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gb.GbmoeError):
        gb.moe_gemm_gateup_act(x, None, w, w, activation=7)


def test_forward_matches_golden_fixture(built):
    from tests.test_golden import load_tiny
    gb = built
    g = load_tiny()
    case = device_case(synth.CONFIGS["tiny"], DEV, host_weights=True)
    ids = torch.empty((64, 2), dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, ids_log=ids)
    assert np.array_equal(_np(ids), np.array(g["ids_log"]))
    assert_within_tol(_bf(out), synth.bf16_to_f32(g["out"]), "out vs golden")


def test_host_buffer_forward(built):
    gb = built
    case, ref = case_and_ref("mini_hash")
    cfg = case.cfg
    x_h = case.x.cpu().pin_memory()
    ids_h = case.input_ids.cpu().pin_memory()
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    il_h = torch.empty((cfg.T, cfg.k), dtype=torch.int32).pin_memory()
    gb.moe_forward_host(case.layer, x_h, input_ids_host=ids_h, out_host=out_h, ids_log_host=il_h)
    torch.cuda.synchronize()
    assert np.array_equal(il_h.numpy(), ref["ids_log"])
    assert_within_tol(out_h.float().numpy(), synth.bf16_to_f32(ref["out"]), "host out")


# ------------------------------------------------------------ edge cases
def _forward_vs_oracle(gb, cfg, logits=None, T=None):
    """Forward a (possibly truncated) small workload; compare with the oracle."""
    if T is not None:
        cfg = cfg.with_T(T)
    case = device_case(cfg, DEV, host_weights=True)
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids, ids_log=ids)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(ids), ref["ids_log"])
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), f"{cfg.name} T={cfg.T}")
    return ref


@pytest.mark.parametrize("T", [1, 2, 17, 33])
def test_small_and_ragged_token_counts(built, T):
    _forward_vs_oracle(built, synth.MINI["mini_decode"], T=T)
    _forward_vs_oracle(built, synth.MINI["mini_skew"], T=T)


def test_zero_tokens_is_a_noop(built):
    gb = built
    case, _ = case_and_ref("tiny")
    x0 = case.x[:0]
    out = gb.moe_forward(case.layer, x0)
    assert out.shape == (0, case.cfg.H)
    assert gb.check_device_status() == 0


def test_all_tokens_on_one_expert_and_empty_experts(built):
    gb = built
    # every token routed to experts {3, 0}: one group holds all rows (> 128: several
    # token blocks), six experts are empty
    cfg = synth.MINI["tiny"].with_T(300)
    case = device_case(cfg, DEV, host_weights=True)
    l = np.full((cfg.T, cfg.E), -4.0, np.float32)
    l[:, 3] = 5.0
    l[:, 0] = 4.0
    lt = torch.from_numpy(l).to(DEV)
    o = gb.moe_route(case.layer.cfg, logits=lt)
    assert (_np(o["ids_log"]) == np.array([3, 0])).all()
    perm = gb.moe_permute(o["ids_phys"], cfg.P, x=case.x)
    assert _np(perm["counts"]).tolist() == [300, 0, 0, 300, 0, 0, 0, 0]
    offs = perm["offsets"]
    act = gb.moe_gemm_gateup_act(perm["x_perm"], offs, case.dev["w_gate"], case.dev["w_up"])
    y = gb.moe_gemm_down(act, offs, case.dev["w_down"])
    out = gb.moe_combine(y, perm["flat_to_row"], o["weights"])
    assert gb.check_device_status() == 0
    ref = oracle.moe_forward(oracle.cfg_from(cfg), case.inputs["x"], cfg.H, cfg.I, logits=l,
                             wg=case.weights_host[0], wu=case.weights_host[1],
                             wd=case.weights_host[2])
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), "one-expert out")


def test_bad_table_entry_sets_device_status(built):
    gb = built
    case, _ = case_and_ref("mini_hash")
    bad = case.dev["tid2eid"].clone()
    row = int(case.inputs["input_ids"][0])
    bad[row, 1] = case.cfg.E + 7  # out of range: recorded, clamped, no fault
    gb.moe_route(case.layer.cfg, x=case.x, w_router=case.dev["w_router"],
                 input_ids=case.input_ids, tid2eid=bad)
    assert gb.check_device_status() == 5
    assert gb.check_device_status() == 0  # cleared by the read


@pytest.mark.parametrize("T", [300, 1500])  # one-block permutation; multi-kernel path
def test_out_of_range_ids_get_no_row(built, T):
    """Ids outside [0, P) are reported, not counted and get no row: their
    flat_to_row entries are -1, x_perm rows past offsets[P] are zero-filled
    (x is read only through rows the permutation wrote) and the combine adds
    nothing for them."""
    gb = built
    cfg = synth.MINI["mini_decode"].with_T(T)
    case = device_case(cfg, DEV, host_weights=False)
    k, P, H = cfg.k, cfg.P, cfg.H
    o = gb.moe_route(case.layer.cfg, x=case.x, w_router=case.dev["w_router"],
                     corr_bias=case.dev["corr_bias"])
    ids = o["ids_phys"].clone()
    bad = [(0, 1, P + 5), (T // 2, 0, -2), (T - 1, k - 1, 1 << 20)]
    for t, j, v in bad:
        ids[t, j] = v
    assert gb.check_device_status() == 0
    perm = gb.moe_permute(ids, P, x=case.x)
    assert gb.check_device_status() == 5  # GBMOE_ERR_DEVICE, then cleared
    ids_h = _np(ids).reshape(-1)
    valid = (ids_h >= 0) & (ids_h < P)
    n_ok = int(valid.sum())
    assert n_ok == T * k - len(bad)
    counts = np.bincount(ids_h[valid], minlength=P)
    assert np.array_equal(_np(perm["counts"]), counts)
    offs = np.concatenate([[0], np.cumsum(counts)])
    assert np.array_equal(_np(perm["offsets"]), offs)
    # stable order over the valid flat indices
    f_ok = np.nonzero(valid)[0]
    order = f_ok[np.argsort(ids_h[f_ok], kind="stable")]
    assert np.array_equal(_np(perm["row_to_token"])[:n_ok], order // k)
    f2r = _np(perm["flat_to_row"])
    exp_f2r = np.full(T * k, -1, np.int64)
    exp_f2r[order] = np.arange(n_ok)
    assert np.array_equal(f2r, exp_f2r)
    xp = _np(perm["x_perm"].view(torch.int16))
    xh = _np(case.x.view(torch.int16))
    assert np.array_equal(xp[:n_ok], xh[order // k])
    assert not xp[n_ok:].any()
    # combine over the same flat_to_row: the bad slots contribute nothing
    g = torch.Generator(device="cpu").manual_seed(5)
    y = torch.randn((T * k, H), generator=g).to(DEV)
    w = torch.rand((T, k), generator=g).to(DEV)
    out = gb.moe_combine(y, perm["flat_to_row"], w)
    assert gb.check_device_status() == 5
    yh, wh = _np(y).astype(np.float64), _np(w).astype(np.float64)
    exp = np.zeros((T, H))
    for f in range(T * k):
        if f2r[f] >= 0:
            exp[f // k] += wh[f // k, f % k] * yh[f2r[f]]
    got = _bf(out).astype(np.float64)
    assert np.all(np.abs(got - exp) <= 2.0 ** -7 * np.abs(exp) + 1e-5)


def test_device_generator_matches_host(built):
    cfg = synth.MINI["mini_decode"]
    n = cfg.I * cfg.H
    d = synth.normal_bf16_device(cfg.seed, synth.TAG_WG, 3, n, cfg.w_sigma, DEV)
    h = synth.normal_bf16(cfg.seed, synth.TAG_WG, 3, n, cfg.w_sigma)
    assert np.array_equal(_np(d.view(torch.int16)).view(np.uint16), h)


# every tile variant of the grouped GEMMs: gate/up with 128-token tiles (two
# accumulator buffers) and 256-token tiles (groups averaging >= 96 rows);
# down with paired 256-row weight blocks (H % 256 == 0) and, for other H,
# 128- and 256-token single-block tiles; empty, one-row and ragged groups
GEMM_SHAPES = [
    (384, 256, [150, 200, 300, 1, 0]),  # 256-token gate/up; 256-token unpaired down
    (384, 128, [40, 3, 17, 0, 90]),     # 128-token gate/up; 128-token unpaired down
    (512, 128, [40, 3, 17, 0, 90]),     # 128-token gate/up; paired down
    (256, 384, [260, 140]),             # 256-token gate/up; paired down
    (768, 256, [513, 129]),             # several token blocks per group; paired down
    # CTA-pair tiles (groups averaging >= 96 rows): gate/up with I % 256 == 0,
    # down with H % 512 == 0; ragged groups leave the odd CTA of a pair some,
    # or none, of a tile's token rows
    (1024, 512, [300, 5, 0, 400, 129]),
    (512, 256, [97, 33, 700, 1]),
]


def _gemm_case(shape):
    """Random bf16 tokens and expert weights for grouped GEMMs with the given
    (H, I, rows per group), and the oracle's act and y."""
    H, I, rows = shape
    rng = np.random.default_rng(H + I + len(rows))
    P = len(rows)
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(offs[-1])
    x = (rng.standard_normal((N, H))).astype(np.float32)
    from tests.test_oracle_mlp import _bf16_bits
    xb = _bf16_bits(x)
    W = [tuple(_bf16_bits(rng.standard_normal(s) * 0.05) for s in ((I, H), (I, H), (H, I)))
         for _ in range(P)]
    act_o = np.zeros((N, I), np.uint16)
    y_o = np.zeros((N, H), np.float32)
    for p in range(P):
        if rows[p]:
            a, y = oracle.expert_ffn_rows(xb[offs[p]:offs[p + 1]], *W[p], nthreads=4)
            act_o[offs[p]:offs[p + 1]] = a
            y_o[offs[p]:offs[p + 1]] = y
    dev = {"offs": torch.from_numpy(offs).to(DEV), "x": bf16_dev(xb, DEV),
           "wg": bf16_dev(np.stack([w[0] for w in W]), DEV),
           "wu": bf16_dev(np.stack([w[1] for w in W]), DEV),
           "wd": bf16_dev(np.stack([w[2] for w in W]), DEV)}
    return dev, act_o, y_o


@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_gemm_tile_variants(built, shape):
    gb = built
    d, act_o, y_o = _gemm_case(shape)
    act = gb.moe_gemm_gateup_act(d["x"], d["offs"], d["wg"], d["wu"])
    y = gb.moe_gemm_down(bf16_dev(act_o, DEV), d["offs"], d["wd"])
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(act), synth.bf16_to_f32(act_o), f"act {shape}")
    assert_within_tol(_np(y), y_o, f"y {shape}")
    # run-to-run determinism (bitwise), here also for the CTA-pair kernels'
    # TMA-store epilogues (blocks of 16 token rows written through shared memory)
    act2 = gb.moe_gemm_gateup_act(d["x"], d["offs"], d["wg"], d["wu"])
    y2 = gb.moe_gemm_down(bf16_dev(act_o, DEV), d["offs"], d["wd"])
    assert torch.equal(act.view(torch.int16), act2.view(torch.int16))
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


# both GEMMs through moe_expert_mlp: fused in one launch (groups averaging
# < 96 rows, H % 256 == 0) or as two launches; the 64-group shape has more
# tiles than SMs, so down tiles wait on gate/up tiles of other CTAs
MLP_SHAPES = [
    ((512, 128, [40, 3, 17, 0, 90]), True),
    ((256, 256, [1, 0, 0, 7, 64, 33, 2, 95]), True),
    ((1024, 512, [20 + (p * 7) % 23 for p in range(64)]), True),
    ((768, 256, [513, 129]), False),
    ((384, 128, [40, 3, 17, 0, 90]), False),
    ((1024, 512, [300, 5, 0, 400, 129]), False),  # CTA-pair tiles for both GEMMs
]


@pytest.mark.parametrize("shape,fused", MLP_SHAPES)
@pytest.mark.parametrize("gather", [False, True])
def test_expert_mlp_fused_and_separate(built, shape, fused, gather):
    gb = built
    H, I, rows = shape
    assert gb.expert_mlp_fused(len(rows), sum(rows), H) == fused
    d, act_o, y_o = _gemm_case(shape)
    ready = torch.full((len(rows),), 12345, dtype=torch.int32, device=DEV)
    offs = _np(d["offs"])
    wd = _bf(d["wd"]).astype(np.float64)
    src, r2t = d["x"], None
    if gather:
        # the same operand rows, gathered from a shuffled source with extra rows
        N = d["x"].shape[0]
        rng = np.random.default_rng(N + H)
        T = N + 37
        place = rng.permutation(T)[:N]
        xs = torch.zeros((T, H), dtype=torch.bfloat16, device=DEV)
        xs[torch.from_numpy(place).to(DEV)] = d["x"]
        src, r2t = xs, torch.from_numpy(place.astype(np.int32)).to(DEV)
    for rd in (ready, None):
        act, y = gb.moe_expert_mlp(src, d["offs"], d["wg"], d["wu"], d["wd"], ready=rd,
                                   row_to_token=r2t)
        assert gb.check_device_status() == 0
        assert_within_tol(_bf(act), synth.bf16_to_f32(act_o), f"act {shape}")
        # y is the down GEMM of the GPU's own activations (a one-ulp flip of a
        # large bf16 activation moves y by more than the output tolerance, so
        # y is checked against y = act . W_down^T taken in fp64 from those
        # activations, to within fp32 accumulation error)
        a64 = _bf(act).astype(np.float64)
        y_ref = np.zeros_like(y_o, dtype=np.float64)
        bound = np.zeros_like(y_ref)
        for p in range(len(rows)):
            r0, r1 = offs[p], offs[p + 1]
            y_ref[r0:r1] = a64[r0:r1] @ wd[p].T
            bound[r0:r1] = np.abs(a64[r0:r1]) @ np.abs(wd[p]).T
        err = np.abs(_np(y).astype(np.float64) - y_ref)
        assert np.all(err <= 2.0 ** -12 * bound + 1e-30), f"y {shape}: max err {err.max()}"
        if rd is not None and fused:
            # every gate/up tile of every group published exactly once: a group
            # of r rows is cut into ceil(r / 128) equal token blocks (a multiple
            # of 16 rows each), times I / 128 weight blocks
            def blocks(r):
                if r == 0:
                    return 0
                rpb = 16 * math.ceil(math.ceil(r / math.ceil(r / 128)) / 16)
                return math.ceil(r / rpb)
            assert _np(ready).tolist() == [(I // 128) * blocks(r) for r in rows]


def test_bounded_waits_report_timeout_and_context_survives(built):
    """A wait limit of 1 us on the fused launch (64 groups, more tiles than
    SMs): a down tile's wait for its expert's activations -- a poll of a
    counter that the other CTAs' gate/up tiles publish -- runs out, the CTA
    gives up (every role stops, drains its in-flight copies and MMAs, frees
    tensor memory), the CTAs waiting on its unpublished tiles give up too,
    and the launch reports GBMOE_ERR_TIMEOUT through the device status; the
    next launch with the default limit is correct.  (The pipeline's mbarrier
    waits check the clock between suspended polls, so a tiny limit does not
    reliably trip them in a short launch.)"""
    gb = built
    shape, fused = MLP_SHAPES[2]
    assert fused
    H, I, rows = shape
    d, act_o, _ = _gemm_case(shape)
    ready = torch.zeros((len(rows),), dtype=torch.int32, device=DEV)
    assert gb.check_device_status() == 0
    prev = gb.set_wait_limit_ns(1000)
    try:
        gb.moe_expert_mlp(d["x"], d["offs"], d["wg"], d["wu"], d["wd"], ready=ready)
        assert gb.check_device_status() == 6  # GBMOE_ERR_TIMEOUT
    finally:
        assert gb.set_wait_limit_ns(prev) == 1000
    assert gb.set_wait_limit_ns(0) == prev  # 0 restores the default
    act, y = gb.moe_expert_mlp(d["x"], d["offs"], d["wg"], d["wu"], d["wd"], ready=ready)
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(act), synth.bf16_to_f32(act_o), f"act after timeout {shape}")
    # the full layer still runs on this context
    case, ref = case_and_ref("mini_decode")
    out = gb.moe_forward(case.layer, case.x)
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), "forward after timeout")


# randomized forwards (the GPU machine has no hypothesis: a seeded draw of
# workload, token count and activation per case): ids bit-exact, outputs
# within tolerance, over token counts that cross the permutation's one-block
# limit and the GEMM variants' thresholds
def _random_cases(n=12, seed=2026):
    rng = np.random.default_rng(seed)
    names = sorted(synth.MINI)
    acts = ["swiglu", "swiglu_oai", "geglu", "geglu_tanh"]
    return [(names[rng.integers(len(names))], int(rng.integers(1, 700)),
             acts[rng.integers(len(acts))]) for _ in range(n)]


@pytest.mark.parametrize("name,T,act", _random_cases())
def test_random_forwards_match_oracle(built, name, T, act):
    gb = built
    cfg = synth.MINI[name].with_T(T)
    case = device_case(cfg, DEV, host_weights=True, activation=act)
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host, activation=act)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    idp = torch.empty_like(ids)
    cnt = torch.empty(cfg.P, dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids, ids_log=ids,
                         ids_phys=idp, counts=cnt)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(ids), ref["ids_log"])
    assert np.array_equal(_np(idp), ref["ids_phys"])
    assert np.array_equal(_np(cnt), ref["counts"])
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), f"{name} T={T} {act}")


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid", "sqrtsoftplus"])
def test_hash_forward_every_scoring(built, scoring):
    """Hash routing through moe_forward with every scoring function: with an
    elementwise score (sigmoid, sqrtsoftplus) only the logits of each token's
    hashed experts are computed, softmax needs them all; ids, routing
    weights and counts bit-exact against the oracle either way ([K3]
    "Stage 2: Select Experts", hash routing through tid2eid)."""
    import dataclasses
    gb = built
    cfg = dataclasses.replace(synth.MINI["mini_hash"], scoring=scoring, T=301)
    case = device_case(cfg, DEV, host_weights=True)
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
    ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    idp = torch.empty_like(ids)
    wts = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.P, dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids, ids_log=ids,
                         ids_phys=idp, weights=wts, counts=cnt)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(ids), ref["ids_log"])
    assert np.array_equal(_np(idp), ref["ids_phys"])
    assert np.array_equal(_np(wts).view(np.uint32), ref["weights"].view(np.uint32))
    assert np.array_equal(_np(cnt), ref["counts"])
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref["out"]), f"hash {scoring}")
