"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times (one moe_forward call over the whole batch).

For every token: router logits, expert ids (logical and physical), routing
weights and counts are compared bit for bit with the oracle, and the
permutation (offsets, row_to_token, flat_to_row) too.  Outputs are compared
on a seeded sample of tokens (at least 32 per workload, with the first and
the last) that the oracle recomputes one by one from host-generated expert
weights (the GPU's weights come from the bit-identical device generator,
which is also checked here on one expert).  The expert MLP is compared row by
row on every routed row of the two most- and the two least-loaded experts
(activations and expert outputs, through the same kernels moe_forward runs:
the largest groups span many token blocks and every K stage of H = 7168).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import device_case

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
N_SAMPLE = int(os.environ.get("GBMOE_TEST_SAMPLE", "32"))


def _np(t):
    return t.cpu().numpy()


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import routed_mixture_experts_gemm_gb300 as m
    return m


def _sampled_outputs(cfg, d, tokens, ids_phys, weights):
    """Oracle outputs of the sampled tokens, expert by expert."""
    pl = d["placement"]
    need = {}
    for t in tokens:
        for j in range(cfg.k):
            need.setdefault(int(pl.phys_to_log[ids_phys[t, j]]), []).append((t, j))
    y = {}

    def one(e):
        wg, wu, wd = synth.expert_weights_host(cfg, e)
        rows = need[e]
        _, ye = oracle.expert_ffn_rows(d["x"][[t for t, _ in rows]], wg, wu, wd, nthreads=1)
        return e, rows, ye

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        for e, rows, ye in ex.map(one, sorted(need)):
            for (t, j), r in zip(rows, ye):
                y[(t, j)] = r
    ys = None
    sw = synth.shared_weights_host(cfg)
    if sw is not None:
        _, ys = oracle.expert_ffn_rows(d["x"][tokens], *sw)
    outs = []
    for i, t in enumerate(tokens):
        yt = np.stack([y[(t, j)] for j in range(cfg.k)])
        outs.append(oracle.combine(yt, np.arange(cfg.k, dtype=np.int32), weights[t:t + 1],
                                   None if ys is None else ys[i:i + 1])[0])
    return np.stack(outs)


def _assert_tol(got, exp, what):
    got = np.asarray(got, np.float64)
    exp = np.asarray(exp, np.float64)
    err = np.abs(got - exp)
    bad = err > 1e-2 + 1e-2 * np.abs(exp)
    assert not bad.any(), f"{what}: {bad.sum()} of {err.size} outside tolerance, max {err.max()}"


def _check_extreme_experts(gb, cfg, case, perm):
    """Every routed row of the two most- and two least-loaded (non-empty)
    physical experts: act and y of moe_expert_mlp (the kernels and variant
    moe_forward runs for this shape) against the oracle's expert MLP."""
    d = case.inputs
    pl = d["placement"]
    dv = case.dev
    counts = _np(perm["counts"])
    offs = _np(perm["offsets"])
    r2t = _np(perm["row_to_token"])
    ready = torch.zeros(cfg.P, dtype=torch.int32, device=DEV)
    act, y = gb.moe_expert_mlp(case.x, perm["offsets"], dv["w_gate"], dv["w_up"], dv["w_down"],
                               ready=ready, row_to_token=perm["row_to_token"])
    assert gb.check_device_status() == 0
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    picks = sorted({*order[:2].tolist(), *order[-2:].tolist()})
    for p in picks:
        r0, r1 = int(offs[p]), int(offs[p + 1])
        wg, wu, wd = synth.expert_weights_host(cfg, int(pl.phys_to_log[p]))
        act_o, y_o = oracle.expert_ffn_rows(d["x"][r2t[r0:r1]], wg, wu, wd)
        _assert_tol(_np(act[r0:r1].float()), synth.bf16_to_f32(act_o),
                    f"act of slot {p} ({r1 - r0} rows)")
        _assert_tol(_np(y[r0:r1]), y_o, f"y of slot {p} ({r1 - r0} rows)")
    del act, y
    return [(int(p), int(counts[p])) for p in picks]


@pytest.mark.parametrize("name", ["decode", "prefill", "hash", "skew"])
def test_full_size(gb, name):
    cfg = synth.CONFIGS[name]
    case = device_case(cfg, DEV, host_weights=False)
    d = case.inputs
    pl = d["placement"]
    T, k = cfg.T, cfg.k
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    idp = torch.empty_like(ids)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    cnt = torch.empty(cfg.P, dtype=torch.int32, device=DEV)
    out = gb.moe_forward(case.layer, case.x, input_ids=case.input_ids, ids_log=ids,
                         ids_phys=idp, weights=w, counts=cnt)
    assert gb.check_device_status() == 0

    # routing of every token, bit for bit
    logits = oracle.router_logits(d["x"], d["w_router"], d["router_bias"])
    ids_o, idp_o, w_o = oracle.route(oracle.cfg_from(cfg), logits, corr_bias=d["corr_bias"],
                                     input_ids=d["input_ids"], tid2eid=d["tid2eid"],
                                     log2phy=pl.log2phy, replica_cnt=pl.replica_cnt)
    assert np.array_equal(_np(ids), ids_o)
    assert np.array_equal(_np(idp), idp_o)
    assert np.array_equal(_np(w).view(np.uint32), w_o.view(np.uint32))
    counts_o, offs_o, r2t_o, f2r_o = oracle.permute(idp_o, cfg.P)
    assert np.array_equal(_np(cnt), counts_o)
    perm = gb.moe_permute(idp, cfg.P)
    assert np.array_equal(_np(perm["offsets"]), offs_o)
    assert np.array_equal(_np(perm["row_to_token"]), r2t_o)
    assert np.array_equal(_np(perm["flat_to_row"]), f2r_o)
    picked = _check_extreme_experts(gb, cfg, case, perm)
    assert len(picked) >= 2, picked
    rl = gb.moe_route(case.layer.cfg, x=case.x, w_router=case.dev["w_router"],
                      router_bias=case.dev["router_bias"], corr_bias=case.dev["corr_bias"],
                      input_ids=case.input_ids, tid2eid=case.dev["tid2eid"],
                      log2phy=case.dev["log2phy"], replica_cnt=case.dev["replica_cnt"])
    assert np.array_equal(_np(rl["logits"]).view(np.uint32), logits.view(np.uint32))

    # the device-generated weights are the host generator's bits (one expert)
    e0 = int(pl.phys_to_log[int(idp_o[0, 0])])
    wg_h = synth.expert_weights_host(cfg, e0)[0]
    wg_d = case.dev["w_gate"][int(idp_o[0, 0])]
    assert np.array_equal(_np(wg_d.view(torch.int16)).view(np.uint16), wg_h)

    # sampled outputs, including the first and last token
    rng = np.random.default_rng(cfg.seed + 100)
    sample = sorted({0, T - 1, *rng.choice(T, min(T, N_SAMPLE), replace=False).tolist()})
    assert len(sample) >= min(T, 32)
    exp = synth.bf16_to_f32(_sampled_outputs(cfg, d, sample, idp_o, w_o)).astype(np.float64)
    got = _np(out[sample].float()).astype(np.float64)
    err = np.abs(got - exp)
    bad = err > 1e-2 + 1e-2 * np.abs(exp)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert not bad.any(), (f"{bad.sum()} of {err.size} outside tolerance; max err {err.max()} "
                           f"at |oracle| {abs(exp[i])}; rms err {np.sqrt((err ** 2).mean())}")
    assert err.max() <= 2 * 2.0 ** -8 * np.abs(exp).max()
    del case, out
    torch.cuda.empty_cache()


# ---- quantized routed experts at full size (FP8 rows; MX E4M3 / E2M1)
QKINDS = {"fp8_row": None, "mxfp8": "e4m3", "w4a8": "e2m1"}


def _quantized_layer(gb, case, kind):
    dv = case.dev
    kw = dict(router_bias=dv["router_bias"], corr_bias=dv["corr_bias"], tid2eid=dv["tid2eid"],
              log2phy=dv["log2phy"], replica_cnt=dv["replica_cnt"], shared=dv["shared"])
    fmt = QKINDS[kind]
    if fmt is None:
        q = [gb.quantize_experts_fp8(dv[n]) for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, dv["w_router"], None, None, None,
                            fp8=[a for pair in q for a in pair], **kw)
    else:
        q = [gb.quantize_experts_mx(dv[n], fmt) for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, dv["w_router"], None, None, None,
                            mx=[fmt] + [a for pair in q for a in pair], **kw)
    return layer, q


def _oracle_quantized_rows(cfg, d, kind, q_dev, need, tokens):
    """y of the sampled (token, slot) pairs from the oracle's quantized MLP,
    expert by expert, after checking the GPU's weight codes of each expert."""
    fmt = QKINDS[kind]
    xs_rows = d["x"][tokens]
    pos = {t: i for i, t in enumerate(tokens)}
    if fmt is None:
        xq, xsc = oracle.quantize_rows(xs_rows)
    else:
        xq, xsc = oracle.mx_quantize_rows(xs_rows, "e4m3")
    pl = d["placement"]

    def one(p):
        e = int(pl.phys_to_log[p])
        mats = synth.expert_weights_host(cfg, e)
        qo = []
        for m, (wq, ws) in zip(mats, q_dev):
            cq, cs = (oracle.quantize_rows(m) if fmt is None else oracle.mx_quantize_rows(m, fmt))
            assert np.array_equal(_np(wq[p]), cq.reshape(wq[p].shape)), f"codes of slot {p}"
            assert np.array_equal(_np(ws[p]).view(np.uint8), cs.reshape(ws[p].shape)
                                  .view(np.uint8)), f"scales of slot {p}"
            qo += [cq[None], cs[None]]
        rows = need[p]
        r2t = np.array([pos[t] for t, _ in rows], np.int32)
        offs = np.array([0, len(rows)], np.int32)
        if fmt is None:
            _, y = oracle.ffn_grouped_fp8(xq, xsc, r2t, offs, *qo, nthreads=1)
        else:
            _, _, _, y = oracle.ffn_grouped_mx(xq, xsc, r2t, offs, *qo, wfmt=fmt, nthreads=1)
        return rows, y

    out = {}
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        for rows, y in ex.map(one, sorted(need)):
            for (t, j), r in zip(rows, y):
                out[(t, j)] = r
    return out


@pytest.mark.parametrize("name,kind", [("decode", "fp8_row"), ("decode", "mxfp8"),
                                       ("decode", "w4a8"), ("prefill", "fp8_row"),
                                       ("prefill", "mxfp8"), ("prefill", "w4a8"),
                                       ("hash", "w4a8"), ("skew", "fp8_row")])
def test_full_size_quantized(gb, name, kind):
    cfg = synth.CONFIGS[name]
    case = device_case(cfg, DEV, host_weights=False)
    d = case.inputs
    pl = d["placement"]
    T, k = cfg.T, cfg.k
    layer, q = _quantized_layer(gb, case, kind)
    idp = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    out = gb.moe_forward(layer, case.x, input_ids=case.input_ids, ids_phys=idp, weights=w)
    assert gb.check_device_status() == 0
    # routing of every token, bit for bit (the router is not quantized)
    logits = oracle.router_logits(d["x"], d["w_router"], d["router_bias"])
    _, idp_o, w_o = oracle.route(oracle.cfg_from(cfg), logits, corr_bias=d["corr_bias"],
                                 input_ids=d["input_ids"], tid2eid=d["tid2eid"],
                                 log2phy=pl.log2phy, replica_cnt=pl.replica_cnt)
    assert np.array_equal(_np(idp), idp_o)
    assert np.array_equal(_np(w).view(np.uint32), w_o.view(np.uint32))
    # sampled outputs, including the first and last token
    rng = np.random.default_rng(cfg.seed + 200)
    sample = sorted({0, T - 1, *rng.choice(T, max(2, N_SAMPLE // 2), replace=False).tolist()})
    ys = None
    sw = synth.shared_weights_host(cfg)
    if sw is not None:  # the shared expert stays bf16
        _, ys = oracle.expert_ffn_rows(d["x"][sample], *sw)
    need = {}
    for t in sample:
        for j in range(k):
            need.setdefault(int(idp_o[t, j]), []).append((t, j))
    y = _oracle_quantized_rows(cfg, d, kind, q, need, sample)
    exp = []
    for i, t in enumerate(sample):
        yt = np.stack([y[(t, j)] for j in range(k)])
        exp.append(oracle.combine(yt, np.arange(k, dtype=np.int32), w_o[t:t + 1],
                                  None if ys is None else ys[i:i + 1])[0])
    exp = synth.bf16_to_f32(np.stack(exp)).astype(np.float64)
    got = _np(out[sample].float()).astype(np.float64)
    err = np.abs(got - exp)
    bad = err > 1e-2 + 1e-2 * np.abs(exp)
    assert not bad.any(), f"{kind} {name}: {bad.sum()} of {err.size} outside, max {err.max()}"
    assert err.max() <= 2 * 2.0 ** -8 * np.abs(exp).max()
    del case, out, layer, q
    torch.cuda.empty_cache()
