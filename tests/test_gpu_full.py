"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times (one moe_forward call over the whole batch).

For every token: router logits, expert ids (logical and physical), routing
weights and counts are compared bit for bit with the oracle, and the
permutation (offsets, row_to_token, flat_to_row) too.  Outputs are compared
on a seeded sample of tokens that the oracle recomputes one by one from
host-generated expert weights (the GPU's weights come from the bit-identical
device generator, which is also checked here on one expert).
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
N_SAMPLE = int(os.environ.get("GBMOE_TEST_SAMPLE", "6"))


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
    sample = sorted({0, T - 1, *rng.choice(T, N_SAMPLE, replace=False).tolist()})
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
