"""Device tensors and an MoELayer for a synth workload (plumbing for the tests,
the smoke check and the benchmark; no MoE arithmetic).

Small workloads take every input from the host generator (so the oracle sees
the same bits); large ones generate the expert weight stacks directly on the
device with the bit-identical torch restatement of the generator.
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import synth


@dataclass
class Case:
    cfg: synth.MoEConfig
    inputs: dict
    x: torch.Tensor
    input_ids: Optional[torch.Tensor]
    layer: object
    dev: dict
    weights_host: Optional[tuple]


def _t(a, device, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def bf16_dev(bits, device):
    return _t(np.ascontiguousarray(bits, dtype=np.uint16), device, torch.bfloat16)


def device_case(cfg: synth.MoEConfig, device, host_weights: Optional[bool] = None,
                activation: str = "swiglu") -> Case:
    import routed_mixture_experts_gemm_gb300 as gb
    d = synth.make_inputs(cfg)
    pl = d["placement"]
    if host_weights is None:
        host_weights = cfg.P * cfg.I * cfg.H <= (1 << 26)
    if host_weights:
        wh = synth.all_expert_weights_host(cfg)
        wg, wu, wd = (bf16_dev(w, device) for w in wh)
    else:
        wh = None
        wg, wu, wd = synth.expert_weights_device(cfg, device)
    shared = None
    if cfg.shared_I:
        if host_weights:
            shared = tuple(bf16_dev(w, device) for w in synth.shared_weights_host(cfg))
        else:
            shared = synth.shared_weights_device(cfg, device)
    dev = {
        "w_router": _t(d["w_router"], device),
        "router_bias": _t(d["router_bias"], device),
        "corr_bias": _t(d["corr_bias"], device),
        "tid2eid": _t(d["tid2eid"], device),
        "log2phy": _t(pl.log2phy, device),
        "replica_cnt": _t(pl.replica_cnt, device),
        "w_gate": wg, "w_up": wu, "w_down": wd, "shared": shared,
    }
    rc = gb.route_cfg(cfg.E, cfg.k, cfg.scoring, E_phys=cfg.P, n_group=cfg.n_group,
                      topk_group=cfg.topk_group, group_score=cfg.group_score_mode,
                      renormalize=cfg.renormalize, routed_scaling=cfg.routed_scaling,
                      use_hash=cfg.use_hash)
    layer = gb.MoELayer(rc, dev["w_router"], wg, wu, wd, router_bias=dev["router_bias"],
                        corr_bias=dev["corr_bias"], tid2eid=dev["tid2eid"],
                        log2phy=dev["log2phy"], replica_cnt=dev["replica_cnt"], shared=shared,
                        activation=activation)
    x = bf16_dev(d["x"], device)
    ids = _t(d["input_ids"], device)
    return Case(cfg, d, x, ids, layer, dev, wh)
