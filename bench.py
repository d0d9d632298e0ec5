"""Benchmark of the routed-MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode]
                    [--impl reference]

One step = one moe_forward over one batch of the workload (router scoring and
grouped top-k, permutation, grouped gate/up GEMM + SwiGLU, grouped down GEMM,
combine; shared expert where the workload has one), inputs and weights
resident in HBM.  Prints ONE JSON line (rank 0):

  value     tokens/s of the headline workload (decode shape, T=128), device
            time by CUDA events on the launching stream, max over ranks
  e2e       the same metric through moe_forward_host with pinned host
            buffers: host->device copy of x and device->host copy of out
            inside the timed region
  sustained the decode step repeated for >= 1 s, with its clock samples
  prefill   the same measurement at T=8192 (the metric's second batch size),
  hash      at T=2048 with hash routing over 384 experts, and
  skew      at T=4096 with Zipf-skewed load, replicated hot experts and a
            shared expert (each timed for >= 1 s, with per-stage times)
  roofline  the dominant kernel (the fused expert launch, or the gate/up
            grouped GEMM) against the measured peak of its bound: HBM bytes
            of the touched experts' weights and x when the expert groups sit
            below the ridge (decode, hash, skew), tensor FLOPs at or above it
            (prefill)
  cpu_baseline  the CPU oracle timed on this host on a bounded token sample
  quantized both workloads again with quantized routed experts: FP8 E4M3
            with one scale per row, MXFP8 (E4M3, a power-of-two scale per 32
            elements) and W4A8 (MX E2M1 weights, MX E4M3 activations):
            throughput, the expert-stage kernel times and the gate/up GEMM's
            roofline (--no-quant skips them)

--impl reference times the CPU oracle itself (the only reference there is:
the pages publish no implementation), on the same workload and metric.

Multi-GPU (torchrun, N > 1): every rank runs an independent replica of the
workload (weak scaling, no collective on the data path); value = tokens all
ranks processed / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import datetime
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s at T=128 and T=8192; % of HBM / bf16 TC roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ["routed_mixture_experts_gemm_gb300/csrc/gemm.cu",
                "routed_mixture_experts_gemm_gb300/csrc/common.cuh"]

# small twins of the decode / prefill shapes for ncu captures (weights > L2,
# a few GB on the device): same H, I, k and rows-per-expert character
PROFILE_WORKLOADS = {
    "decode_e16": synth.MoEConfig("decode_e16", 21, T=8, H=7168, I=2048, E=16, k=8,
                                  scoring="sigmoid", n_group=8, topk_group=4,
                                  routed_scaling=2.5, corr_bias_sigma=0.1),
    "prefill_e16": synth.MoEConfig("prefill_e16", 22, T=512, H=7168, I=2048, E=16, k=8,
                                   scoring="sigmoid", n_group=8, topk_group=4,
                                   routed_scaling=2.5, corr_bias_sigma=0.1, router_sigma=None),
    # 256 rows per expert like prefill, 32 experts (2.8 GB of weights)
    "prefill_e32": synth.MoEConfig("prefill_e32", 24, T=1024, H=7168, I=2048, E=32, k=8,
                                   scoring="sigmoid", n_group=8, topk_group=4,
                                   routed_scaling=2.5, corr_bias_sigma=0.1, router_sigma=None),
    # the hash workload's character: hash routing, ~43 rows per expert (the
    # fused launch), 48 experts (4.2 GB of weights)
    "hash_e48": synth.MoEConfig("hash_e48", 26, T=256, H=7168, I=2048, E=48, k=8,
                                scoring="sqrtsoftplus", routed_scaling=2.5, hash_vocab=163840),
    # the skew workload's character: Zipf(1.1) router bias, the hottest
    # experts replicated (36 slots, ~114 rows per slot: CTA-pair gate/up below
    # the ridge), a shared expert; 3.3 GB of weights
    "skew_e32": synth.MoEConfig("skew_e32", 27, T=512, H=7168, I=2048, E=32, k=8,
                                scoring="sigmoid", routed_scaling=2.5, zipf_s=1.1,
                                n_hot_replicas=4, shared_I=2048),
    # the decode router / permutation / combine shapes with small experts
    "decode_i128": synth.MoEConfig("decode_i128", 25, T=128, H=7168, I=128, E=256, k=8,
                                   scoring="sigmoid", n_group=8, topk_group=4,
                                   routed_scaling=2.5, corr_bias_sigma=0.1),
    # the prefill router / permutation / combine shapes with small experts
    "prefill_i128": synth.MoEConfig("prefill_i128", 23, T=8192, H=7168, I=128, E=256, k=8,
                                    scoring="sigmoid", n_group=8, topk_group=4,
                                    routed_scaling=2.5, corr_bias_sigma=0.1, router_sigma=None),
}


def workload(name):
    if name in synth.CONFIGS:
        return synth.CONFIGS[name]
    return PROFILE_WORKLOADS[name]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash():
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, wl: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{wl}")
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle reasons;
    only samples taken between mark_start() and mark_end() are summarised."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                clk, m = float(f[1]), float(f[2])
            except (ValueError, IndexError):
                continue
            if self.t0 is not None and not (self.t0 <= ts <= self.t1):
                continue
            sm.append(clk)
            mx = m
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_median": statistics.median(pw) if pw else None}


# --------------------------------------------------------------- GPU path
class Workload:
    """Device inputs, weights and preallocated buffers of one workload."""

    def __init__(self, cfg, device):
        import torch
        from synth.device import device_case
        import routed_mixture_experts_gemm_gb300 as gb
        self.cfg = cfg
        self.gb = gb
        self.lib = gb.library()
        self.case = device_case(cfg, device, host_weights=False)
        T, k, P = cfg.T, cfg.k, cfg.P
        self.torch = torch
        self.out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=device)
        self.ids = torch.empty((T, k), dtype=torch.int32, device=device)
        self.idp = torch.empty((T, k), dtype=torch.int32, device=device)
        self.w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.counts = torch.empty(P, dtype=torch.int32, device=device)
        self.ws = self.case.layer.workspace(T)
        # staged buffers (same kernels as moe_forward, one call per stage)
        N = T * k
        e = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device=device)  # noqa: E731
        self.logits = e(T, cfg.E, dt=torch.float32)
        self.offsets = e(P + 1, dt=torch.int32)
        self.r2t = e(N, dt=torch.int32)
        self.f2r = e(N, dt=torch.int32)
        self.act = e(N, cfg.I)
        self.y = e(N, cfg.H, dt=torch.float32)
        if cfg.shared_I:
            self.act_s = e(T, cfg.shared_I)
            self.ys = e(T, cfg.H, dt=torch.float32)
        self.pws = e(max(1, self.lib.gbmoe_permute_workspace_size(T, k, P)), dt=torch.uint8)
        self.ready = e(P, dt=torch.int32)
        # moe_forward runs both expert GEMMs as one launch for small groups
        self.fused = bool(self.lib.gbmoe_expert_mlp_fused(P, N, cfg.H))
        self.stream = torch.cuda.current_stream()

    def forward(self):
        c = self.case
        self.gb.moe_forward(c.layer, c.x, input_ids=c.input_ids, out=self.out, ids_log=self.ids,
                            ids_phys=self.idp, weights=self.w, counts=self.counts, ws=self.ws,
                            stream=self.stream)

    def staged(self, ev):
        """The forward as separate C-ABI calls with an event after each stage."""
        L, cfg, c, s = self.lib, self.cfg, self.case, self.stream.cuda_stream
        d = c.dev
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        R = 1 if d["log2phy"] is None else d["log2phy"].shape[1]
        rows = 0 if d["tid2eid"] is None else d["tid2eid"].shape[0]
        T, k, P, H, I = cfg.T, cfg.k, cfg.P, cfg.H, cfg.I
        N = T * k
        ev[0].record(self.stream)
        st = L.moe_route(ctypes.byref(c.layer.cfg), p(c.x), T, H, p(d["w_router"]), p(self.logits),
                         p(d["router_bias"]), p(d["corr_bias"]), p(c.input_ids), p(d["tid2eid"]),
                         rows, p(d["log2phy"]), p(d["replica_cnt"]), R, p(self.ids), p(self.idp),
                         p(self.w), None, s)
        ev[1].record(self.stream)
        # the permutation writes no x_perm: the gate/up GEMM gathers the rows
        st |= L.moe_permute(p(self.idp), T, k, P, None, 0, p(self.counts), p(self.offsets),
                            p(self.r2t), p(self.f2r), None, p(self.pws), self.pws.numel(), s)
        ev[2].record(self.stream)
        if self.fused:
            st |= L.moe_expert_mlp(p(c.x), p(self.r2t), T, p(self.offsets), P, N, H, I,
                                   p(d["w_gate"]), p(d["w_up"]), p(d["w_down"]), 0, p(self.act),
                                   p(self.y), p(self.ready), s)
            ev[3].record(self.stream)
        else:
            st |= L.moe_gemm_gateup_act_rows(p(c.x), p(self.r2t), T, p(self.offsets), P, N, H,
                                             I, p(d["w_gate"]), p(d["w_up"]), 0, p(self.act), s)
            ev[3].record(self.stream)
            st |= L.moe_gemm_down(p(self.act), p(self.offsets), P, N, H, I, p(d["w_down"]),
                                  p(self.y), s)
        ev[4].record(self.stream)
        ys = None
        if cfg.shared_I:
            sg, su, sd = d["shared"]
            st |= L.moe_gemm_gateup_act(p(c.x), None, 1, T, H, cfg.shared_I, p(sg), p(su), 0,
                                        p(self.act_s), s)
            st |= L.moe_gemm_down(p(self.act_s), None, 1, T, H, cfg.shared_I, p(sd), p(self.ys), s)
            ys = self.ys
        ev[5].record(self.stream)
        st |= L.moe_combine(p(self.y), p(self.f2r), p(self.w), p(ys), T, k, H, p(self.out), s)
        ev[6].record(self.stream)
        if st:
            raise RuntimeError(f"staged forward failed (status bits {st})")

    # ---- quantized routed experts: "fp8_row" (E4M3, one fp32 scale per row),
    # "mxfp8" (MX E4M3 weights and activations), "w4a8" (MX E2M1 weights, MX
    # E4M3 activations)
    QUANT = ("fp8_row", "mxfp8", "w4a8")

    def enable_quant(self, kind):
        """Quantized copies of the routed experts' weights (made on the device
        by the library's quantizers) and a layer that runs on them."""
        c, d, T, cfg = self.case, self.case.dev, self.cfg.T, self.cfg
        e = lambda *s, dt: self.torch.empty(s, dtype=dt, device=c.x.device)  # noqa: E731
        u8, f32 = self.torch.uint8, self.torch.float32
        kw = dict(router_bias=d["router_bias"], corr_bias=d["corr_bias"], tid2eid=d["tid2eid"],
                  log2phy=d["log2phy"], replica_cnt=d["replica_cnt"], shared=d["shared"])
        self.qkind = kind
        if kind == "fp8_row":
            q = [self.gb.quantize_experts_fp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
            self.wq = [a for pair in q for a in pair]
            self.layer_q = self.gb.MoELayer(c.layer.cfg, d["w_router"], None, None, None,
                                            fp8=self.wq, **kw)
            self.xs, self.as_ = e(T, dt=f32), e(cfg.N, dt=f32)
        else:
            self.wfmt = "e4m3" if kind == "mxfp8" else "e2m1"
            q = [self.gb.quantize_experts_mx(d[k], self.wfmt) for k in ("w_gate", "w_up",
                                                                          "w_down")]
            self.wq = [a for pair in q for a in pair]
            self.layer_q = self.gb.MoELayer(c.layer.cfg, d["w_router"], None, None, None,
                                            mx=[self.wfmt] + self.wq, **kw)
            # the GEMMs called stage by stage take the weight scales tiled
            self.wq = [self.gb.moe_mx_tile_scales(a) if i % 2 else a
                       for i, a in enumerate(self.wq)]
            self.xs, self.as_ = e(T, cfg.H // 32, dt=u8), e(cfg.N, cfg.I // 32, dt=u8)
        self.ws_q = self.layer_q.workspace(T)
        self.xq = e(T, cfg.H, dt=u8)
        self.aq = e(cfg.N, cfg.I, dt=u8)

    def disable_quant(self):
        for k in ("wq", "layer_q", "ws_q", "xq", "aq", "xs", "as_"):
            setattr(self, k, None)

    def forward_q(self):
        c = self.case
        self.gb.moe_forward(self.layer_q, c.x, input_ids=c.input_ids, out=self.out,
                            ids_log=self.ids, ids_phys=self.idp, weights=self.w,
                            counts=self.counts, ws=self.ws_q, stream=self.stream)

    def staged_q_experts(self, ev):
        """The quantized expert stage as separate C-ABI calls (the routing and
        the permutation from the last staged() call).  fp8_row: quantize x,
        gate/up, quantize act, down; MX: quantize x, gate/up with the
        activation quantized in its epilogue, down."""
        L, cfg, c, s = self.lib, self.cfg, self.case, self.stream.cuda_stream
        p = lambda t: t.data_ptr()  # noqa: E731
        T, P, N, H, I = cfg.T, cfg.P, cfg.N, cfg.H, cfg.I
        wg, sg, wu, su, wd, sd = self.wq
        ev[0].record(self.stream)
        if self.qkind == "fp8_row":
            st = L.moe_quantize_fp8_rows(p(c.x), T, H, p(self.xq), p(self.xs), s)
            ev[1].record(self.stream)
            st |= L.moe_gemm_gateup_act_fp8(p(self.xq), p(self.xs), p(self.r2t), T,
                                            p(self.offsets), P, N, H, I, p(wg), p(sg), p(wu),
                                            p(su), 0, p(self.act), s)
            ev[2].record(self.stream)
            st |= L.moe_quantize_fp8_rows(p(self.act), N, I, p(self.aq), p(self.as_), s)
            ev[3].record(self.stream)
            st |= L.moe_gemm_down_fp8(p(self.aq), p(self.as_), p(self.offsets), P, N, H, I, p(wd),
                                      p(sd), p(self.y), s)
        else:
            f = 0 if self.wfmt == "e4m3" else 1
            st = L.moe_quantize_mx_rows(p(c.x), T, H, 0, p(self.xq), p(self.xs), s)
            ev[1].record(self.stream)
            st |= L.moe_gemm_gateup_act_mx(p(self.xq), p(self.xs), p(self.r2t), T,
                                           p(self.offsets), P, N, H, I, f, p(wg), p(sg), p(wu),
                                           p(su), 0, p(self.aq), p(self.as_), s)
            ev[2].record(self.stream)
            ev[3].record(self.stream)
            st |= L.moe_gemm_down_mx(p(self.aq), p(self.as_), p(self.offsets), P, N, H, I, f,
                                     p(wd), p(sd), p(self.y), s)
        ev[4].record(self.stream)
        if st:
            raise RuntimeError(f"staged {self.qkind} experts failed (status bits {st})")

    def launches_per_step_q(self):
        # the bf16 step with the expert MLP replaced: fp8_row 4 launches
        # (quantize x, gate/up, quantize act, down), MX 3 (quantize x, gate/up
        # with the quantized activation, down)
        cfg = self.cfg
        perm = 1 if (cfg.N <= 4096 and cfg.P <= 1024) else 3
        mlp = 4 if self.qkind == "fp8_row" else 3
        return 2 + perm + mlp + (2 if cfg.shared_I else 0) + 1

    def launches_per_step(self):
        cfg = self.cfg
        # route: logits + select; permute: one block (N <= 4096, P <= 1024) or
        # histogram, column scan, scatter (the GEMM gathers the rows); gate/up
        # GEMM and down GEMM, or both in one fused launch (+2 for the shared
        # expert); combine
        perm = 1 if (cfg.N <= 4096 and cfg.P <= 1024) else 3
        return 2 + perm + (1 if self.fused else 2) + (2 if cfg.shared_I else 0) + 1


def time_device(fn, steps, warmup, torch, barrier=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1) / 1000.0


def stage_times(wl, steps, torch):
    names = ["route", "permute", "expert_mlp_fused" if wl.fused else "gemm_gateup",
             "gemm_down", "shared_expert", "combine"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for _ in range(3):
        wl.staged(evs[0])
    torch.cuda.synchronize()
    for i in range(steps):
        wl.staged(evs[i])
    torch.cuda.synchronize()
    out = {}
    for j, n in enumerate(names):
        if n == "gemm_down" and wl.fused:
            continue
        out[n] = sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
    return out  # ms per step


def touched_bytes(cfg, counts, fused=False):
    """Algorithmic bytes of the gate/up GEMM (the survey's definition: the
    weights of the experts with rows, plus the hidden states read once -- the
    GEMM gathers the routed rows from x, repeats hit L2); fused with the down
    GEMM, all three weight matrices of the touched experts.  Returned apart:
    the intermediate bytes the launch also moves and that are not credited
    (the activation written; fused: read back too, and the fp32 expert
    outputs written)."""
    touched = int((counts > 0).sum())
    w = touched * (3 if fused else 2) * cfg.I * cfg.H * 2
    x = cfg.T * cfg.H * 2
    inter = cfg.N * cfg.I * 2
    if fused:
        inter += cfg.N * cfg.I * 2 + cfg.N * cfg.H * 4
    return w + x, touched, inter


def q_stage_times(wl, steps, torch):
    names = ["quantize_x", "gemm_gateup", "quantize_act", "gemm_down"]
    wl.staged([torch.cuda.Event(enable_timing=True) for _ in range(7)])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for _ in range(3):
        wl.staged_q_experts(evs[0])
    torch.cuda.synchronize()
    for i in range(steps):
        wl.staged_q_experts(evs[i])
    torch.cuda.synchronize()
    out = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
           for j, n in enumerate(names)}
    if wl.qkind != "fp8_row":
        del out["quantize_act"]  # fused into the gate/up epilogue
    return out


def q_bytes(cfg, counts, kind):
    """Algorithmic bytes of the quantized gate/up and down GEMMs: weight codes
    of the experts with rows (1 byte per element, 1/2 for E2M1) and their
    scales (fp32 per row, or one byte per 32 elements), plus the token
    operand read once: gate/up reads each token's codes and scales (gathered,
    repeats hit L2), down the activation codes and scales.  The outputs
    written (the activation, the fp32 expert outputs) are intermediates of the
    layer and not credited."""
    touched = int((counts > 0).sum())
    H, I, T, N = cfg.H, cfg.I, cfg.T, cfg.N
    if kind == "fp8_row":
        g = touched * 2 * I * (H + 4) + T * (H + 4)
        d = touched * H * (I + 4) + N * (I + 4)
    else:
        wb = 1.0 if kind == "mxfp8" else 0.5
        g = touched * 2 * I * (H * wb + H / 32) + T * (H + H / 32)
        d = touched * H * (I * wb + I / 32) + N * (I + I / 32)
    return g, d


def q_measure(wl, kind, steps, warmup, torch, barrier, peaks, peak_src, world, bound, local):
    """The same workload with quantized routed experts: whole-layer throughput,
    the expert-stage kernel times and the gate/up GEMM's roofline."""
    wl.enable_quant(kind)
    wl.forward_q()
    torch.cuda.synchronize()
    est = time_device(wl.forward_q, 3, warmup, torch, barrier) / 3
    n = max(steps, int(1.0 / max(est, 1e-6)))
    with ClockSampler(local) as clk:
        clk.mark_start()
        secs = time_device(wl.forward_q, n, 1, torch, barrier)
        clk.mark_end()
    stg = q_stage_times(wl, min(steps, 20), torch)
    cfg = wl.cfg
    gb_, db_ = q_bytes(cfg, wl.counts.cpu().numpy(), kind)
    g1 = stg["gemm_gateup"] / 1000.0
    g2 = stg["gemm_down"] / 1000.0
    kname = {"fp8_row": "grouped_gemm FP8 gate/up + SwiGLU (tcgen05 kind::f8f6f4)",
             "mxfp8": "grouped_gemm MXFP8 gate/up + SwiGLU + MX quantization "
                      "(tcgen05 kind::mxf8f6f4 block_scale)",
             "w4a8": "grouped_gemm E2M1 x E4M3 gate/up + SwiGLU + MX quantization "
                     "(tcgen05 kind::mxf8f6f4 block_scale)"}[kind]
    if bound == "hbm":
        hbm = peaks["hbm_gbs"]
        roof = {"kernel": kname, "bound": "hbm", "achieved": gb_ / g1 / 1e9, "peak": hbm,
                "unit": "GB/s", "frac": gb_ / g1 / 1e9 / hbm,
                "traffic": profiled_traffic(f"{kind}_gateup", cfg.name),
                "algorithmic_bytes": gb_,
                "down": {"achieved": db_ / g2 / 1e9, "frac": db_ / g2 / 1e9 / hbm,
                         "algorithmic_bytes": db_},
                "peak_source": f"{peak_src} hbm_gbs"}
    else:
        # nominal fp8 / bf16 dense tensor ratio 2 on the measured bf16 peak
        # (E2M1 x E4M3 runs at the fp8 rate)
        pk = 2.0 * peaks["bf16_tflops_sustained"]
        f1 = 2.0 * cfg.N * 2 * cfg.H * cfg.I
        f2 = 2.0 * cfg.N * cfg.H * cfg.I
        roof = {"kernel": kname, "bound": "tensor", "achieved": f1 / g1 / 1e12, "peak": pk,
                "unit": "TFLOP/s", "frac": f1 / g1 / 1e12 / pk,
                "traffic": profiled_traffic(f"{kind}_gateup", cfg.name),
                "down": {"achieved": f2 / g2 / 1e12, "frac": f2 / g2 / 1e12 / pk},
                "peak_source": f"{peak_src} bf16_tflops_sustained x 2 (nominal fp8/bf16 ratio)"}
    res = {"workload": cfg.name, "T": cfg.T,
           "dtype": {"fp8_row": "e4m3 x e4m3 -> f32, fp32 row scales",
                     "mxfp8": "e4m3 x e4m3 -> f32, UE8M0 scales per 32",
                     "w4a8": "e2m1 x e4m3 -> f32, UE8M0 scales per 32"}[kind],
           "value": world * cfg.T * n / secs, "unit": UNIT, "ms_per_step": 1000.0 * secs / n,
           "steps": n, "stages_ms": stg, "clocks": clk.summary(), "roofline": roof}
    launches = wl.launches_per_step_q() * n
    wl.disable_quant()
    torch.cuda.empty_cache()
    return res, launches


def sustained_run(wl, warmup, torch, barrier, local, world, seconds=1.0):
    """The workload's forward repeated for about `seconds` (at least 3 steps)
    with nvidia-smi clock samples over the timed region: the sustained clock
    and power state of that step."""
    est = time_device(wl.forward, 3, warmup, torch, barrier) / 3
    n = max(3, int(seconds / max(est, 1e-6)))
    with ClockSampler(local) as clk:
        clk.mark_start()
        secs = time_device(wl.forward, n, 1, torch, barrier)
        clk.mark_end()
    return {"value": world * wl.cfg.T * n / secs, "unit": UNIT,
            "ms_per_step": 1000.0 * secs / n, "steps": n, "clocks": clk.summary()}


def roofline_of(wl, stages, counts, peaks, peak_src):
    """Roofline of the step's dominant kernel: the fused gate/up + down launch
    (small groups), else the gate/up launch.  Its bound follows the expert
    groups' arithmetic intensity: a touched expert's gate/up weights (2 I H
    bf16) serve its rows at 2 * 2 I H flops per row, i.e. `rows` flop per
    weight byte; at or above the ridge (measured sustained bf16 flop/s over
    the measured copy bandwidth) the kernel is tensor-bound, below it
    HBM-bound.  The other fraction is reported beside it."""
    cfg = wl.cfg
    alg_bytes, touched, inter = touched_bytes(cfg, counts, wl.fused)
    key = "expert_mlp_fused" if wl.fused else "gemm_gateup"
    t = stages[key] / 1000.0
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops_sustained"]
    flops = 2.0 * cfg.N * (3 if wl.fused else 2) * cfg.H * cfg.I
    rows = cfg.N / max(touched, 1)
    ridge = tc * 1e12 / (hbm * 1e9)
    gbs, tfs = alg_bytes / t / 1e9, flops / t / 1e12
    kname = ("grouped_gemm gate/up + SwiGLU + down, one launch (tcgen05)" if wl.fused
             else "grouped_gemm gate/up + SwiGLU (tcgen05)")
    hbm_part = {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "peak_source": f"{peak_src} hbm_gbs"}
    tc_part = {"achieved": tfs, "peak": tc, "unit": "TFLOP/s", "frac": tfs / tc,
               "peak_source": f"{peak_src} bf16_tflops_sustained"}
    tensor = rows >= ridge and not wl.fused
    main, other = (tc_part, hbm_part) if tensor else (hbm_part, tc_part)
    roof = {"kernel": kname, "bound": "tensor" if tensor else "hbm", **main,
            "traffic": profiled_traffic(key, cfg.name), "algorithmic_bytes": alg_bytes,
            "uncredited_intermediate_bytes": inter, "touched_experts": touched,
            "rows_per_touched_expert": rows, "ridge_rows": ridge,
            "other_bound": {"bound": "hbm" if tensor else "tensor", **other}}
    return roof, touched


def e2e_time(wl, steps, warmup, torch):
    import routed_mixture_experts_gemm_gb300 as gb
    c = wl.case
    cfg = wl.cfg
    x_h = c.x.cpu().pin_memory()
    ids_h = c.input_ids.cpu().pin_memory() if c.input_ids is not None else None
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    ws = c.layer.workspace(cfg.T, host=True)
    fn = lambda: gb.moe_forward_host(c.layer, x_h, input_ids_host=ids_h, out_host=out_h,  # noqa
                                     ws=ws, stream=wl.stream)
    t = time_device(fn, steps, warmup, torch)
    h2d = cfg.T * cfg.H * 2 + (cfg.T * 4 if ids_h is not None else 0)
    d2h = cfg.T * cfg.H * 2
    return t, h2d, d2h


# ------------------------------------------------------------ CPU oracle
def oracle_step(cfg, d, tokens, cache, nthreads):
    """The CPU oracle over a sample of tokens: routing, permutation, every
    touched expert's SwiGLU on its rows, combine.  Returns seconds of oracle
    time (expert weights are generated beforehand, outside the timing)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    pl = d["placement"]
    x = np.ascontiguousarray(d["x"][tokens])
    ids_in = d["input_ids"][tokens] if d["input_ids"] is not None else None
    t0 = time.perf_counter()
    lg = oracle.router_logits(x, d["w_router"], d["router_bias"], nthreads=nthreads)
    t_route = time.perf_counter() - t0
    # replica choice uses the token's batch position: route the sample with
    # its own positions (the sample is a prefix of the batch)
    ids, idp, w = oracle.route(oracle.cfg_from(cfg), lg, corr_bias=d["corr_bias"],
                               input_ids=ids_in, tid2eid=d["tid2eid"], log2phy=pl.log2phy,
                               replica_cnt=pl.replica_cnt)
    counts, offs, r2t, f2r = oracle.permute(idp, cfg.P)
    t_route = time.perf_counter() - t0
    need = [p for p in range(cfg.P) if counts[p] > 0]
    for p in need:
        e = int(pl.phys_to_log[p])
        if e not in cache:
            cache[e] = synth.expert_weights_host(cfg, e)
    y = np.empty((len(tokens) * cfg.k, cfg.H), np.uint16)

    def one(p):
        e = int(pl.phys_to_log[p])
        rows = np.arange(offs[p], offs[p + 1])
        a0 = time.perf_counter()
        _, yp = oracle.expert_ffn_rows(x[r2t[rows]], *cache[e], nthreads=1)
        y[rows] = yp
        return time.perf_counter() - a0

    t1 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=nthreads) as ex:
        list(ex.map(one, need))
    ys = None
    if cfg.shared_I:
        if "shared" not in cache:
            cache["shared"] = synth.shared_weights_host(cfg)
        _, ys = oracle.expert_ffn_rows(x, *cache["shared"], nthreads=nthreads)
    oracle.combine(y, f2r, w, ys)
    return t_route + (time.perf_counter() - t1)


def cpu_baseline(cfg, n_tokens, nthreads, reps=1, cache=None):
    d = synth.make_inputs(cfg)
    cache = {} if cache is None else cache
    tokens = np.arange(min(n_tokens, cfg.T))
    oracle_step(cfg, d, tokens, cache, nthreads)  # generates and caches weights, warms up
    secs = [oracle_step(cfg, d, tokens, cache, nthreads) for _ in range(reps)]
    sec = float(np.mean(secs))
    return {"value": len(tokens) / sec, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"first {len(tokens)} of the {cfg.T} tokens of the {cfg.name} workload "
                      f"(routing, permutation, every touched expert's SwiGLU, combine); "
                      f"tokens/s = sample tokens / oracle seconds, mean of {reps}",
            "seconds": sec}


# ------------------------------------------------------------ aggregation
def aggregate(times, tokens_per_rank, steps):
    """Whole-job throughput from per-rank elapsed seconds (max over ranks)."""
    t = max(times)
    return {"value": len(times) * tokens_per_rank * steps / t, "seconds": t,
            "ms_per_step": 1000.0 * t / steps}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--secondary", default="prefill,hash,skew",
                    help="comma-separated further workloads reported in the same line, each "
                         "under its own key ('' to skip); quantized experts are measured on "
                         "the first of them")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--sustained-s", type=float, default=1.0,
                    help="seconds of the sustained runs (decode companion, further workloads); "
                         "0 runs them for 3 steps (short launch lists under a profiler)")
    ap.add_argument("--cpu-tokens", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quant", action="store_true",
                    help="skip the quantized-expert measurements (FP8 rows, MXFP8, W4A8)")
    ap.add_argument("--quant", default=",".join(Workload.QUANT),
                    help="comma-separated quantized kinds to measure (fp8_row, mxfp8, w4a8)")
    args = ap.parse_args(argv)
    kinds = [k for k in args.quant.split(",") if k]
    if any(k not in Workload.QUANT for k in kinds):
        ap.error(f"--quant takes {', '.join(Workload.QUANT)}")
    world, rank, local = dist_setup()
    cfg = workload(args.workload)
    nthreads = os.cpu_count() or 1

    if args.impl == "reference":
        if rank != 0:
            return 0
        cache = {}
        d = synth.make_inputs(cfg)
        n = max(1, min(cfg.T, 4))
        tokens = np.arange(n)
        for _ in range(max(args.warmup, 1)):
            oracle_step(cfg, d, tokens, cache, nthreads)
        secs = sum(oracle_step(cfg, d, tokens, cache, nthreads) for _ in range(args.steps))
        value = n * args.steps / secs
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (CPU oracle)",
                "data": "synthetic (seeded generator)",
                "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E,
                           "I": cfg.I, "k": cfg.k},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads,
                                 "kind": "oracle",
                                 "sample": f"first {n} tokens of the {cfg.name} batch per step"},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        barrier = dist.barrier

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if barrier:
        barrier()
    __graft_entry__.build()

    wl = Workload(cfg, dev)
    wl.forward()
    torch.cuda.synchronize()
    import routed_mixture_experts_gemm_gb300 as gb
    st = gb.check_device_status()
    if st:
        raise RuntimeError(f"device status {st} after the first forward")

    with ClockSampler(local) as clk:
        clk.mark_start()
        secs = time_device(wl.forward, args.steps, args.warmup, torch, barrier)
        clk.mark_end()
    clocks = clk.summary()
    times = [secs]
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([secs], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        times = [float(t.item())] * world
    agg = aggregate(times, cfg.T, args.steps)

    stages = stage_times(wl, min(args.steps, 20), torch)
    counts = wl.counts.cpu().numpy()
    peaks, peak_src = load_peaks()
    roof, touched = roofline_of(wl, stages, counts, peaks, peak_src)
    # the same step repeated for >= 1 s: the sustained clock / power state
    sustained = sustained_run(wl, args.warmup, torch, barrier, local, world, args.sustained_s)
    t_e2e, h2d, d2h = e2e_time(wl, args.steps, args.warmup, torch)
    e2e = {"value": world * cfg.T * args.steps / t_e2e, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    line = {
        "metric": METRIC, "value": agg["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": agg["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator; random-init expert weights)",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "P": cfg.P,
                   "I": cfg.I, "k": cfg.k, "scoring": cfg.scoring, "n_group": cfg.n_group,
                   "topk_group": cfg.topk_group, "seed": cfg.seed,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (the step streams the touched experts' weights, "
                         f"{touched * 3 * cfg.I * cfg.H * 2 / 1e9:.1f} GB); no flush"},
        "roofline": roof, "stages_ms": stages, "e2e": e2e,
        "gpu_launches": wl.launches_per_step() * (args.steps + sustained["steps"]),
        "clocks": clocks, "sustained": sustained,
    }
    if not args.no_quant:
        line["quantized"] = {}
        for kind in kinds:
            r, nl = q_measure(wl, kind, args.steps, args.warmup, torch, barrier, peaks, peak_src,
                              world, "hbm", local)
            line["quantized"].setdefault(kind, {})[cfg.name] = r
            line["gpu_launches"] += nl
    del wl
    torch.cuda.empty_cache()

    for i, name2 in enumerate([w for w in args.secondary.split(",") if w]):
        c2 = workload(name2)
        w2 = Workload(c2, dev)
        w2.forward()
        torch.cuda.synchronize()
        res = sustained_run(w2, args.warmup, torch, barrier, local, world, args.sustained_s)
        res = {"workload": c2.name, "T": c2.T, **res}
        stg2 = stage_times(w2, min(args.steps, 10), torch)
        res["stages_ms"] = stg2
        if c2.use_hash and c2.scoring != "softmax":
            res["stages_note"] = ("route: the stand-alone moe_route call, which writes every "
                                  "logit; moe_forward (ms_per_step) computes only the logits "
                                  "of each token's hashed experts")
        res["layer_tflops"] = 2.0 * c2.N * 3 * c2.H * c2.I / (res["ms_per_step"] / 1e3) / 1e12
        res["roofline"], _ = roofline_of(w2, stg2, w2.counts.cpu().numpy(), peaks, peak_src)
        line[c2.name] = res
        line["gpu_launches"] += w2.launches_per_step() * res["steps"]
        if i == 0 and not args.no_quant:
            for kind in kinds:
                r, nl = q_measure(w2, kind, min(args.steps, 20), args.warmup, torch, barrier,
                                  peaks, peak_src, world, "tensor", local)
                line.setdefault("quantized", {}).setdefault(kind, {})[c2.name] = r
                line["gpu_launches"] += nl
        del w2
        torch.cuda.empty_cache()

    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_tokens, nthreads)
        line["cpu_baseline"].pop("seconds", None)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
