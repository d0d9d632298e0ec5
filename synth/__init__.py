"""Seeded synthetic inputs for the routed-MoE workloads.

This module holds no MoE arithmetic.  It defines the workloads (sizes,
routing features and value distributions of the five configurations the
layer is benchmarked on, plus small "mini" twins used for full parity
checks) and turns (seed, tensor, index) into numbers with the counter-based
generator written out in ``synth/gen.c``.  Two bit-identical implementations
of that generator exist:

* the host one (``gen.c`` through ctypes), which the CPU oracle's inputs come
  from, for whole tensors or for any slice of one (one expert's weights);
* a torch restatement (:func:`normal_bf16_device`) used to fill the multi-GB
  expert weight tensors directly in GPU memory, where host generation and
  upload would dominate run time.

Distributions (all seeded, synthetic):
  x ~ N(0, 1) bf16; expert W_gate/W_up [I, H] and W_down [H, I] ~ N(0, 0.02)
  bf16; router weight fp32 ~ N(0, 0.02) (N(0, 1/H) for the prefill shape,
  whose router logits are meant to be ~N(0, 1)); correction bias fp32
  ~ N(0, 0.1); token ids uniform in [0, V); a token-id -> expert table with k
  distinct experts per row; a Zipf(s) router (logit) bias over a seeded rank
  permutation, with the hottest experts replicated onto extra physical slots.
"N(0, s)" is realised as an Irwin-Hall sum of four uniforms scaled to mean 0
and standard deviation s (bounded at about 3.5 s, otherwise close to normal).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

# tensor tags (part of the generator's key)
TAG_X, TAG_WR, TAG_CB, TAG_WG, TAG_WU, TAG_WD = 1, 2, 3, 4, 5, 6
TAG_IDS, TAG_TID, TAG_ZIPF, TAG_SLOT = 7, 8, 9, 10
TAG_WGS, TAG_WUS, TAG_WDS = 11, 12, 13

# std of 2*(sum of four uniforms on {0..65535}) - 262140
_IH4_STD = 2.0 * math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)
_M32 = 0xFFFFFFFF


def normal_scale(sigma: float) -> np.float32:
    """fp32 multiplier that maps the centred Irwin-Hall integer to N(0, sigma)."""
    return np.float32(sigma / _IH4_STD)


# --------------------------------------------------------------------------
# host generator (C)
# --------------------------------------------------------------------------
_lib = None
_lib_lock = threading.Lock()


def build_host_lib(force: bool = False) -> str:
    """Compile gen.c into libsynth.so next to it (plain C, no arch flags)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                           "-shared", "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build_host_lib())
            u32, i32, i64, f32 = ctypes.c_uint32, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            vp = ctypes.c_void_p
            lib.synth_key.argtypes = [u32, u32, u32]
            lib.synth_key.restype = u32
            lib.synth_draw.argtypes = [u32, u32]
            lib.synth_draw.restype = u32
            lib.synth_normal_f32.argtypes = [u32, u32, u32, f32, vp]
            lib.synth_normal_bf16.argtypes = [u32, u32, u32, f32, vp]
            lib.synth_uniform_i32.argtypes = [u32, u32, u32, u32, vp]
            lib.synth_permutation.argtypes = [u32, i32, vp]
            lib.synth_distinct_rows.argtypes = [u32, u32, i64, i64, i32, i32, vp, vp]
            for f in ("synth_normal_f32", "synth_normal_bf16", "synth_uniform_i32",
                      "synth_permutation", "synth_distinct_rows"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def key(seed: int, tag: int, slab: int = 0) -> int:
    return int(_L().synth_key(seed & _M32, tag & _M32, slab & _M32))


def _chunked(n: int, fn, chunk: int = 1 << 22):
    """Run fn(start, count) over [0, n) in chunks on a few threads
    (ctypes releases the GIL during the C call)."""
    if n <= chunk:
        fn(0, n)
        return
    starts = list(range(0, n, chunk))
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(lambda s: fn(s, min(chunk, n - s)), starts))


def normal_f32(seed: int, tag: int, slab: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    k = key(seed, tag, slab)
    sc = float(normal_scale(sigma))
    base = out.ctypes.data
    _chunked(n, lambda s, c: _L().synth_normal_f32(k, s, c, sc, base + 4 * s))
    return out


def normal_bf16(seed: int, tag: int, slab: int, n: int, sigma: float) -> np.ndarray:
    """bf16 values as raw uint16 bits."""
    out = np.empty(n, dtype=np.uint16)
    k = key(seed, tag, slab)
    sc = float(normal_scale(sigma))
    base = out.ctypes.data
    _chunked(n, lambda s, c: _L().synth_normal_bf16(k, s, c, sc, base + 2 * s))
    return out


def uniform_i32(seed: int, tag: int, slab: int, n: int, upper: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _L().synth_uniform_i32(key(seed, tag, slab), 0, n, upper, out.ctypes.data)
    return out


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _L().synth_permutation(key(seed, tag, 0), n, out.ctypes.data)
    return out


def distinct_rows(seed: int, tag: int, nrows: int, E: int, k: int) -> np.ndarray:
    out = np.empty((nrows, k), dtype=np.int32)
    scratch = np.empty(E, dtype=np.int32)
    _L().synth_distinct_rows(seed, tag, 0, nrows, E, k, scratch.ctypes.data, out.ctypes.data)
    return out


# --------------------------------------------------------------------------
# device generator (torch restatement of the same definition)
# --------------------------------------------------------------------------
def _mul32_t(h, c: int):
    # (h * c) mod 2^32 for 0 <= h < 2^32 without leaving int64 range
    lo, hi = c & 0xFFFF, c >> 16
    return (h * lo + (((h * hi) & 0xFFFF) << 16)) & _M32


def _fmix32_t(h):
    h = h ^ (h >> 16)
    h = _mul32_t(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32_t(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def _draw_t(k: int, i):
    return _fmix32_t(_fmix32_t((i + 0x61C88647) & _M32) ^ k)


def normal_bf16_device(seed: int, tag: int, slab: int, n: int, sigma: float, device,
                       out=None):
    """The same values as :func:`normal_bf16`, generated with torch on ``device``
    (bfloat16 tensor of n elements, written into ``out`` when given)."""
    import torch
    k = key(seed, tag, slab)
    sc = torch.tensor(float(normal_scale(sigma)), dtype=torch.float32, device=device)
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=device)
    step = 1 << 23
    for s0 in range(0, n, step):
        c = min(step, n - s0)
        idx = torch.arange(s0, s0 + c, dtype=torch.int64, device=device) * 2
        a = _draw_t(k, idx)
        b = _draw_t(k, idx + 1)
        s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16)
        v = (2 * s - 262140).to(torch.float32) * sc
        out[s0:s0 + c] = v.to(torch.bfloat16)
        del idx, a, b, s, v
    return out


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class MoEConfig:
    name: str
    seed: int
    T: int          # tokens
    H: int          # hidden
    I: int          # expert intermediate
    E: int          # logical experts
    k: int          # top-k
    scoring: str    # "softmax" | "sigmoid" | "sqrtsoftplus"
    n_group: int = 1
    topk_group: int = 1
    group_score: str = "auto"      # "max" | "top2sum" | "auto"
    renormalize: bool = True
    routed_scaling: float = 1.0
    corr_bias_sigma: float = 0.0   # > 0: a selection-only correction bias
    router_sigma: Optional[float] = 0.02   # None: 1/sqrt(H)
    hash_vocab: int = 0            # > 0: hash routing through a [V, k] table
    zipf_s: float = 0.0            # > 0: Zipf(s) router (logit) bias
    n_hot_replicas: int = 0        # hottest logical experts given a 2nd slot
    shared_I: int = 0              # > 0: always-on shared SwiGLU expert
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    note: str = ""

    @property
    def P(self) -> int:
        return self.E + self.n_hot_replicas

    @property
    def N(self) -> int:
        return self.T * self.k

    @property
    def group_score_mode(self) -> str:
        if self.group_score != "auto":
            return self.group_score
        return "top2sum" if self.corr_bias_sigma > 0 else "max"

    @property
    def use_hash(self) -> bool:
        return self.hash_vocab > 0

    def with_T(self, T: int) -> "MoEConfig":
        return replace(self, T=T)


CONFIGS = {
    "tiny": MoEConfig("tiny", 0, T=64, H=256, I=128, E=8, k=2, scoring="softmax",
                      routed_scaling=1.0),
    "decode": MoEConfig("decode", 1, T=128, H=7168, I=2048, E=256, k=8,
                        scoring="sigmoid", n_group=8, topk_group=4,
                        routed_scaling=2.5, corr_bias_sigma=0.1),
    "prefill": MoEConfig("prefill", 2, T=8192, H=7168, I=2048, E=256, k=8,
                         scoring="sigmoid", n_group=8, topk_group=4,
                         routed_scaling=2.5, corr_bias_sigma=0.1, router_sigma=None),
    "hash": MoEConfig("hash", 3, T=2048, H=7168, I=2048, E=384, k=8,
                      scoring="sqrtsoftplus", routed_scaling=2.5, hash_vocab=163840),
    "skew": MoEConfig("skew", 4, T=4096, H=7168, I=2048, E=256, k=8, scoring="sigmoid",
                      routed_scaling=2.5, zipf_s=1.1, n_hot_replicas=32, shared_I=2048),
}

# Small twins with the same routing features, small enough for a full
# element-by-element oracle comparison, sized to span several GEMM tiles and
# leave ragged tails (T not a multiple of anything, experts with > 128 rows).
MINI = {
    "tiny": CONFIGS["tiny"],
    "mini_decode": MoEConfig("mini_decode", 11, T=100, H=384, I=256, E=32, k=8,
                             scoring="sigmoid", n_group=8, topk_group=4,
                             routed_scaling=2.5, corr_bias_sigma=0.1),
    "mini_prefill": MoEConfig("mini_prefill", 12, T=520, H=256, I=256, E=16, k=4,
                              scoring="sigmoid", n_group=4, topk_group=2,
                              routed_scaling=2.5, corr_bias_sigma=0.1, router_sigma=None),
    "mini_hash": MoEConfig("mini_hash", 13, T=77, H=256, I=128, E=48, k=8,
                           scoring="sqrtsoftplus", routed_scaling=2.5, hash_vocab=1000),
    "mini_skew": MoEConfig("mini_skew", 14, T=130, H=256, I=128, E=32, k=8,
                           scoring="sigmoid", routed_scaling=2.5, zipf_s=1.1,
                           n_hot_replicas=8, shared_I=128),
}


def router_sigma(cfg: MoEConfig) -> float:
    return cfg.router_sigma if cfg.router_sigma is not None else 1.0 / math.sqrt(cfg.H)


@dataclass
class Placement:
    """Logical -> physical expert placement (identity unless replicated)."""
    log2phy: Optional[np.ndarray]      # int32 [E, R_max] or None (identity)
    replica_cnt: Optional[np.ndarray]  # int32 [E] or None
    phys_to_log: np.ndarray            # int32 [P]
    R_max: int


def placement(cfg: MoEConfig) -> Placement:
    if cfg.n_hot_replicas == 0:
        return Placement(None, None, np.arange(cfg.E, dtype=np.int32), 1)
    rank = permutation(cfg.seed, TAG_ZIPF, cfg.E) + 1          # Zipf rank of expert e
    hot = sorted(int(e) for e in np.nonzero(rank <= cfg.n_hot_replicas)[0])
    entries = [(e, 0) for e in range(cfg.E)] + [(e, 1) for e in hot]
    slot = permutation(cfg.seed, TAG_SLOT, len(entries))
    R = 2
    l2p = np.full((cfg.E, R), -1, dtype=np.int32)
    cnt = np.ones(cfg.E, dtype=np.int32)
    p2l = np.empty(len(entries), dtype=np.int32)
    for i, (e, r) in enumerate(entries):
        l2p[e, r] = slot[i]
        p2l[slot[i]] = e
    for e in hot:
        cnt[e] = 2
    l2p[:, 1] = np.where(cnt == 2, l2p[:, 1], l2p[:, 0])  # unused column mirrors col 0
    return Placement(l2p, cnt, p2l, R)


def zipf_router_bias(cfg: MoEConfig) -> Optional[np.ndarray]:
    """Additive router-logit bias b_e = ln p_{r(e)} - mean ln p, p_r ~ r^-s."""
    if cfg.zipf_s <= 0:
        return None
    rank = (permutation(cfg.seed, TAG_ZIPF, cfg.E) + 1).astype(np.float64)
    lp = -cfg.zipf_s * np.log(rank)
    return (lp - lp.mean()).astype(np.float32)


def make_inputs(cfg: MoEConfig) -> dict:
    """Everything except the expert weights, generated on the host."""
    d = {"cfg": cfg}
    d["x"] = normal_bf16(cfg.seed, TAG_X, 0, cfg.T * cfg.H, cfg.x_sigma).reshape(cfg.T, cfg.H)
    d["w_router"] = normal_f32(cfg.seed, TAG_WR, 0, cfg.E * cfg.H,
                               router_sigma(cfg)).reshape(cfg.E, cfg.H)
    d["corr_bias"] = (normal_f32(cfg.seed, TAG_CB, 0, cfg.E, cfg.corr_bias_sigma)
                      if cfg.corr_bias_sigma > 0 else None)
    d["router_bias"] = zipf_router_bias(cfg)
    if cfg.use_hash:
        d["input_ids"] = uniform_i32(cfg.seed, TAG_IDS, 0, cfg.T, cfg.hash_vocab)
        d["tid2eid"] = distinct_rows(cfg.seed, TAG_TID, cfg.hash_vocab, cfg.E, cfg.k)
    else:
        d["input_ids"] = None
        d["tid2eid"] = None
    d["placement"] = placement(cfg)
    return d


def expert_weights_host(cfg: MoEConfig, e: int):
    """(W_gate [I,H], W_up [I,H], W_down [H,I]) of logical expert e, bf16 bits."""
    n = cfg.I * cfg.H
    wg = normal_bf16(cfg.seed, TAG_WG, e, n, cfg.w_sigma).reshape(cfg.I, cfg.H)
    wu = normal_bf16(cfg.seed, TAG_WU, e, n, cfg.w_sigma).reshape(cfg.I, cfg.H)
    wd = normal_bf16(cfg.seed, TAG_WD, e, n, cfg.w_sigma).reshape(cfg.H, cfg.I)
    return wg, wu, wd


def shared_weights_host(cfg: MoEConfig):
    if cfg.shared_I == 0:
        return None
    n = cfg.shared_I * cfg.H
    wg = normal_bf16(cfg.seed, TAG_WGS, 0, n, cfg.w_sigma).reshape(cfg.shared_I, cfg.H)
    wu = normal_bf16(cfg.seed, TAG_WUS, 0, n, cfg.w_sigma).reshape(cfg.shared_I, cfg.H)
    wd = normal_bf16(cfg.seed, TAG_WDS, 0, n, cfg.w_sigma).reshape(cfg.H, cfg.shared_I)
    return wg, wu, wd


def all_expert_weights_host(cfg: MoEConfig):
    """Physical-slot weight stacks [P,I,H], [P,I,H], [P,H,I] (small configs)."""
    pl = placement(cfg)
    per = [expert_weights_host(cfg, e) for e in range(cfg.E)]
    wg = np.stack([per[pl.phys_to_log[p]][0] for p in range(cfg.P)])
    wu = np.stack([per[pl.phys_to_log[p]][1] for p in range(cfg.P)])
    wd = np.stack([per[pl.phys_to_log[p]][2] for p in range(cfg.P)])
    return wg, wu, wd


def expert_weights_device(cfg: MoEConfig, device):
    """Physical-slot weight stacks generated directly on ``device`` (bf16):
    W_gate/W_up [P, I, H], W_down [P, H, I]; replicas are byte copies."""
    import torch
    pl = placement(cfg)
    P, I, H = cfg.P, cfg.I, cfg.H
    wg = torch.empty((P, I, H), dtype=torch.bfloat16, device=device)
    wu = torch.empty((P, I, H), dtype=torch.bfloat16, device=device)
    wd = torch.empty((P, H, I), dtype=torch.bfloat16, device=device)
    first_slot = {}
    for p in range(P):
        e = int(pl.phys_to_log[p])
        if e in first_slot:
            q = first_slot[e]
            wg[p].copy_(wg[q]); wu[p].copy_(wu[q]); wd[p].copy_(wd[q])
            continue
        first_slot[e] = p
        normal_bf16_device(cfg.seed, TAG_WG, e, I * H, cfg.w_sigma, device, out=wg[p].view(-1))
        normal_bf16_device(cfg.seed, TAG_WU, e, I * H, cfg.w_sigma, device, out=wu[p].view(-1))
        normal_bf16_device(cfg.seed, TAG_WD, e, I * H, cfg.w_sigma, device, out=wd[p].view(-1))
    return wg, wu, wd


def shared_weights_device(cfg: MoEConfig, device):
    import torch
    if cfg.shared_I == 0:
        return None
    Is, H = cfg.shared_I, cfg.H
    wg = torch.empty((Is, H), dtype=torch.bfloat16, device=device)
    wu = torch.empty((Is, H), dtype=torch.bfloat16, device=device)
    wd = torch.empty((H, Is), dtype=torch.bfloat16, device=device)
    normal_bf16_device(cfg.seed, TAG_WGS, 0, Is * H, cfg.w_sigma, device, out=wg.view(-1))
    normal_bf16_device(cfg.seed, TAG_WUS, 0, Is * H, cfg.w_sigma, device, out=wu.view(-1))
    normal_bf16_device(cfg.seed, TAG_WDS, 0, Is * H, cfg.w_sigma, device, out=wd.view(-1))
    return wg, wu, wd


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
