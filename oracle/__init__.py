"""CPU oracle for the routed mixture-of-experts layer forward (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The GPU library never
imports, links or calls anything here, and nothing here imports the GPU
library.  The arithmetic lives in ``oracle.c`` (plain C, fp32 with pinned
order for routing, double-accumulated dot products for the expert MLP);
this file only marshals numpy arrays.

Each function cites the passage of the vLLM-Ascend "Kimi K3 MoE Forward
Insight" page it follows; the readings of what the page leaves open are
listed at the top of ``oracle.c``.

Pins: every function here is pinned by a CPU test against something other
than itself (closed forms, brute force, library routines, invariants); see
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

SOFTMAX, SIGMOID, SQRTSOFTPLUS = 0, 1, 2
GROUP_MAX, GROUP_TOP2SUM = 0, 1
_SCORING = {"softmax": SOFTMAX, "sigmoid": SIGMOID, "sqrtsoftplus": SQRTSOFTPLUS}
_GROUP = {"max": GROUP_MAX, "top2sum": GROUP_TOP2SUM}
# gated activations of the expert MLP (reading R15)
ACTIVATIONS = {"swiglu": 0, "swiglu_oai": 1, "geglu": 2, "geglu_tanh": 3}


def _act(a) -> int:
    return ACTIVATIONS[a] if isinstance(a, str) else int(a)


class RouteCfg(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("P", ctypes.c_int), ("k", ctypes.c_int),
                ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("scoring", ctypes.c_int), ("group_score", ctypes.c_int),
                ("renormalize", ctypes.c_int), ("routed_scaling", ctypes.c_float),
                ("use_hash", ctypes.c_int)]


def route_cfg(E, k, scoring="softmax", P=None, n_group=1, topk_group=1, group_score="max",
              renormalize=True, routed_scaling=1.0, use_hash=False) -> RouteCfg:
    if isinstance(scoring, str):
        scoring = _SCORING[scoring]
    if isinstance(group_score, str):
        group_score = _GROUP[group_score]
    if not (1 <= k <= E) or n_group < 1 or E % n_group or not (1 <= topk_group <= n_group):
        raise ValueError("bad routing configuration")
    if n_group > 1 and topk_group * (E // n_group) < k:
        raise ValueError("topk_group groups hold fewer than k experts")
    return RouteCfg(E, E if P is None else P, k, n_group, topk_group, scoring, group_score,
                    int(bool(renormalize)), float(routed_scaling), int(bool(use_hash)))


def cfg_from(mcfg) -> RouteCfg:
    """RouteCfg of a synth.MoEConfig."""
    return route_cfg(mcfg.E, mcfg.k, mcfg.scoring, P=mcfg.P, n_group=mcfg.n_group,
                     topk_group=mcfg.topk_group, group_score=mcfg.group_score_mode,
                     renormalize=mcfg.renormalize, routed_scaling=mcfg.routed_scaling,
                     use_hash=mcfg.use_hash)


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c (plain C11; -ffp-contract=off keeps a*b+c as two roundings)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f, vp, i, i64 = ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            for name in ("orc_exp", "orc_log1p", "orc_sigmoid", "orc_sqrtsoftplus"):
                getattr(lib, name).argtypes = [f]
                getattr(lib, name).restype = f
            lib.orc_f32_to_bf16.argtypes = [f]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_router_logit.argtypes = [vp, vp, i]
            lib.orc_router_logit.restype = f
            lib.oracle_router_logits.argtypes = [vp, i, i, vp, i, vp, vp, i]
            lib.oracle_router_logits.restype = None
            lib.orc_scores.argtypes = [vp, i, i, vp]
            lib.orc_scores.restype = None
            lib.oracle_route.argtypes = [ctypes.POINTER(RouteCfg), vp, i, vp, vp, vp, i64, vp, vp,
                                         i, vp, vp, vp]
            lib.oracle_route.restype = i
            lib.oracle_expert_counts.argtypes = [vp, i, i, i, vp, i]
            lib.oracle_expert_counts.restype = None
            lib.oracle_permute.argtypes = [vp, i, i, i, vp, vp, vp, vp]
            lib.oracle_permute.restype = None
            lib.orc_act_value.argtypes = [i, ctypes.c_double, ctypes.c_double]
            lib.orc_act_value.restype = ctypes.c_double
            lib.oracle_expert_ffn_rows.argtypes = [vp, i64, i, i, vp, vp, vp, i, vp, vp, i]
            lib.oracle_expert_ffn_rows.restype = None
            lib.oracle_ffn_grouped.argtypes = [vp, vp, vp, i, i, i, vp, vp, vp, i, vp, vp, i]
            lib.oracle_ffn_grouped.restype = None
            lib.oracle_combine.argtypes = [vp, vp, vp, vp, i, i, i, vp]
            lib.oracle_combine.restype = None
            lib.oracle_moe_forward.argtypes = (
                [ctypes.POINTER(RouteCfg), vp, i, i, i, vp, vp, vp, vp, vp, vp, i64, vp, vp, i,
                 vp, vp, vp, i, i, vp, vp, vp] + [vp] * 12 + [i])
            lib.oracle_moe_forward.restype = i
            lib.orc_f32_to_e4m3.argtypes = [f]
            lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
            lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f32.restype = f
            lib.oracle_quantize_rows.argtypes = [vp, i64, i, vp, vp]
            lib.oracle_quantize_rows.restype = None
            lib.oracle_ffn_grouped_fp8.argtypes = [vp, vp, vp, vp, i, i, i, vp, vp, vp, vp, vp,
                                                   vp, i, vp, vp, i]
            lib.oracle_ffn_grouped_fp8.restype = None
            lib.orc_f32_to_e2m1.argtypes = [f]
            lib.orc_f32_to_e2m1.restype = ctypes.c_uint8
            lib.orc_e2m1_to_f32.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_to_f32.restype = f
            lib.orc_mx_block_exp.argtypes = [f, i]
            lib.orc_mx_block_exp.restype = i
            lib.oracle_mx_quantize_rows.argtypes = [vp, i64, i, i, vp, vp]
            lib.oracle_mx_quantize_rows.restype = None
            lib.oracle_ffn_grouped_mx.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, vp, vp, vp, vp,
                                                  vp, i, vp, vp, vp, vp, i]
            lib.oracle_ffn_grouped_mx.restype = None
            lib.oracle_rmsnorm_row.argtypes = [vp, i, vp, f, vp]
            lib.oracle_rmsnorm_row.restype = None
            lib.oracle_latent_tail.argtypes = [vp, i, i, vp, f, vp, i, vp, vp, i]
            lib.oracle_latent_tail.restype = None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --- elementary functions (Stage 2 scoring; pinned definitions in oracle.c) ---
def exp(x: float) -> float:
    return _L().orc_exp(x)


def log1p(y: float) -> float:
    return _L().orc_log1p(y)


def sigmoid(x: float) -> float:
    return _L().orc_sigmoid(x)


def sqrtsoftplus(x: float) -> float:
    return _L().orc_sqrtsoftplus(x)


def f32_to_bf16(x: float) -> int:
    return int(_L().orc_f32_to_bf16(x))


# --- routing (Runner Initialization + Stage 2: Select Experts) ---
def router_logits(x_bits, w_router, router_bias=None, nthreads=None) -> np.ndarray:
    """fp32 logits [T, E] in the pinned summation order (reading R1)."""
    x_bits = _c(x_bits, np.uint16)
    w_router = _c(w_router, np.float32)
    T, H = x_bits.shape
    E = w_router.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    rb = _c(router_bias, np.float32)
    _L().oracle_router_logits(_p(x_bits), T, H, _p(w_router), E, _p(rb), _p(out),
                              nthreads or default_threads())
    return out


def scores(logits_row, scoring) -> np.ndarray:
    l = _c(logits_row, np.float32)
    out = np.empty_like(l)
    _L().orc_scores(_p(l), l.shape[0], _SCORING.get(scoring, scoring), _p(out))
    return out


def route(cfg: RouteCfg, logits, corr_bias=None, input_ids=None, tid2eid=None,
          log2phy=None, replica_cnt=None):
    """(ids_log, ids_phys, weights) for logits [T, E] (Stage 2 + Stage 4 step 2)."""
    logits = _c(logits, np.float32)
    T = logits.shape[0]
    ids_log = np.empty((T, cfg.k), dtype=np.int32)
    ids_phys = np.empty((T, cfg.k), dtype=np.int32)
    w = np.empty((T, cfg.k), dtype=np.float32)
    cb = _c(corr_bias, np.float32)
    ii = _c(input_ids, np.int32)
    tt = _c(tid2eid, np.int32)
    lp = _c(log2phy, np.int32)
    rc_ = _c(replica_cnt, np.int32)
    V = 0 if tt is None else tt.shape[0]
    R = 1 if lp is None else lp.shape[1]
    rc = _L().oracle_route(ctypes.byref(cfg), _p(logits), T, _p(cb), _p(ii), _p(tt), V, _p(lp),
                           _p(rc_), R, _p(ids_log), _p(ids_phys), _p(w))
    if rc:
        raise ValueError(f"oracle_route rejected its input (code {rc})")
    return ids_log, ids_phys, w


# --- dispatch / load tracking (Stage 4 AllGather row, Stage 6) ---
def expert_counts(ids_phys, P, counts=None):
    ids = _c(ids_phys, np.int32)
    T, k = ids.shape
    acc = counts is not None
    if counts is None:
        counts = np.zeros(P, dtype=np.int32)
    _L().oracle_expert_counts(_p(ids), T, k, P, _p(counts), int(acc))
    return counts


def permute(ids_phys, P):
    """(counts [P], offsets [P+1], row_to_token [N], flat_to_row [N]) (reading R9)."""
    ids = _c(ids_phys, np.int32)
    T, k = ids.shape
    counts = np.empty(P, dtype=np.int32)
    offsets = np.empty(P + 1, dtype=np.int32)
    r2t = np.empty(T * k, dtype=np.int32)
    f2r = np.empty(T * k, dtype=np.int32)
    _L().oracle_permute(_p(ids), T, k, P, _p(counts), _p(offsets), _p(r2t), _p(f2r))
    return counts, offsets, r2t, f2r


# --- expert MLP (Stage 4: grouped gate/up -> activation -> grouped down) ---
def act_value(activation, g, u) -> float:
    """The gated activation of one (g, u) pair in double (reading R15)."""
    return _L().orc_act_value(_act(activation), float(g), float(u))


def expert_ffn_rows(x_rows, wg, wu, wd, nthreads=None, activation="swiglu"):
    """act [n, I] (bf16 bits) and y [n, H] (fp32) of rows through one gated expert."""
    x_rows = _c(x_rows, np.uint16)
    n, H = x_rows.shape
    I = wg.shape[0]
    act = np.empty((n, I), dtype=np.uint16)
    y = np.empty((n, H), dtype=np.float32)
    _L().oracle_expert_ffn_rows(_p(x_rows), n, H, I, _p(_c(wg, np.uint16)), _p(_c(wu, np.uint16)),
                                _p(_c(wd, np.uint16)), _act(activation), _p(act), _p(y),
                                nthreads or default_threads())
    return act, y


def ffn_grouped(x, row_to_token, offsets, wg, wu, wd, nthreads=None, activation="swiglu"):
    x = _c(x, np.uint16)
    P, I, H = wg.shape
    N = int(offsets[P])
    act = np.empty((N, I), dtype=np.uint16)
    y = np.empty((N, H), dtype=np.float32)
    _L().oracle_ffn_grouped(_p(x), _p(_c(row_to_token, np.int32)), _p(_c(offsets, np.int32)), P, H,
                            I, _p(_c(wg, np.uint16)), _p(_c(wu, np.uint16)),
                            _p(_c(wd, np.uint16)), _act(activation), _p(act), _p(y),
                            nthreads or default_threads())
    return act, y


def combine(y, flat_to_row, weights, ys=None):
    """out [T, H] bf16 bits from fp32 y [T*k, H] (and fp32 ys [T, H])
    (Stage 4 AllGather combine: restore token order, apply the probabilities)."""
    y = _c(y, np.float32)
    w = _c(weights, np.float32)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.uint16)
    _L().oracle_combine(_p(y), _p(_c(flat_to_row, np.int32)), _p(w), _p(_c(ys, np.float32)), T, k,
                        H, _p(out))
    return out


def moe_forward(cfg: RouteCfg, x, H, I, w_router=None, logits=None, router_bias=None,
                corr_bias=None, input_ids=None, tid2eid=None, log2phy=None, replica_cnt=None,
                wg=None, wu=None, wd=None, shared=None, nthreads=None,
                activation="swiglu") -> dict:
    """The whole layer, stage by stage; returns every intermediate."""
    x = _c(x, np.uint16)
    T = x.shape[0]
    k, P, E = cfg.k, cfg.P, cfg.E
    N = T * k
    lg = np.empty((T, E), dtype=np.float32) if logits is None else _c(logits, np.float32)
    o = {
        "logits": lg,
        "ids_log": np.empty((T, k), np.int32), "ids_phys": np.empty((T, k), np.int32),
        "weights": np.empty((T, k), np.float32), "counts": np.empty(P, np.int32),
        "offsets": np.empty(P + 1, np.int32), "row_to_token": np.empty(N, np.int32),
        "flat_to_row": np.empty(N, np.int32), "act": np.empty((N, I), np.uint16),
        "y": np.empty((N, H), np.float32), "out": np.empty((T, H), np.uint16),
    }
    Is = 0
    sg = su = sd = None
    if shared is not None:
        sg, su, sd = (_c(a, np.uint16) for a in shared)
        Is = sg.shape[0]
        o["act_s"] = np.empty((T, Is), np.uint16)
        o["ys"] = np.empty((T, H), np.float32)
    tt = _c(tid2eid, np.int32)
    lp = _c(log2phy, np.int32)
    rc = _L().oracle_moe_forward(
        ctypes.byref(cfg), _p(x), T, H, I, _p(_c(w_router, np.float32)),
        _p(_c(router_bias, np.float32)), _p(lg), _p(_c(corr_bias, np.float32)),
        _p(_c(input_ids, np.int32)), _p(tt), 0 if tt is None else tt.shape[0], _p(lp),
        _p(_c(replica_cnt, np.int32)), 1 if lp is None else lp.shape[1],
        _p(_c(wg, np.uint16)), _p(_c(wu, np.uint16)), _p(_c(wd, np.uint16)), _act(activation),
        Is, _p(sg), _p(su),
        _p(sd), _p(o["ids_log"]), _p(o["ids_phys"]), _p(o["weights"]), _p(o["counts"]),
        _p(o["offsets"]), _p(o["row_to_token"]), _p(o["flat_to_row"]), _p(o["act"]), _p(o["y"]),
        _p(o.get("act_s")), _p(o.get("ys")), _p(o["out"]), nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle_moe_forward rejected its input (code {rc})")
    return o


def run_config(mcfg, inputs=None, weights=None, nthreads=None, activation="swiglu") -> dict:
    """Oracle forward of a synth.MoEConfig from its seeded inputs."""
    import synth
    d = inputs if inputs is not None else synth.make_inputs(mcfg)
    if weights is None:
        weights = synth.all_expert_weights_host(mcfg)
    pl = d["placement"]
    return moe_forward(cfg_from(mcfg), d["x"], mcfg.H, mcfg.I, w_router=d["w_router"],
                       router_bias=d["router_bias"], corr_bias=d["corr_bias"],
                       input_ids=d["input_ids"], tid2eid=d["tid2eid"], log2phy=pl.log2phy,
                       replica_cnt=pl.replica_cnt, wg=weights[0], wu=weights[1], wd=weights[2],
                       shared=synth.shared_weights_host(mcfg), nthreads=nthreads,
                       activation=activation)


# --- latent MoE tail (LatentMoERunner page, tier 1 with one rank; reading R16) ---
def rmsnorm_row(v_bits, w_bits, eps: float) -> np.ndarray:
    """bf16 RMSNorm of one row in the pinned fp32 order (reading R16)."""
    v = _c(v_bits, np.uint16)
    z = np.empty_like(v)
    _L().oracle_rmsnorm_row(_p(v), v.shape[0], _p(_c(w_bits, np.uint16)), float(eps), _p(z))
    return z


def latent_tail(latent, up_proj, norm_w=None, eps: float = 1e-6, shared=None,
                nthreads=None) -> np.ndarray:
    """out [T, Hm] = bf16(rmsnorm(latent) . up_proj^T + shared) (bf16 bits in and out)."""
    latent = _c(latent, np.uint16)
    up = _c(up_proj, np.uint16)
    T, L = latent.shape
    Hm = up.shape[0]
    out = np.empty((T, Hm), dtype=np.uint16)
    _L().oracle_latent_tail(_p(latent), T, L, _p(_c(norm_w, np.uint16)), float(eps), _p(up), Hm,
                            _p(_c(shared, np.uint16)), _p(out), nthreads or default_threads())
    return out


# --- FP8 experts (Stage 4 quantized paths, W8A8FP; reading R17) ---
def f32_to_e4m3(x: float) -> int:
    """OCP FP8 E4M3 code of an fp32 value: round to nearest even, saturate to +-448."""
    return int(_L().orc_f32_to_e4m3(float(x)))


def e4m3_to_f32(code: int) -> float:
    return float(_L().orc_e4m3_to_f32(int(code)))


def quantize_rows(x_bits):
    """bf16 rows [n, K] -> (E4M3 codes uint8 [n, K], fp32 scales [n]), s = amax / 448."""
    x = _c(x_bits, np.uint16)
    n, K = x.shape
    q = np.empty((n, K), dtype=np.uint8)
    sc = np.empty(n, dtype=np.float32)
    _L().oracle_quantize_rows(_p(x), n, K, _p(q), _p(sc))
    return q, sc


def ffn_grouped_fp8(xq, sx, row_to_token, offsets, wg, sg, wu, su, wd, sd, nthreads=None,
                    activation="swiglu"):
    """FP8 grouped expert MLP: act [N, I] bf16 bits, y [N, H] fp32 (reading R17)."""
    xq = _c(xq, np.uint8)
    P, I, H = wg.shape
    N = int(offsets[P])
    act = np.empty((N, I), dtype=np.uint16)
    y = np.empty((N, H), dtype=np.float32)
    _L().oracle_ffn_grouped_fp8(_p(xq), _p(_c(sx, np.float32)), _p(_c(row_to_token, np.int32)),
                                _p(_c(offsets, np.int32)), P, H, I, _p(_c(wg, np.uint8)),
                                _p(_c(sg, np.float32)), _p(_c(wu, np.uint8)),
                                _p(_c(su, np.float32)), _p(_c(wd, np.uint8)),
                                _p(_c(sd, np.float32)), _act(activation), _p(act), _p(y),
                                nthreads or default_threads())
    return act, y


# --- MX block-scaled experts (Stage 4 quantized paths, MXFP and W4A8; reading R18) ---
MX_FORMATS = {"e4m3": 0, "e2m1": 1}
MX_BLOCK = 32


def f32_to_e2m1(x: float) -> int:
    """FP4 E2M1 code (sign bit 3) of an fp32 value: nearest, ties to even, saturate to +-6."""
    return int(_L().orc_f32_to_e2m1(float(x)))


def e2m1_to_f32(code: int) -> float:
    return float(_L().orc_e2m1_to_f32(int(code)))


def mx_block_exp(amax: float, fmt: str) -> int:
    """Shared exponent e of an MX block (scale 2^e) with largest magnitude amax."""
    return int(_L().orc_mx_block_exp(float(amax), MX_FORMATS[fmt]))


def mx_quantize_rows(x_bits, fmt="e4m3"):
    """bf16 rows [n, K] -> (codes uint8 [n, K] for E4M3 or [n, K/2] packed E2M1,
    UE8M0 block-scale bytes uint8 [n, K/32])."""
    x = _c(x_bits, np.uint16)
    n, K = x.shape
    q = np.empty((n, K // 2 if fmt == "e2m1" else K), dtype=np.uint8)
    sc = np.empty((n, K // MX_BLOCK), dtype=np.uint8)
    _L().oracle_mx_quantize_rows(_p(x), n, K, MX_FORMATS[fmt], _p(q), _p(sc))
    return q, sc


def ffn_grouped_mx(xq, xs, row_to_token, offsets, wg, sg, wu, su, wd, sd, wfmt="e4m3",
                   nthreads=None, activation="swiglu"):
    """MX grouped expert MLP (reading R18): x as MX E4M3 codes [T, H] + scales
    [T, H/32]; weights as MX codes in format wfmt with their block scales.
    Returns act bf16 bits [N, I], its MX E4M3 codes [N, I] and scales [N, I/32],
    and y fp32 [N, H]."""
    xq = _c(xq, np.uint8)
    P, I = wg.shape[0], wg.shape[1]
    H = xq.shape[1]
    N = int(offsets[P])
    act = np.empty((N, I), dtype=np.uint16)
    aq = np.empty((N, I), dtype=np.uint8)
    as_ = np.empty((N, I // MX_BLOCK), dtype=np.uint8)
    y = np.empty((N, H), dtype=np.float32)
    u8 = lambda a: _p(_c(a, np.uint8))  # noqa: E731
    _L().oracle_ffn_grouped_mx(_p(xq), u8(xs), _p(_c(row_to_token, np.int32)),
                               _p(_c(offsets, np.int32)), P, H, I, MX_FORMATS[wfmt], u8(wg),
                               u8(sg), u8(wu), u8(su), u8(wd), u8(sd), _act(activation),
                               _p(act), _p(aq), _p(as_), _p(y), nthreads or default_threads())
    return act, aq, as_, y
