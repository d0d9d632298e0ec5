"""Routed mixture-of-experts layer forward on GB300 (sm_103a).

Thin Python binding over libgbmoe.so (C ABI: include/gbmoe.h).  Every step
of the layer runs in the library's CUDA kernels; this module only marshals
arguments (torch tensors for device memory and streams) and raises on a
non-zero status.  There is no CPU or Python fallback: without the built
library every call raises.

Functions carry the C names: moe_route, moe_permute, moe_gemm_gateup_act,
moe_gemm_down, moe_expert_mlp, moe_combine, moe_expert_counts, moe_forward,
moe_forward_host.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import ACTIVATION, ACT_SWIGLU, GROUP, MX_FORMAT, SCORE, Layer, RouteCfg

__all__ = ["GbmoeError", "route_cfg", "moe_route", "moe_expert_counts", "moe_permute",
           "moe_gemm_gateup_act", "moe_gemm_gateup_act_rows", "moe_gemm_down", "moe_expert_mlp", "expert_mlp_fused",
           "moe_combine", "moe_quantize_fp8_rows",
           "moe_gemm_gateup_act_fp8", "moe_gemm_down_fp8", "quantize_experts_fp8",
           "moe_quantize_mx_rows", "moe_mx_tile_scales", "moe_gemm_gateup_act_mx",
           "moe_gemm_down_mx",
           "quantize_experts_mx", "moe_latent_tail", "MoELayer", "moe_forward",
           "moe_forward_host", "check_device_status", "set_wait_limit_ns", "library"]


class GbmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.load().gbmoe_status_string(status).decode()
        super().__init__(f"{what}: {_lib.STATUS_NAMES.get(status, status)} ({msg})")


def library():
    return _lib.load()


def _check(st: int, what: str):
    if st != 0:
        raise GbmoeError(st, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def route_cfg(E_log: int, top_k: int, scoring="softmax", E_phys: Optional[int] = None,
              n_group: int = 1, topk_group: int = 1, group_score="max", renormalize=True,
              routed_scaling: float = 1.0, use_hash=False) -> RouteCfg:
    return RouteCfg(E_log, E_log if E_phys is None else E_phys, top_k, n_group, topk_group,
                    SCORE[scoring] if isinstance(scoring, str) else scoring,
                    GROUP[group_score] if isinstance(group_score, str) else group_score,
                    int(bool(renormalize)), float(routed_scaling), int(bool(use_hash)))


def moe_route(cfg: RouteCfg, x=None, w_router=None, logits=None, router_bias=None,
              corr_bias=None, input_ids=None, tid2eid=None, log2phy=None, replica_cnt=None,
              with_counts=True, stream=None) -> dict:
    """Router scoring + selection + log2phy.  Give w_router (and x) to compute
    the logits, or logits [T, E_log] to score caller-provided logits."""
    lib = _lib.load()
    if w_router is not None:
        T, H = x.shape
        dev = x.device
        logits = torch.empty((T, cfg.E_log), dtype=torch.float32, device=dev)
    else:
        T, H = logits.shape[0], 0
        dev = logits.device
    k = cfg.top_k
    out = {
        "logits": logits,
        "ids_log": torch.empty((T, k), dtype=torch.int32, device=dev),
        "ids_phys": torch.empty((T, k), dtype=torch.int32, device=dev),
        "weights": torch.empty((T, k), dtype=torch.float32, device=dev),
        "counts": torch.empty(cfg.E_phys, dtype=torch.int32, device=dev) if with_counts else None,
    }
    R = 1 if log2phy is None else log2phy.shape[1]
    rows = 0 if tid2eid is None else tid2eid.shape[0]
    st = lib.moe_route(ctypes.byref(cfg), _ptr(x) if w_router is not None else None, T, H,
                       _ptr(w_router), _ptr(logits), _ptr(router_bias), _ptr(corr_bias),
                       _ptr(input_ids), _ptr(tid2eid), rows, _ptr(log2phy), _ptr(replica_cnt), R,
                       _ptr(out["ids_log"]), _ptr(out["ids_phys"]), _ptr(out["weights"]),
                       _ptr(out["counts"]), _stream(stream))
    _check(st, "moe_route")
    return out


def moe_expert_counts(ids_phys, E_phys: int, counts=None, accumulate=False, stream=None):
    lib = _lib.load()
    T, k = ids_phys.shape
    if counts is None:
        counts = torch.empty(E_phys, dtype=torch.int32, device=ids_phys.device)
        accumulate = False
    _check(lib.moe_expert_counts(_ptr(ids_phys), T, k, E_phys, _ptr(counts), int(accumulate),
                                 _stream(stream)), "moe_expert_counts")
    return counts


def moe_permute(ids_phys, E_phys: int, x=None, ws=None, stream=None) -> dict:
    lib = _lib.load()
    T, k = ids_phys.shape
    dev = ids_phys.device
    N = T * k
    o = {
        "counts": torch.empty(E_phys, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E_phys + 1, dtype=torch.int32, device=dev),
        "row_to_token": torch.empty(N, dtype=torch.int32, device=dev),
        "flat_to_row": torch.empty(N, dtype=torch.int32, device=dev),
        "x_perm": None if x is None else torch.empty((N, x.shape[1]), dtype=x.dtype, device=dev),
    }
    need = lib.gbmoe_permute_workspace_size(T, k, E_phys)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(lib.moe_permute(_ptr(ids_phys), T, k, E_phys, _ptr(x), 0 if x is None else x.shape[1],
                           _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["row_to_token"]),
                           _ptr(o["flat_to_row"]), _ptr(o["x_perm"]), _ptr(ws), ws.numel(),
                           _stream(stream)), "moe_permute")
    return o


def _act(activation) -> int:
    return ACTIVATION[activation] if isinstance(activation, str) else int(activation)


def moe_gemm_gateup_act(x_perm, offsets, w_gate, w_up, act=None, stream=None,
                        activation="swiglu"):
    """act = bf16(f(x W_gate^T, x W_up^T)) per expert group, f the gated
    activation ("swiglu", "swiglu_oai", "geglu", "geglu_tanh"); offsets None =
    one group."""
    lib = _lib.load()
    N, H = x_perm.shape
    P, I, _ = w_gate.shape
    if act is None:
        act = torch.empty((N, I), dtype=torch.bfloat16, device=x_perm.device)
    _check(lib.moe_gemm_gateup_act(_ptr(x_perm), _ptr(offsets), P, N, H, I, _ptr(w_gate),
                                   _ptr(w_up), _act(activation), _ptr(act), _stream(stream)),
           "moe_gemm_gateup_act")
    return act


def moe_gemm_gateup_act_rows(x, row_to_token, offsets, w_gate, w_up, act=None, stream=None,
                             activation="swiglu"):
    """moe_gemm_gateup_act with row r of the operand gathered as x[row_to_token[r]]."""
    lib = _lib.load()
    T, H = x.shape
    N = row_to_token.shape[0]
    P, I, _ = w_gate.shape
    if act is None:
        act = torch.empty((N, I), dtype=torch.bfloat16, device=x.device)
    _check(lib.moe_gemm_gateup_act_rows(_ptr(x), _ptr(row_to_token), T, _ptr(offsets), P, N, H,
                                        I, _ptr(w_gate), _ptr(w_up), _act(activation), _ptr(act),
                                        _stream(stream)), "moe_gemm_gateup_act_rows")
    return act


def moe_gemm_down(act, offsets, w_down, y=None, stream=None):
    """y = act W_down^T per expert group, fp32 output [N, H]."""
    lib = _lib.load()
    N, I = act.shape
    P, H, _ = w_down.shape
    if y is None:
        y = torch.empty((N, H), dtype=torch.float32, device=act.device)
    _check(lib.moe_gemm_down(_ptr(act), _ptr(offsets), P, N, H, I, _ptr(w_down), _ptr(y),
                             _stream(stream)), "moe_gemm_down")
    return y


def moe_expert_mlp(x_rows, offsets, w_gate, w_up, w_down, act=None, y=None, ready=None,
                   row_to_token=None, stream=None, activation="swiglu"):
    """Both grouped GEMMs (gate/up + SwiGLU, then down) as moe_forward runs them;
    returns (act, y).  x_rows is x_perm [N, H], or with row_to_token [N] the
    unpermuted x [T, H] whose rows the GEMM gathers.  `ready` ([E_phys] int32
    scratch) enables the fused launch."""
    lib = _lib.load()
    P, I, H = w_gate.shape
    if row_to_token is None:
        N, T = x_rows.shape[0], 0
    else:
        N, T = row_to_token.shape[0], x_rows.shape[0]
    dev = x_rows.device
    if act is None:
        act = torch.empty((N, I), dtype=torch.bfloat16, device=dev)
    if y is None:
        y = torch.empty((N, H), dtype=torch.float32, device=dev)
    _check(lib.moe_expert_mlp(_ptr(x_rows), _ptr(row_to_token), T, _ptr(offsets), P, N, H, I,
                              _ptr(w_gate), _ptr(w_up), _ptr(w_down), _act(activation),
                              _ptr(act), _ptr(y), _ptr(ready), _stream(stream)),
           "moe_expert_mlp")
    return act, y


def expert_mlp_fused(E_phys: int, N: int, H: int) -> bool:
    """Whether moe_expert_mlp / moe_forward fuse the two GEMMs for this shape."""
    return bool(_lib.load().gbmoe_expert_mlp_fused(E_phys, N, H))


def moe_combine(y, flat_to_row, weights, shared_y=None, out=None, stream=None):
    """out = bf16(sum_j w_j y[flat_to_row] + shared_y); y, shared_y fp32."""
    lib = _lib.load()
    T, k = weights.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    _check(lib.moe_combine(_ptr(y), _ptr(flat_to_row), _ptr(weights), _ptr(shared_y), T, k, H,
                           _ptr(out), _stream(stream)), "moe_combine")
    return out


def moe_quantize_fp8_rows(x, q=None, scales=None, stream=None):
    """bf16 rows [n, K] -> (E4M3 codes uint8 [n, K], fp32 scales [n]), s = amax / 448."""
    lib = _lib.load()
    n, K = x.shape
    if q is None:
        q = torch.empty((n, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(n, dtype=torch.float32, device=x.device)
    _check(lib.moe_quantize_fp8_rows(_ptr(x), n, K, _ptr(q), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8_rows")
    return q, scales


def moe_gemm_gateup_act_fp8(xq, sx, offsets, wgq, sg, wuq, su, row_to_token=None, act=None,
                            activation="swiglu", stream=None):
    """FP8 gate/up GEMM: act = bf16(f((xq wgq^T) sx sg, (xq wuq^T) sx su)); xq [T, H]
    codes gathered through row_to_token [N] (or the N permuted rows)."""
    lib = _lib.load()
    P, I, H = wgq.shape
    if row_to_token is None:
        N, T = xq.shape[0], 0
    else:
        N, T = row_to_token.shape[0], xq.shape[0]
    if act is None:
        act = torch.empty((N, I), dtype=torch.bfloat16, device=xq.device)
    _check(lib.moe_gemm_gateup_act_fp8(_ptr(xq), _ptr(sx), _ptr(row_to_token), T, _ptr(offsets),
                                       P, N, H, I, _ptr(wgq), _ptr(sg), _ptr(wuq), _ptr(su),
                                       _act(activation), _ptr(act), _stream(stream)),
           "moe_gemm_gateup_act_fp8")
    return act


def moe_gemm_down_fp8(aq, sa, offsets, wdq, sd, y=None, stream=None):
    """FP8 down GEMM: y = (aq wdq^T) sa sd in fp32 [N, H]."""
    lib = _lib.load()
    N, I = aq.shape
    P, H, _ = wdq.shape
    if y is None:
        y = torch.empty((N, H), dtype=torch.float32, device=aq.device)
    _check(lib.moe_gemm_down_fp8(_ptr(aq), _ptr(sa), _ptr(offsets), P, N, H, I, _ptr(wdq),
                                 _ptr(sd), _ptr(y), _stream(stream)), "moe_gemm_down_fp8")
    return y


def quantize_experts_fp8(w, stream=None):
    """bf16 expert weights [E, R, K] -> (E4M3 codes uint8 [E, R, K], fp32 per-row
    scales [E, R]) with moe_quantize_fp8_rows."""
    E, R, K = w.shape
    q, sc = moe_quantize_fp8_rows(w.reshape(E * R, K), stream=stream)
    return q.reshape(E, R, K), sc.reshape(E, R)


def _mx(fmt) -> int:
    return MX_FORMAT[fmt] if isinstance(fmt, str) else int(fmt)


def moe_quantize_mx_rows(x, fmt="e4m3", q=None, scales=None, stream=None):
    """bf16 rows [n, K] -> MX codes (uint8 [n, K] for E4M3, [n, K/2] packed E2M1)
    and UE8M0 block-scale bytes uint8 [n, K/32] (blocks of 32 along K)."""
    lib = _lib.load()
    n, K = x.shape
    f = _mx(fmt)
    if q is None:
        q = torch.empty((n, K // 2 if f == MX_FORMAT["e2m1"] else K), dtype=torch.uint8,
                        device=x.device)
    if scales is None:
        scales = torch.empty((n, K // 32), dtype=torch.uint8, device=x.device)
    _check(lib.moe_quantize_mx_rows(_ptr(x), n, K, f, _ptr(q), _ptr(scales), _stream(stream)),
           "moe_quantize_mx_rows")
    return q, scales


def quantize_experts_mx(w, fmt="e4m3", stream=None):
    """bf16 expert weights [E, R, K] -> (MX codes [E, R, K or K/2], scale bytes
    [E, R, K/32]) with moe_quantize_mx_rows."""
    E, R, K = w.shape
    q, sc = moe_quantize_mx_rows(w.reshape(E * R, K), fmt, stream=stream)
    return q.reshape(E, R, -1), sc.reshape(E, R, K // 32)


def moe_mx_tile_scales(sf, stream=None):
    """MX weight scale bytes [..., R, K/32] (row-major, as moe_quantize_mx_rows
    writes them) -> the same bytes in the tiled layout the MX GEMMs read
    (moe_mx_tile_scales of the C ABI), as a new tensor of the same shape."""
    lib = _lib.load()
    K = sf.shape[-1] * 32
    rows = sf.numel() // (K // 32)
    out = torch.empty_like(sf)
    _check(lib.moe_mx_tile_scales(_ptr(sf), rows, K, _ptr(out), _stream(stream)),
           "moe_mx_tile_scales")
    return out


def moe_gemm_gateup_act_mx(xq, xs, offsets, wgq, sg, wuq, su, w_fmt="e4m3", row_to_token=None,
                           act_q=None, act_s=None, activation="swiglu", stream=None,
                           scales_tiled=False):
    """MX gate/up GEMM: act = bf16(f(x wg^T, x wu^T)) over the dequantized MX
    operands, returned quantized to MX E4M3: (codes uint8 [N, I], scale bytes
    [N, I/32]).  xq [T, H] codes + xs [T, H/32] gathered through row_to_token
    [N] (or the N permuted rows); weights in format w_fmt with row-major
    scale bytes sg / su (tiled here by moe_mx_tile_scales), or already tiled
    with scales_tiled=True."""
    lib = _lib.load()
    if not scales_tiled:
        sg, su = moe_mx_tile_scales(sg, stream), moe_mx_tile_scales(su, stream)
    P, I = wgq.shape[0], wgq.shape[1]
    H = xq.shape[1]
    if row_to_token is None:
        N, T = xq.shape[0], 0
    else:
        N, T = row_to_token.shape[0], xq.shape[0]
    if act_q is None:
        act_q = torch.empty((N, I), dtype=torch.uint8, device=xq.device)
    if act_s is None:
        act_s = torch.empty((N, I // 32), dtype=torch.uint8, device=xq.device)
    _check(lib.moe_gemm_gateup_act_mx(_ptr(xq), _ptr(xs), _ptr(row_to_token), T, _ptr(offsets),
                                      P, N, H, I, _mx(w_fmt), _ptr(wgq), _ptr(sg), _ptr(wuq),
                                      _ptr(su), _act(activation), _ptr(act_q), _ptr(act_s),
                                      _stream(stream)), "moe_gemm_gateup_act_mx")
    return act_q, act_s


def moe_gemm_down_mx(aq, as_, offsets, wdq, sd, w_fmt="e4m3", y=None, stream=None,
                     scales_tiled=False):
    """MX down GEMM: y = a . wd^T over the dequantized MX operands, fp32 [N, H];
    sd row-major (tiled here) or tiled with scales_tiled=True."""
    lib = _lib.load()
    if not scales_tiled:
        sd = moe_mx_tile_scales(sd, stream)
    N, I = aq.shape
    P, H = wdq.shape[0], wdq.shape[1]
    if y is None:
        y = torch.empty((N, H), dtype=torch.float32, device=aq.device)
    _check(lib.moe_gemm_down_mx(_ptr(aq), _ptr(as_), _ptr(offsets), P, N, H, I, _mx(w_fmt),
                                _ptr(wdq), _ptr(sd), _ptr(y), _stream(stream)),
           "moe_gemm_down_mx")
    return y


def moe_latent_tail(latent, up_proj, norm_w=None, eps=1e-6, shared=None, out=None, ws=None,
                    stream=None):
    """out = bf16(rmsnorm(latent) . up_proj^T + shared): the latent-MoE tail on
    one GPU.  latent [T, L], up_proj [Hm, L], norm_w [L] or None, shared
    [T, Hm] or None (bf16 device tensors)."""
    lib = _lib.load()
    T, L = latent.shape
    Hm = up_proj.shape[0]
    if out is None:
        out = torch.empty((T, Hm), dtype=torch.bfloat16, device=latent.device)
    need = lib.gbmoe_latent_tail_workspace_size(T, L, Hm)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=latent.device)
    _check(lib.moe_latent_tail(_ptr(latent), T, L, _ptr(norm_w), float(eps), _ptr(up_proj), Hm,
                               _ptr(shared), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_latent_tail")
    return out


class MoELayer:
    """A layer's routing settings and device weights, as the C struct moe_forward takes.

    Weights are torch tensors on the device: w_router fp32 [E_log, H];
    w_gate / w_up bf16 [E_phys, I, H]; w_down bf16 [E_phys, H, I]; optional
    router_bias / corr_bias fp32 [E_log], tid2eid int32 [V, top_k],
    log2phy int32 [E_log, R_max] + replica_cnt int32 [E_log], shared expert
    (w_gate_shared, w_up_shared [I_s, H], w_down_shared [H, I_s]).
    """

    def __init__(self, cfg: RouteCfg, w_router, w_gate, w_up, w_down, router_bias=None,
                 corr_bias=None, tid2eid=None, log2phy=None, replica_cnt=None, shared=None,
                 activation="swiglu", fp8=None, mx=None):
        """fp8 = (w_gate_q, s_gate, w_up_q, s_up, w_down_q, s_down): FP8 routed
        experts (E4M3 codes uint8 [E_phys, I, H] / [E_phys, H, I] and fp32
        per-row scales, e.g. from quantize_experts_fp8); the bf16 w_gate / w_up /
        w_down may then be None.
        mx = (fmt, w_gate_mx, sf_gate, w_up_mx, sf_up, w_down_mx, sf_down): MX
        block-scaled routed experts ("e4m3" or "e2m1" codes and UE8M0 scale
        bytes per 32 elements along K, row-major as from quantize_experts_mx;
        the layer keeps copies in the GEMMs' tiled layout)."""
        self.cfg = cfg
        if mx:
            mx = [mx[0], mx[1], moe_mx_tile_scales(mx[2]), mx[3], moe_mx_tile_scales(mx[4]),
                  mx[5], moe_mx_tile_scales(mx[6])]
        self._keep = [w_router, w_gate, w_up, w_down, router_bias, corr_bias, tid2eid, log2phy,
                      replica_cnt] + list(shared or []) + list(fp8 or []) + list(mx or [])[1:]
        if w_gate is not None:
            (P, I, H), ref = w_gate.shape, w_gate
        elif fp8 is not None:
            (P, I, H), ref = fp8[0].shape, fp8[0]
        else:  # MX: H from the scale bytes (the codes of E2M1 hold H/2 bytes)
            (P, I), H, ref = mx[1].shape[:2], mx[2].shape[2] * 32, mx[1]
        Is = 0 if shared is None else shared[0].shape[0]
        self.H, self.I, self.I_shared = H, I, Is
        self.device = ref.device
        s = shared or (None, None, None)
        self.c = Layer(cfg, H, I, Is, _ptr(w_router), _ptr(router_bias), _ptr(corr_bias),
                       _ptr(tid2eid), 0 if tid2eid is None else tid2eid.shape[0], _ptr(log2phy),
                       _ptr(replica_cnt), 1 if log2phy is None else log2phy.shape[1],
                       _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(s[0]), _ptr(s[1]),
                       _ptr(s[2]), _act(activation), *[_ptr(a) for a in (fp8 or [None] * 6)],
                       _mx(mx[0]) if mx else 0, *[_ptr(a) for a in (mx[1:] if mx else [None] * 6)])
        self._ws = None

    def workspace_size(self, T_max: int, host: bool = False) -> int:
        lib = _lib.load()
        fn = lib.gbmoe_forward_host_workspace_size if host else lib.gbmoe_forward_workspace_size
        n = fn(ctypes.byref(self.c), T_max)
        if n == 0 and T_max > 0:
            raise GbmoeError(1, "gbmoe_forward_workspace_size")
        return n

    def workspace(self, T_max: int, host: bool = False):
        need = self.workspace_size(T_max, host)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 1), dtype=torch.uint8, device=self.device)
        return self._ws


def moe_forward(layer: MoELayer, x, input_ids=None, out=None, ids_log=None, ids_phys=None,
                weights=None, counts=None, ws=None, stream=None):
    lib = _lib.load()
    T = x.shape[0]
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = layer.workspace(T)
    _check(lib.moe_forward(ctypes.byref(layer.c), _ptr(x), T, _ptr(input_ids), _ptr(out),
                           _ptr(ids_log), _ptr(ids_phys), _ptr(weights), _ptr(counts), _ptr(ws),
                           ws.numel(), _stream(stream)), "moe_forward")
    return out


def moe_forward_host(layer: MoELayer, x_host, input_ids_host=None, out_host=None,
                     ids_log_host=None, ws=None, stream=None):
    """Host (ideally pinned) x in, host out; copies are enqueued on the stream.
    Synchronise the stream before reading out_host."""
    lib = _lib.load()
    T = x_host.shape[0]
    if out_host is None:
        out_host = torch.empty((T, layer.H), dtype=torch.bfloat16, pin_memory=True)
    if ws is None:
        ws = layer.workspace(T, host=True)
    _check(lib.moe_forward_host(ctypes.byref(layer.c), _ptr(x_host), T, _ptr(input_ids_host),
                                _ptr(out_host), _ptr(ids_log_host), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_forward_host")
    return out_host


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the grouped GEMMs' bounded waits for launches made from now
    on (0: the default, 4 s); returns the previous limit."""
    return int(_lib.load().gbmoe_set_wait_limit_ns(int(ns)))


def check_device_status(stream=None) -> int:
    """Synchronise and return (then clear) the device-side error status."""
    lib = _lib.load()
    st = ctypes.c_int(0)
    _check(lib.gbmoe_check_device_status(_stream(stream), ctypes.byref(st)),
           "gbmoe_check_device_status")
    return st.value
