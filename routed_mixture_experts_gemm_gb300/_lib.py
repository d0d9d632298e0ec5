"""ctypes declarations of libgbmoe.so (the C ABI in include/gbmoe.h)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbmoe.so")

GBMOE_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA",
                5: "DEVICE", 6: "TIMEOUT"}
SCORE = {"softmax": 0, "sigmoid": 1, "sqrtsoftplus": 2}
GROUP = {"max": 0, "top2sum": 1}
ACT_SWIGLU = 0
ACTIVATION = {"swiglu": 0, "swiglu_oai": 1, "geglu": 2, "geglu_tanh": 3}
MX_FORMAT = {"e4m3": 0, "e2m1": 1}

# every function the header declares, with (restype, argtypes)
_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class RouteCfg(ctypes.Structure):
    _fields_ = [("E_log", _i), ("E_phys", _i), ("top_k", _i), ("n_group", _i),
                ("topk_group", _i), ("scoring", _i), ("group_score", _i), ("renormalize", _i),
                ("routed_scaling", _f), ("use_hash", _i)]


class Layer(ctypes.Structure):
    _fields_ = [("route", RouteCfg), ("H", _i), ("I", _i), ("I_shared", _i),
                ("w_router", _vp), ("router_bias", _vp), ("corr_bias", _vp),
                ("tid2eid", _vp), ("tid2eid_rows", _i64), ("log2phy", _vp),
                ("replica_cnt", _vp), ("R_max", _i), ("w_gate", _vp), ("w_up", _vp),
                ("w_down", _vp), ("w_gate_shared", _vp), ("w_up_shared", _vp),
                ("w_down_shared", _vp), ("activation", _i), ("w_gate_q", _vp), ("s_gate", _vp),
                ("w_up_q", _vp), ("s_up", _vp), ("w_down_q", _vp), ("s_down", _vp),
                ("mx_format", _i), ("w_gate_mx", _vp), ("sf_gate", _vp), ("w_up_mx", _vp),
                ("sf_up", _vp), ("w_down_mx", _vp), ("sf_down", _vp)]


_P = ctypes.POINTER
SIGNATURES = {
    "gbmoe_status_string": (ctypes.c_char_p, [_i]),
    "gbmoe_validate_route_cfg": (_i, [_P(RouteCfg)]),
    "gbmoe_validate_log2phy": (_i, [_vp, _vp, _i, _i, _i]),
    "gbmoe_check_device_status": (_i, [_vp, _P(_i)]),
    "gbmoe_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "moe_route": (_i, [_P(RouteCfg), _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp,
                       _i, _vp, _vp, _vp, _vp, _vp]),
    "moe_expert_counts": (_i, [_vp, _i, _i, _i, _vp, _i, _vp]),
    "gbmoe_permute_workspace_size": (_sz, [_i, _i, _i]),
    "moe_permute": (_i, [_vp, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_permute_static": (_i, [_vp, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_gemm_gateup_act": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp]),
    "moe_gemm_gateup_act_rows": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _i, _vp,
                                      _vp]),
    "moe_gemm_down": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "moe_expert_mlp": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _vp,
                            _vp, _vp]),
    "gbmoe_expert_mlp_fused": (_i, [_i, _i, _i]),
    "moe_combine": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "moe_quantize_fp8_rows": (_i, [_vp, _i64, _i, _vp, _vp, _vp]),
    "moe_gemm_gateup_act_fp8": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                                     _i, _vp, _vp]),
    "moe_gemm_down_fp8": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "moe_quantize_mx_rows": (_i, [_vp, _i64, _i, _i, _vp, _vp, _vp]),
    "moe_mx_tile_scales": (_i, [_vp, _i64, _i, _vp, _vp]),
    "moe_gemm_gateup_act_mx": (_i, [_vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp,
                                    _vp, _i, _vp, _vp, _vp]),
    "moe_gemm_down_mx": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "gbmoe_latent_tail_workspace_size": (_sz, [_i, _i, _i]),
    "moe_latent_tail": (_i, [_vp, _i, _i, _vp, ctypes.c_float, _vp, _i, _vp, _vp, _vp, _sz,
                             _vp]),
    "gbmoe_forward_workspace_size": (_sz, [_P(Layer), _i]),
    "moe_forward": (_i, [_P(Layer), _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "gbmoe_forward_host_workspace_size": (_sz, [_P(Layer), _i]),
    "moe_forward_host": (_i, [_P(Layer), _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libgbmoe.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m routed_mixture_experts_gemm_gb300.build` "
            "(there is no CPU or Python fallback for the routed-MoE kernels)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
