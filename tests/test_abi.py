"""The C-ABI library loads, exports every function include/gbmoe.h declares,
and rejects bad arguments on the host before any device work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbmoe.h")


@pytest.fixture(scope="module")
def lib():
    from routed_mixture_experts_gemm_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^(?:const\s+)?(?:int|size_t|uint64_t|char\s*\*|const char\s*\*)\s*\**\s*(\w+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("moe_route", "moe_permute", "moe_gemm_gateup_act", "moe_gemm_down",
                 "moe_combine", "moe_forward", "moe_expert_counts", "moe_forward_host",
                 "gbmoe_status_string", "gbmoe_check_device_status"):
        assert want in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(lib):
    from routed_mixture_experts_gemm_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # and the binding declares a signature for each of them
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert lib.gbmoe_status_string(0) == b"ok"
    assert b"invalid" in lib.gbmoe_status_string(1)
    assert lib.gbmoe_status_string(99) == b"unknown status"


def _cfg(**kw):
    from routed_mixture_experts_gemm_gb300 import route_cfg
    base = dict(E_log=32, top_k=8, scoring="sigmoid", n_group=8, topk_group=4,
                group_score="top2sum", routed_scaling=2.5)
    base.update(kw)
    return route_cfg(**base)


@pytest.mark.parametrize("bad", [dict(top_k=40), dict(top_k=0), dict(n_group=5),
                                 dict(topk_group=1), dict(topk_group=9), dict(E_log=2000),
                                 dict(E_phys=16), dict(scoring=7), dict(group_score=3),
                                 dict(use_hash=True)])
def test_route_cfg_validation(lib, bad):
    assert lib.gbmoe_validate_route_cfg(ctypes.byref(_cfg())) == 0
    assert lib.gbmoe_validate_route_cfg(ctypes.byref(_cfg(**bad))) == 1


def test_entry_points_reject_bad_arguments_on_host(lib):
    c = _cfg(top_k=40)
    fake = ctypes.c_void_p(0x1000)
    # bad configuration: rejected before any CUDA call
    assert lib.moe_route(ctypes.byref(c), fake, 4, 256, fake, fake, None, None, None, None, 0,
                         None, None, 1, fake, fake, fake, None, None) == 1
    c = _cfg()
    # logits / outputs missing
    assert lib.moe_route(ctypes.byref(c), fake, 4, 256, fake, None, None, None, None, None, 0,
                         None, None, 1, fake, fake, fake, None, None) == 1
    # unsupported GEMM shapes (H, I must be multiples of 128)
    assert lib.moe_gemm_gateup_act(fake, fake, 8, 64, 200, 128, fake, fake, 0, fake, None) == 2
    assert lib.moe_gemm_down(fake, fake, 8, 64, 256, 100, fake, fake, None) == 2
    assert lib.moe_gemm_gateup_act(fake, fake, 8, 64, 256, 128, fake, fake, 5, fake, None) == 2
    # multiple groups without offsets
    assert lib.moe_gemm_down(fake, None, 8, 64, 256, 128, fake, fake, None) == 1
    # combine: k beyond the supported maximum, H not a multiple of 8
    assert lib.moe_combine(fake, fake, fake, None, 4, 33, 256, fake, None) == 1
    assert lib.moe_combine(fake, fake, fake, None, 4, 2, 250, fake, None) == 1
    # permute without workspace
    assert lib.moe_permute(fake, 4, 2, 8, None, 0, fake, fake, fake, fake, None, None, 0,
                           None) == 3
    # T = 0 is a no-op that needs no device
    assert lib.moe_combine(None, None, None, None, 0, 2, 256, None, None) == 0


def test_workspace_sizes_grow_with_capacity(lib):
    from routed_mixture_experts_gemm_gb300 import _lib
    c = _cfg()
    L = _lib.Layer(c, 256, 128, 0, 0x1000, None, None, None, 0, None, None, 1, 0x1000, 0x1000,
                   0x1000, None, None, None)
    a = lib.gbmoe_forward_workspace_size(ctypes.byref(L), 64)
    b = lib.gbmoe_forward_workspace_size(ctypes.byref(L), 128)
    assert 0 < a < b
    assert lib.gbmoe_forward_host_workspace_size(ctypes.byref(L), 64) > a
    assert lib.gbmoe_permute_workspace_size(100, 8, 32) > 0


def test_log2phy_validation(lib):
    E, R, P = 4, 2, 6
    l2p = np.array([[0, 4], [1, 1], [2, 5], [3, 3]], np.int32)
    cnt = np.array([2, 1, 2, 1], np.int32)
    ok = lib.gbmoe_validate_log2phy(l2p.ctypes.data, cnt.ctypes.data, E, R, P)
    assert ok == 0
    bad = l2p.copy()
    bad[2, 1] = 4  # slot shared by two logical experts
    assert lib.gbmoe_validate_log2phy(bad.ctypes.data, cnt.ctypes.data, E, R, P) == 1
    bad = l2p.copy()
    bad[0, 1] = 6  # out of range
    assert lib.gbmoe_validate_log2phy(bad.ctypes.data, cnt.ctypes.data, E, R, P) == 1
    c0 = cnt.copy()
    c0[1] = 0      # a logical expert left unplaced
    assert lib.gbmoe_validate_log2phy(l2p.ctypes.data, c0.ctypes.data, E, R, P) == 1


def test_quantized_entry_points_reject_bad_arguments_on_host(lib):
    fake, odd4, odd16 = (ctypes.c_void_p(a) for a in (0x1000, 0x1004, 0x1010))
    # FP8 rows: K a multiple of 8, H % 256 for the GEMMs, known activations
    assert lib.moe_quantize_fp8_rows(fake, 4, 100, fake, fake, None) == 2
    assert lib.moe_gemm_gateup_act_fp8(fake, fake, fake, 8, fake, 4, 16, 384, 128, fake, fake,
                                       fake, fake, 0, fake, None) == 2
    assert lib.moe_gemm_gateup_act_fp8(fake, fake, fake, 8, fake, 4, 16, 512, 128, fake, fake,
                                       fake, fake, 9, fake, None) == 2
    assert lib.moe_gemm_down_fp8(fake, fake, fake, 4, 16, 512, 100, fake, fake, fake, None) == 2
    # MX quantizer: unknown format, K % 32, misaligned codes; n = 0 is a no-op
    assert lib.moe_quantize_mx_rows(fake, 4, 256, 7, fake, fake, None) == 2
    assert lib.moe_quantize_mx_rows(fake, 4, 48, 0, fake, fake, None) == 2
    assert lib.moe_quantize_mx_rows(fake, 4, 256, 0, odd4, fake, None) == 1
    assert lib.moe_quantize_mx_rows(None, 0, 256, 0, None, None, None) == 0
    # MX GEMMs: H % 256, unknown weight format, E2M1 weights 32-byte aligned,
    # weight scales 16-byte aligned, known activations, missing outputs
    gu = lambda H, fmt, wg, sg, act, aq: lib.moe_gemm_gateup_act_mx(  # noqa: E731
        fake, fake, fake, 8, fake, 4, 16, H, 128, fmt, wg, sg, fake, fake, act, aq, fake, None)
    assert gu(384, 0, fake, fake, 0, fake) == 2
    assert gu(512, 3, fake, fake, 0, fake) == 2
    assert gu(512, 1, odd16, fake, 0, fake) == 1
    assert gu(512, 0, fake, odd4, 0, fake) == 1
    assert gu(512, 0, fake, fake, 9, fake) == 2
    assert gu(512, 0, fake, fake, 0, None) == 1
    dn = lambda H, I, fmt, sd: lib.moe_gemm_down_mx(  # noqa: E731
        fake, fake, fake, 4, 16, H, I, fmt, fake, sd, fake, None)
    assert dn(384, 128, 0, fake) == 2
    assert dn(512, 96, 0, fake) == 2
    assert dn(512, 128, 2, fake) == 2
    assert dn(512, 128, 1, odd4) == 1


def test_quantized_layers_validate_and_size_their_workspace(lib):
    from routed_mixture_experts_gemm_gb300 import _lib
    c = _cfg()
    base = [c, 256, 128, 0, 0x1000, None, None, None, 0, None, None, 1]
    bf16 = _lib.Layer(*base, 0x1000, 0x1000, 0x1000, None, None, None)
    fp8 = _lib.Layer(*base, None, None, None, None, None, None, 0, *([0x1000] * 6))
    mx = _lib.Layer(*base, None, None, None, None, None, None, 0, *([None] * 6), 1,
                    *([0x1000] * 6))
    a, b, m = (lib.gbmoe_forward_workspace_size(ctypes.byref(L), 64) for L in (bf16, fp8, mx))
    assert 0 < a < b and a < m        # quantized tokens / activations on top
    # an MX layer with an unknown format, E2M1 weights off a 32-byte boundary,
    # or H % 256 != 0 is rejected (size 0)
    bad_fmt = _lib.Layer(*base, None, None, None, None, None, None, 0, *([None] * 6), 5,
                         *([0x1000] * 6))
    bad_al = _lib.Layer(*base, None, None, None, None, None, None, 0, *([None] * 6), 1,
                        0x1010, *([0x1000] * 5))
    base_h = [c, 384] + base[2:]
    bad_h = _lib.Layer(*base_h, None, None, None, None, None, None, 0, *([None] * 6), 0,
                       *([0x1000] * 6))
    for L in (bad_fmt, bad_al, bad_h):
        assert lib.gbmoe_forward_workspace_size(ctypes.byref(L), 64) == 0


def test_wait_limit_setting_is_host_side(lib):
    # process-wide limit of the GEMMs' bounded waits: returns the previous
    # value, 0 restores the 4 s default (no device work involved)
    default = 4_000_000_000
    assert lib.gbmoe_set_wait_limit_ns(0) == default
    assert lib.gbmoe_set_wait_limit_ns(12345) == default
    assert lib.gbmoe_set_wait_limit_ns(0) == 12345
    assert lib.gbmoe_set_wait_limit_ns(0) == default


def test_mx_tile_scales_validates_on_the_host(lib):
    # rows and K multiples of 128, the source 4-byte and the destination
    # 16-byte aligned, the two not overlapping; rows = 0 enqueues nothing
    a, b = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    assert lib.moe_mx_tile_scales(a, 100, 256, b, None) == 2
    assert lib.moe_mx_tile_scales(a, 128, 96, b, None) == 2
    assert lib.moe_mx_tile_scales(ctypes.c_void_p(0x100002), 128, 256, b, None) == 1
    assert lib.moe_mx_tile_scales(a, 128, 256, ctypes.c_void_p(0x200004), None) == 1
    assert lib.moe_mx_tile_scales(a, 128, 256, ctypes.c_void_p(0x100200), None) == 1  # overlap
    assert lib.moe_mx_tile_scales(None, 0, 256, None, None) == 0
    assert lib.moe_mx_tile_scales(a, -128, 256, b, None) == 1
