"""moe_permute_static: the permutation for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Checked
through the C ABI against moe_permute with a caller workspace, bit for bit,
on two calls in a row with different inputs, and for its size limit.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import routed_mixture_experts_gemm_gb300 as gb
    return gb.library()


def _p(t):
    return None if t is None else t.data_ptr()


def _outputs(T, k, P, H):
    N = T * k
    return {"counts": torch.full((P,), -1, dtype=torch.int32, device=DEV),
            "offsets": torch.full((P + 1,), -1, dtype=torch.int32, device=DEV),
            "r2t": torch.full((N,), -1, dtype=torch.int32, device=DEV),
            "f2r": torch.full((N,), -1, dtype=torch.int32, device=DEV),
            "x_perm": torch.zeros((N, H), dtype=torch.bfloat16, device=DEV)}


def _run(lib, static, ids, x, P):
    T, k = ids.shape
    H = x.shape[1]
    o = _outputs(T, k, P, H)
    s = torch.cuda.current_stream().cuda_stream
    args = (_p(ids), T, k, P, _p(x), H, _p(o["counts"]), _p(o["offsets"]), _p(o["r2t"]),
            _p(o["f2r"]), _p(o["x_perm"]))
    if static:
        st = lib.moe_permute_static(*args, s)
    else:
        need = lib.gbmoe_permute_workspace_size(T, k, P)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        st = lib.moe_permute(*args, _p(ws), need, s)
    torch.cuda.synchronize()
    return st, o


def test_static_scratch_permute_matches_workspace_permute(lib):
    gen = torch.Generator(device="cpu").manual_seed(7)
    cases = [(300, 8, 40, 256), (1000, 4, 64, 128)]  # two calls in a row, different sizes
    for T, k, P, H in cases:
        ids = torch.stack([torch.randperm(P, generator=gen)[:k] for _ in range(T)])
        ids = ids.to(torch.int32).to(DEV)
        x = torch.randn((T, H), generator=gen).to(torch.bfloat16).to(DEV)
        st_s, got = _run(lib, True, ids, x, P)
        st_w, ref = _run(lib, False, ids, x, P)
        assert st_s == 0 and st_w == 0
        for key in ("counts", "offsets", "r2t", "f2r"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))


def test_static_scratch_rejects_requests_beyond_its_limit(lib):
    T, k, P = 40000, 8, 1024   # ceil(320000/256) * 1024 * 4 bytes > 1 MiB
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    o = _outputs(T, k, P, 8)
    st = lib.moe_permute_static(_p(ids), T, k, P, None, 0, _p(o["counts"]), _p(o["offsets"]),
                                _p(o["r2t"]), _p(o["f2r"]), None,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 3  # GBMOE_ERR_WORKSPACE
    assert lib.gbmoe_status_string(st) == b"workspace missing or too small"
    assert bool((o["counts"] == -1).all())  # nothing was enqueued
