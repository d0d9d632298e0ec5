"""moe_permute_static: the permutation for callers that cannot allocate
device memory (a latency-bound loop that cannot afford the device-wide
synchronisation cudaMalloc/cudaFree may cause, or a process whose GPU memory
belongs to another framework's pool).  Its scratch is a fixed array inside
the library.

Checked through the C ABI, bit for bit, against moe_permute with a caller
workspace and against the oracle's counting sort, on several calls in a row
whose sizes differ (the array keeps the previous call's contents): batches
of more than 4096 routed rows run the histogram / column-scan / scatter
kernels, which keep their per-worker histograms and completion counter in
the array; small batches run the one-block kernel.  Also checked: requests
beyond the array's size are refused before anything is enqueued.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

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


def _ids(gen, T, k, P, skew):
    """k distinct experts per token; with skew, half of the picks fall on the
    first eighth of the experts (uneven histograms across workers)."""
    w = torch.ones(P)
    if skew:
        w[: max(1, P // 8)] = 8.0 * 7.0
    ids = torch.multinomial(w.expand(T, P), k, replacement=False, generator=gen)
    return ids.to(torch.int32)


# (T, k, P, H, skewed): the first three take the multi-kernel path through
# the static scratch (T*k > 4096) with different worker and expert counts, so
# every call finds the previous one's histograms and counter in the array;
# the fourth takes the one-block path (T*k <= 4096), the fifth the scratch
# path again.
CASES = [(2048, 8, 288, 128, True), (3000, 4, 64, 256, False), (700, 8, 1000, 64, True),
         (300, 8, 40, 256, False), (1200, 6, 7, 128, True)]


def test_static_scratch_permute_matches_workspace_permute_and_oracle(lib):
    gen = torch.Generator(device="cpu").manual_seed(7)
    for T, k, P, H, skew in CASES:
        ids_h = _ids(gen, T, k, P, skew)
        ids = ids_h.to(DEV)
        x = torch.randn((T, H), generator=gen).to(torch.bfloat16).to(DEV)
        st_s, got = _run(lib, True, ids, x, P)
        assert st_s == 0, (T, k, P)
        assert lib.gbmoe_permute_workspace_size(T, k, P) > 0
        # the oracle's stable counting sort (reading R9), bit for bit
        counts, offs, r2t, f2r = oracle.permute(ids_h.numpy(), P)
        for key, ref in (("counts", counts), ("offsets", offs), ("r2t", r2t), ("f2r", f2r)):
            assert np.array_equal(got[key].cpu().numpy(), ref), (key, T, k, P)
        x_h = x.cpu().view(torch.int16).numpy()
        assert np.array_equal(got["x_perm"].cpu().view(torch.int16).numpy(), x_h[r2t])
        # and the workspace entry point, bit for bit
        st_w, ref = _run(lib, False, ids, x, P)
        assert st_w == 0
        for key in ("counts", "offsets", "r2t", "f2r"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16))
    status = ctypes.c_int(-1)
    assert lib.gbmoe_check_device_status(torch.cuda.current_stream().cuda_stream,
                                         ctypes.byref(status)) == 0
    assert status.value == 0


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
    # the largest request that fits still runs (E_phys = 256: T*k up to 261,888)
    T, k, P = 32736, 8, 256
    assert lib.gbmoe_permute_workspace_size(T, k, P) <= 1 << 20
    gen = torch.Generator(device="cpu").manual_seed(11)
    ids_h = _ids(gen, T, k, P, True)
    o = _outputs(T, k, P, 8)
    st = lib.moe_permute_static(_p(ids_h.to(DEV)), T, k, P, None, 0, _p(o["counts"]),
                                _p(o["offsets"]), _p(o["r2t"]), _p(o["f2r"]), None,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    counts, offs, r2t, f2r = oracle.permute(ids_h.numpy(), P)
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["r2t"].cpu().numpy(), r2t)
    assert np.array_equal(o["f2r"].cpu().numpy(), f2r)
