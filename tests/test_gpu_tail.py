"""GPU parity of the latent-MoE tail (NVIDIA LatentMoERunner page, tier-1 tail
with one rank): out = bf16(rmsnorm(latent) . up_proj^T + shared), through the
C ABI, against the CPU oracle on the same seeded inputs, element by element
within |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (and 2 bf16 ulps of the output
scale).  Shapes cover one and many tokens, ragged token counts, every
up-projection tile variant (Hm % 256 == 0 or not), with and without the norm
and the shared term.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import bf16_dev
from tests.test_gpu_parity import DEV, _bf, assert_within_tol
from tests.test_oracle_mlp import _bf16_bits

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256, 256), (37, 512, 384), (300, 256, 1024), (128, 1024, 512), (2048, 256, 256)]


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import routed_mixture_experts_gemm_gb300 as g
    return g


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("norm,shared", [(True, True), (True, False), (False, True)])
def test_latent_tail(gb, shape, norm, shared):
    T, L, Hm = shape
    rng = np.random.default_rng(T + L + Hm + 2 * norm + shared)
    lat = _bf16_bits(rng.standard_normal((T, L)) * 2)
    w = _bf16_bits(1.0 + 0.2 * rng.standard_normal(L)) if norm else None
    up = _bf16_bits(rng.standard_normal((Hm, L)) / np.sqrt(L))
    sh = _bf16_bits(rng.standard_normal((T, Hm))) if shared else None
    ref = oracle.latent_tail(lat, up, w, eps=1e-6, shared=sh, nthreads=8)
    out = gb.moe_latent_tail(bf16_dev(lat, DEV), bf16_dev(up, DEV),
                             None if w is None else bf16_dev(w, DEV), eps=1e-6,
                             shared=None if sh is None else bf16_dev(sh, DEV))
    assert gb.check_device_status() == 0
    assert_within_tol(_bf(out), synth.bf16_to_f32(ref), f"tail {shape} norm={norm} shared={shared}")


def test_latent_tail_argument_checks(gb):
    lat = torch.zeros((4, 200), dtype=torch.bfloat16, device=DEV)
    up = torch.zeros((128, 200), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gb.GbmoeError):  # L not a multiple of 128
        gb.moe_latent_tail(lat, up)
    lat = torch.zeros((0, 256), dtype=torch.bfloat16, device=DEV)
    up = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    assert gb.moe_latent_tail(lat, up).shape == (0, 128)
