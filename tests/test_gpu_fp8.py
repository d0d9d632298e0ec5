"""GPU parity of the FP8 (OCP E4M3) expert path ("Stage 4" quantized paths,
W8A8FP; reading R17), through the C ABI, against the CPU oracle:

- row quantization: codes and scales bit-exact (both sides divide in IEEE
  fp32 and round to nearest even with saturation);
- FP8 gate/up GEMM (128- and 256-token tiles, contiguous and gathered
  operands, ragged and empty groups): activations within the output
  tolerance of the oracle;
- FP8 down GEMM: y within fp32 accumulation error of the same products taken
  from the GPU's own activation codes (a one-ulp bf16 flip of an activation can
  move its E4M3 code, so y is checked on identical codes).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import bf16_dev
from tests.test_gpu_parity import DEV, _bf, _np, assert_within_tol
from tests.test_oracle_mlp import _bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import routed_mixture_experts_gemm_gb300 as g
    return g


def test_quantize_rows_bit_exact(gb, rng):
    x = rng.standard_normal((300, 512)) * np.exp(rng.uniform(-8, 8, (300, 1)))
    xb = _bf16_bits(x)
    xb[7] = 0                                  # all-zero row: scale 1
    xb[8, :5] = _bf16_bits(np.float32([448.0, -1e-30, 1e-38, 3e38, -0.0]))
    q_o, s_o = oracle.quantize_rows(xb)
    q, s = gb.moe_quantize_fp8_rows(bf16_dev(xb, DEV))
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(s).view(np.uint32), s_o.view(np.uint32))
    assert np.array_equal(_np(q), q_o)


def _fp8_case(H, I, rows, seed):
    rng = np.random.default_rng(seed)
    P = len(rows)
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(offs[-1])
    T = max(N // 2, 1) + 5
    x = _bf16_bits(rng.standard_normal((T, H)))
    r2t = rng.integers(0, T, N).astype(np.int32)
    W = [[_bf16_bits(rng.standard_normal(sh) * 0.05) for sh in ((I, H), (I, H), (H, I))]
         for _ in range(P)]
    xq, sx = oracle.quantize_rows(x)
    qs = [[oracle.quantize_rows(w) for w in ws] for ws in W]
    st = lambda j, k: np.stack([q[j][k] for q in qs])  # noqa: E731
    return dict(x=x, xq=xq, sx=sx, r2t=r2t, offs=offs, N=N, T=T,
                wg=st(0, 0), sg=st(0, 1), wu=st(1, 0), su=st(1, 1), wd=st(2, 0), sd=st(2, 1))


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("shape", [(256, 128, [40, 3, 17, 0, 90]), (512, 256, [150, 200, 300, 1, 0]),
                                   (1024, 512, [20 + (p * 7) % 23 for p in range(16)])])
@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_fp8_gemms(gb, shape, act):
    H, I, rows = shape
    c = _fp8_case(H, I, rows, H + I + len(rows))
    act_o, y_o = oracle.ffn_grouped_fp8(c["xq"], c["sx"], c["r2t"], c["offs"], c["wg"], c["sg"],
                                        c["wu"], c["su"], c["wd"], c["sd"], nthreads=8,
                                        activation=act)
    d = {k: _dev(v) for k, v in c.items() if isinstance(v, np.ndarray)}
    a1 = gb.moe_gemm_gateup_act_fp8(d["xq"], d["sx"], d["offs"], d["wg"], d["sg"], d["wu"],
                                    d["su"], row_to_token=d["r2t"], activation=act)
    # the same rows permuted up front (contiguous operand)
    xq_p = _dev(c["xq"][c["r2t"]])
    sx_p = _dev(c["sx"][c["r2t"]])
    a2 = gb.moe_gemm_gateup_act_fp8(xq_p, sx_p, d["offs"], d["wg"], d["sg"], d["wu"], d["su"],
                                    activation=act)
    assert gb.check_device_status() == 0
    ref = synth.bf16_to_f32(act_o)
    assert_within_tol(_bf(a1), ref, f"fp8 act gathered {shape}")
    assert_within_tol(_bf(a2), ref, f"fp8 act {shape}")
    # down GEMM on the GPU's own activation codes
    aq, sa = gb.moe_quantize_fp8_rows(a1)
    y = gb.moe_gemm_down_fp8(aq, sa, d["offs"], d["wd"], d["sd"])
    assert gb.check_device_status() == 0
    aq_h, sa_h = _np(aq), _np(sa)
    dq = np.array([oracle.e4m3_to_f32(k) for k in range(256)], dtype=np.float64)
    offs = c["offs"]
    y_h = _np(y).astype(np.float64)
    for p in range(len(rows)):
        r0, r1 = offs[p], offs[p + 1]
        if r0 == r1:
            continue
        wdd = dq[c["wd"][p]] * c["sd"][p][:, None]
        a = dq[aq_h[r0:r1]] * sa_h[r0:r1, None]
        ref_y = a @ wdd.T
        bound = np.abs(a) @ np.abs(wdd).T
        assert np.all(np.abs(y_h[r0:r1] - ref_y) <= 2.0 ** -12 * bound + 1e-30)


@pytest.mark.parametrize("name", ["tiny", "mini_prefill", "mini_hash", "mini_skew"])
def test_fp8_forward_end_to_end(gb, name):
    """moe_forward with FP8 routed experts against the oracle pipeline: the
    same routing and permutation (bit-exact), the weight codes bit-exact, the
    oracle's FP8 MLP on its own codes of x and of the weights, the shared
    expert in bf16, the fixed-order combine."""
    from synth.device import device_case
    cfg = synth.MINI[name]
    case = device_case(cfg, DEV, host_weights=True)
    d = case.dev
    q = [gb.quantize_experts_fp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
    layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                        router_bias=d["router_bias"], corr_bias=d["corr_bias"],
                        tid2eid=d["tid2eid"], log2phy=d["log2phy"],
                        replica_cnt=d["replica_cnt"], shared=d["shared"],
                        fp8=[a for pair in q for a in pair])
    ids_p = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    out = gb.moe_forward(layer, case.x, input_ids=case.input_ids, ids_phys=ids_p)
    assert gb.check_device_status() == 0
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
    assert np.array_equal(_np(ids_p), ref["ids_phys"])
    qo = []
    for (wq, ws), wh in zip(q, case.weights_host):
        P, R, K = wh.shape
        cq, cs = oracle.quantize_rows(wh.reshape(P * R, K))
        assert np.array_equal(_np(wq).reshape(P * R, K), cq)
        assert np.array_equal(_np(ws).reshape(-1).view(np.uint32), cs.view(np.uint32))
        qo += [cq.reshape(P, R, K), cs.reshape(P, R)]
    xq, sx = oracle.quantize_rows(case.inputs["x"])
    _, y = oracle.ffn_grouped_fp8(xq, sx, ref["row_to_token"], ref["offsets"], *qo, nthreads=8)
    out_ref = oracle.combine(y, ref["flat_to_row"], ref["weights"], ref.get("ys"))
    assert_within_tol(_bf(out), synth.bf16_to_f32(out_ref), f"fp8 forward {name}")
    # run-to-run determinism (bitwise)
    out2 = gb.moe_forward(layer, case.x, input_ids=case.input_ids)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_fp8_forward_rejects_unaligned_hidden(gb):
    from synth.device import device_case
    case = device_case(synth.MINI["mini_decode"], DEV, host_weights=True)   # H = 384
    d = case.dev
    q = [gb.quantize_experts_fp8(d[k]) for k in ("w_gate", "w_up", "w_down")]
    layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                        router_bias=d["router_bias"], corr_bias=d["corr_bias"],
                        fp8=[a for pair in q for a in pair])
    with pytest.raises(gb.GbmoeError):
        gb.moe_forward(layer, case.x)
