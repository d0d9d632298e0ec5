"""GPU parity of the MX block-scaled expert path (Stage 4 quantized paths,
MXFP and W4A8; reading R18), through the C ABI, against the CPU oracle:

- MX quantization (E4M3 and E2M1): codes and scale bytes bit-exact (power-of-
  two scaling is exact, both sides round to nearest even with saturation);
- MX gate/up GEMM with the activation quantized in its epilogue (gathered and
  contiguous token operands, ragged and empty groups, E4M3 and E2M1
  weights): the activation's MX codes against the oracle's -- equal codes
  except where the bf16 activation itself differs by an ulp, and every code
  within one E4M3 step of the oracle's activation;
- MX down GEMM: y within fp32 accumulation error of the same products taken
  from the GPU's own activation codes;
- moe_forward with MX routed experts against the oracle pipeline.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import bf16_dev
from tests.test_gpu_parity import DEV, _bf, _np, assert_within_tol
from tests.test_oracle_mlp import _bf16_bits
from tests.test_oracle_mx import deq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import routed_mixture_experts_gemm_gb300 as g
    return g


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("rows,K", [(128, 128), (384, 7168), (256, 2048)])
def test_mx_tile_scales_is_the_documented_rearrangement(gb, rows, K, rng):
    """Tiled weight scales: for row block rb and K stage ks, 512 bytes whose byte
    r*16 + j*4 + b is the scale of row rb*128 + 32j + r, K block 4ks + b."""
    sf = rng.integers(0, 256, (rows, K // 32), dtype=np.uint8)
    got = _np(gb.moe_mx_tile_scales(_dev(sf))).reshape(-1)
    exp = (sf.reshape(rows // 128, 4, 32, K // 128, 4)   # rb, j, r, ks, b
             .transpose(0, 3, 2, 1, 4).reshape(-1))         # rb, ks, r, j, b
    assert np.array_equal(got, exp)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_mx_quantize_bit_exact(gb, fmt, rng):
    x = rng.standard_normal((300, 512)) * np.exp(rng.uniform(-20, 20, (300, 16))).repeat(32, 1)
    xb = _bf16_bits(x)
    xb[7] = 0                                                # all-zero blocks
    xb[8, :32] = _bf16_bits(np.float32([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4))  # E2M1 ties
    xb[9, :32] = _bf16_bits(np.float32([448.0, 480.0, -1e-30, 3e38] + [1.0] * 28))
    xb[10, 32:64] = _bf16_bits(np.float32([2.0 ** -130] * 32))  # bf16 subnormals
    q_o, s_o = oracle.mx_quantize_rows(xb, fmt)
    q, s = gb.moe_quantize_mx_rows(bf16_dev(xb, DEV), fmt)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(s), s_o)
    assert np.array_equal(_np(q), q_o)


def _mx_case(H, I, rows, wfmt, seed):
    rng = np.random.default_rng(seed)
    P = len(rows)
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    N = int(offs[-1])
    T = max(N // 2, 1) + 5
    x = _bf16_bits(rng.standard_normal((T, H)))
    r2t = rng.integers(0, T, N).astype(np.int32)
    W = [[_bf16_bits(rng.standard_normal(sh) * 0.05) for sh in ((I, H), (I, H), (H, I))]
         for _ in range(P)]
    xq, xs = oracle.mx_quantize_rows(x, "e4m3")
    qs = [[oracle.mx_quantize_rows(w, wfmt) for w in ws] for ws in W]
    st = lambda j, k: np.stack([q[j][k] for q in qs])  # noqa: E731
    return dict(x=x, xq=xq, xs=xs, r2t=r2t, offs=offs, N=N, T=T,
                wg=st(0, 0), sg=st(0, 1), wu=st(1, 0), su=st(1, 1), wd=st(2, 0), sd=st(2, 1))


def check_act_codes(aq, as_, aq_o, as_o, act_o, what):
    """GPU activation codes against the oracle's: the bf16 activation may
    differ by an ulp (fp32 accumulation order), which can move a code by one
    step or, rarely, a block's exponent; every dequantized value stays within
    one E4M3 step (plus a bf16 ulp, plus the saturation at 448 X) of the
    oracle's bf16 activation."""
    a_o = synth.bf16_to_f32(act_o).astype(np.float64)
    d = deq(aq, as_, "e4m3")
    X = np.repeat(np.exp2(as_.astype(np.float64) - 127.0), 32, axis=1)
    r = np.abs(a_o) / X
    step = X * np.exp2(np.maximum(np.floor(np.log2(np.maximum(r, 1e-300))), -6) - 3)
    # the scale rule leaves the block maximum in [256, 512) X: values above
    # 448 X saturate to 448 X
    sat = np.maximum(np.abs(a_o) - 448.0 * X, 0.0)
    err = np.abs(d - a_o)
    bad = err > step + sat + 2.0 ** -7 * np.abs(a_o) + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} codes off by more than one step"
    assert np.mean(as_ == as_o) > 0.995, f"{what}: block exponents"
    assert np.mean(aq == aq_o) > 0.99, f"{what}: codes"


@pytest.mark.parametrize("shape", [(256, 128, [40, 3, 17, 0, 90]), (512, 256, [150, 200, 300, 1, 0]),
                                   (1024, 512, [20 + (p * 7) % 23 for p in range(16)])])
@pytest.mark.parametrize("wfmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_mx_gemms(gb, shape, wfmt, act):
    H, I, rows = shape
    c = _mx_case(H, I, rows, wfmt, H + I + len(rows))
    act_o, aq_o, as_o, y_o = oracle.ffn_grouped_mx(
        c["xq"], c["xs"], c["r2t"], c["offs"], c["wg"], c["sg"], c["wu"], c["su"], c["wd"],
        c["sd"], wfmt=wfmt, nthreads=8, activation=act)
    d = {k: _dev(v) for k, v in c.items() if isinstance(v, np.ndarray)}
    aq1, as1 = gb.moe_gemm_gateup_act_mx(d["xq"], d["xs"], d["offs"], d["wg"], d["sg"], d["wu"],
                                         d["su"], w_fmt=wfmt, row_to_token=d["r2t"],
                                         activation=act)
    # the same rows permuted up front (contiguous operand)
    aq2, as2 = gb.moe_gemm_gateup_act_mx(_dev(c["xq"][c["r2t"]]), _dev(c["xs"][c["r2t"]]),
                                         d["offs"], d["wg"], d["sg"], d["wu"], d["su"],
                                         w_fmt=wfmt, activation=act)
    assert gb.check_device_status() == 0
    for aq, as_, how in ((aq1, as1, "gathered"), (aq2, as2, "contiguous")):
        check_act_codes(_np(aq), _np(as_), aq_o, as_o, act_o, f"{how} {shape} {wfmt}")
    assert np.array_equal(_np(aq1), _np(aq2)) and np.array_equal(_np(as1), _np(as2))
    # down GEMM on the GPU's own activation codes
    y = gb.moe_gemm_down_mx(aq1, as1, d["offs"], d["wd"], d["sd"], w_fmt=wfmt)
    assert gb.check_device_status() == 0
    # run-to-run determinism (bitwise), also on the CTA-pair kernels
    aq3, as3 = gb.moe_gemm_gateup_act_mx(d["xq"], d["xs"], d["offs"], d["wg"], d["sg"], d["wu"],
                                         d["su"], w_fmt=wfmt, row_to_token=d["r2t"],
                                         activation=act)
    y3 = gb.moe_gemm_down_mx(aq1, as1, d["offs"], d["wd"], d["sd"], w_fmt=wfmt)
    assert torch.equal(aq1, aq3) and torch.equal(as1, as3)
    assert torch.equal(y.view(torch.int32), y3.view(torch.int32))
    a = deq(_np(aq1), _np(as1), "e4m3")
    y_h = _np(y).astype(np.float64)
    offs = c["offs"]
    for p in range(len(rows)):
        r0, r1 = offs[p], offs[p + 1]
        if r0 == r1:
            continue
        wdd = deq(c["wd"][p], c["sd"][p], wfmt)
        ref_y = a[r0:r1] @ wdd.T
        bound = np.abs(a[r0:r1]) @ np.abs(wdd).T
        assert np.all(np.abs(y_h[r0:r1] - ref_y) <= 2.0 ** -12 * bound + 1e-30), f"y {p}"


@pytest.mark.parametrize("wfmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("name", ["tiny", "mini_prefill", "mini_hash", "mini_skew"])
def test_mx_forward_end_to_end(gb, name, wfmt):
    """moe_forward with MX routed experts against the oracle pipeline: the same
    routing (bit-exact), the weights' MX codes (bit-exact), the oracle's MX MLP
    on its own codes, the shared expert in bf16, the fixed-order combine."""
    from synth.device import device_case
    cfg = synth.MINI[name]
    case = device_case(cfg, DEV, host_weights=True)
    d = case.dev
    q = [gb.quantize_experts_mx(d[k], wfmt) for k in ("w_gate", "w_up", "w_down")]
    layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                        router_bias=d["router_bias"], corr_bias=d["corr_bias"],
                        tid2eid=d["tid2eid"], log2phy=d["log2phy"],
                        replica_cnt=d["replica_cnt"], shared=d["shared"],
                        mx=[wfmt] + [a for pair in q for a in pair])
    ids_p = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    out = gb.moe_forward(layer, case.x, input_ids=case.input_ids, ids_phys=ids_p)
    assert gb.check_device_status() == 0
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
    assert np.array_equal(_np(ids_p), ref["ids_phys"])
    qo = []
    for (wq, ws), wh in zip(q, case.weights_host):
        P, R, K = wh.shape
        cq, cs = oracle.mx_quantize_rows(wh.reshape(P * R, K), wfmt)
        assert np.array_equal(_np(wq).reshape(P * R, -1), cq)
        assert np.array_equal(_np(ws).reshape(P * R, -1), cs)
        qo += [cq.reshape(P, R, -1), cs.reshape(P, R, -1)]
    xq, xs = oracle.mx_quantize_rows(case.inputs["x"], "e4m3")
    _, _, _, y = oracle.ffn_grouped_mx(xq, xs, ref["row_to_token"], ref["offsets"], *qo,
                                       wfmt=wfmt, nthreads=8)
    out_ref = oracle.combine(y, ref["flat_to_row"], ref["weights"], ref.get("ys"))
    assert_within_tol(_bf(out), synth.bf16_to_f32(out_ref), f"mx forward {name} {wfmt}")
    out2 = gb.moe_forward(layer, case.x, input_ids=case.input_ids)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_mx_rejects_bad_arguments(gb):
    x = torch.zeros((16, 384), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gb.GbmoeError):
        gb.moe_quantize_mx_rows(x[:, :48].contiguous(), "e4m3")  # K % 32 != 0
    with pytest.raises(gb.GbmoeError):
        gb.moe_quantize_mx_rows(x, 7)                          # unknown format
    q, s = gb.moe_quantize_mx_rows(x, "e4m3")
    w = torch.zeros((1, 128, 384), dtype=torch.uint8, device=DEV)
    ws = torch.zeros((1, 128, 12), dtype=torch.uint8, device=DEV)
    offs = torch.tensor([0, 16], dtype=torch.int32, device=DEV)
    with pytest.raises(gb.GbmoeError):                         # H % 256 != 0
        gb.moe_gemm_gateup_act_mx(q, s, offs, w, ws, w, ws)


@pytest.mark.parametrize("rows", [[32, 32, 32, 32], [33, 33, 33, 33], [1, 0, 0, 127]])
@pytest.mark.parametrize("wfmt", ["e4m3", "e2m1"])
def test_mx_variant_boundary(gb, rows, wfmt):
    """Both sides of the decode-variant switch (32 rows per group on average)
    and a group of 127 rows next to empty ones."""
    H, I = 256, 128
    c = _mx_case(H, I, rows, wfmt, 7 + sum(rows))
    act_o, aq_o, as_o, _ = oracle.ffn_grouped_mx(
        c["xq"], c["xs"], c["r2t"], c["offs"], c["wg"], c["sg"], c["wu"], c["su"], c["wd"],
        c["sd"], wfmt=wfmt, nthreads=8)
    d = {k: _dev(v) for k, v in c.items() if isinstance(v, np.ndarray)}
    aq, as_ = gb.moe_gemm_gateup_act_mx(d["xq"], d["xs"], d["offs"], d["wg"], d["sg"], d["wu"],
                                        d["su"], w_fmt=wfmt, row_to_token=d["r2t"])
    y = gb.moe_gemm_down_mx(aq, as_, d["offs"], d["wd"], d["sd"], w_fmt=wfmt)
    assert gb.check_device_status() == 0
    check_act_codes(_np(aq), _np(as_), aq_o, as_o, act_o, f"boundary {rows} {wfmt}")
    a = deq(_np(aq), _np(as_), "e4m3")
    offs = c["offs"]
    for p in range(len(rows)):
        r0, r1 = offs[p], offs[p + 1]
        if r0 == r1:
            continue
        wdd = deq(c["wd"][p], c["sd"][p], wfmt)
        bound = np.abs(a[r0:r1]) @ np.abs(wdd).T
        assert np.all(np.abs(_np(y)[r0:r1] - a[r0:r1] @ wdd.T) <= 2.0 ** -12 * bound + 1e-30)


@pytest.mark.parametrize("T", [1, 2, 17])
@pytest.mark.parametrize("kind", ["fp8_row", "w4a8"])
def test_quantized_forward_small_batches(gb, T, kind):
    """moe_forward with quantized experts on batches of 1, 2 and 17 tokens
    (the tiny layer's first T tokens) against the oracle pipeline."""
    import dataclasses
    from synth.device import device_case
    cfg = dataclasses.replace(synth.CONFIGS["tiny"], T=T)
    case = device_case(cfg, DEV, host_weights=True)
    d = case.dev
    kw = dict(router_bias=d["router_bias"], corr_bias=d["corr_bias"], tid2eid=d["tid2eid"],
              log2phy=d["log2phy"], replica_cnt=d["replica_cnt"], shared=d["shared"])
    ref = oracle.run_config(cfg, inputs=case.inputs, weights=case.weights_host)
    qo = []
    if kind == "fp8_row":
        q = [gb.quantize_experts_fp8(d[n]) for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                            fp8=[a for pair in q for a in pair], **kw)
        for w in case.weights_host:
            P, R, K = w.shape
            cq, cs = oracle.quantize_rows(w.reshape(P * R, K))
            qo += [cq.reshape(P, R, K), cs.reshape(P, R)]
        xq, xs = oracle.quantize_rows(case.inputs["x"])
        _, y = oracle.ffn_grouped_fp8(xq, xs, ref["row_to_token"], ref["offsets"], *qo,
                                      nthreads=4)
    else:
        q = [gb.quantize_experts_mx(d[n], "e2m1") for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                            mx=["e2m1"] + [a for pair in q for a in pair], **kw)
        for w in case.weights_host:
            P, R, K = w.shape
            cq, cs = oracle.mx_quantize_rows(w.reshape(P * R, K), "e2m1")
            qo += [cq.reshape(P, R, -1), cs.reshape(P, R, -1)]
        xq, xs = oracle.mx_quantize_rows(case.inputs["x"], "e4m3")
        _, _, _, y = oracle.ffn_grouped_mx(xq, xs, ref["row_to_token"], ref["offsets"], *qo,
                                           wfmt="e2m1", nthreads=4)
    out = gb.moe_forward(layer, case.x)
    assert gb.check_device_status() == 0
    exp = oracle.combine(y, ref["flat_to_row"], ref["weights"], ref.get("ys"))
    assert_within_tol(_bf(out), synth.bf16_to_f32(exp), f"{kind} T={T}")


@pytest.mark.parametrize("kind", ["fp8_row", "mxfp8", "w4a8"])
def test_quantized_forward_with_outliers(gb, kind):
    """moe_forward with quantized experts on hidden states holding a few
    entries at +-20 sigma (the generator's own tails stop near 3.5 sigma): the
    per-row amax of the FP8 scales and the MX block exponents see the outliers,
    on both sides, and the layer still matches the oracle pipeline."""
    from synth.device import bf16_dev, device_case
    cfg = synth.MINI["mini_prefill"]
    case = device_case(cfg, DEV, host_weights=True)
    rng = np.random.default_rng(2024)
    x = case.inputs["x"].copy()
    T, H = x.shape
    spots = [(int(t), int(h)) for t, h in zip(rng.choice(T, 24, replace=False),
                                                rng.integers(0, H, 24))]
    for i, (t, h) in enumerate(spots):
        x[t, h] = 0x41A0 if i % 2 == 0 else 0xC1A0  # bf16 bits of +20.0 / -20.0
    inputs = dict(case.inputs, x=x)
    xd = bf16_dev(x, DEV)
    d = case.dev
    kw = dict(router_bias=d["router_bias"], corr_bias=d["corr_bias"], tid2eid=d["tid2eid"],
              log2phy=d["log2phy"], replica_cnt=d["replica_cnt"], shared=d["shared"])
    ref = oracle.run_config(cfg, inputs=inputs, weights=case.weights_host)
    qo = []
    if kind == "fp8_row":
        q = [gb.quantize_experts_fp8(d[n]) for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                            fp8=[a for pair in q for a in pair], **kw)
        for w in case.weights_host:
            P, R, K = w.shape
            cq, cs = oracle.quantize_rows(w.reshape(P * R, K))
            qo += [cq.reshape(P, R, K), cs.reshape(P, R)]
        xq, xs = oracle.quantize_rows(x)
        _, y = oracle.ffn_grouped_fp8(xq, xs, ref["row_to_token"], ref["offsets"], *qo,
                                      nthreads=4)
        # the device quantizer sees the same amax per token
        xq_d, xs_d = gb.moe_quantize_fp8_rows(xd)
        assert np.array_equal(_np(xq_d), xq)
        assert np.array_equal(_np(xs_d).view(np.uint32), xs.view(np.uint32))
    else:
        wfmt = "e4m3" if kind == "mxfp8" else "e2m1"
        q = [gb.quantize_experts_mx(d[n], wfmt) for n in ("w_gate", "w_up", "w_down")]
        layer = gb.MoELayer(case.layer.cfg, d["w_router"], None, None, None,
                            mx=[wfmt] + [a for pair in q for a in pair], **kw)
        for w in case.weights_host:
            P, R, K = w.shape
            cq, cs = oracle.mx_quantize_rows(w.reshape(P * R, K), wfmt)
            qo += [cq.reshape(P, R, -1), cs.reshape(P, R, -1)]
        xq, xs = oracle.mx_quantize_rows(x, "e4m3")
        _, _, _, y = oracle.ffn_grouped_mx(xq, xs, ref["row_to_token"], ref["offsets"], *qo,
                                           wfmt=wfmt, nthreads=4)
        xq_d, xs_d = gb.moe_quantize_mx_rows(xd, "e4m3")
        assert np.array_equal(_np(xq_d), xq)
        assert np.array_equal(_np(xs_d), xs)
    ids_p = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    out = gb.moe_forward(layer, xd, ids_phys=ids_p)
    assert gb.check_device_status() == 0
    assert np.array_equal(_np(ids_p), ref["ids_phys"])
    exp = oracle.combine(y, ref["flat_to_row"], ref["weights"], ref.get("ys"))
    assert_within_tol(_bf(out), synth.bf16_to_f32(exp), f"{kind} with outliers")
