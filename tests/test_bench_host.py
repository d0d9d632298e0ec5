"""Host logic of bench.py that needs no GPU: the reference arm's JSON line
(the CPU oracle timed on a bounded sample), the DRAM-traffic lookup tied to
the kernel source hash, and the algorithmic-byte formulas behind the
roofline fractions (checked against hand-computed values)."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                         timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["config"]["workload"] == "decode"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_traffic_lookup_follows_the_source_hash(monkeypatch):
    h = bench.source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    e = d["expert_mlp_fused/decode"]
    if e["source_hash"] == h:
        assert bench.profiled_traffic("expert_mlp_fused", "decode") == e["bytes_per_launch"]
    assert bench.profiled_traffic("no_such_kernel", "decode") is None
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic("expert_mlp_fused", "decode") is None


def test_algorithmic_bytes_formulas():
    cfg = SimpleNamespace(T=4, H=256, I=128, k=2, N=8)
    counts = np.array([3, 0, 5, 0, 0], np.int32)      # two experts touched
    H, I = 256, 128
    # credited: the touched experts' weights and x read once; the activation
    # (and, fused, its read-back and the fp32 outputs) reported apart
    b, touched, inter = bench.touched_bytes(cfg, counts, fused=False)
    assert touched == 2
    assert b == 2 * 2 * I * H * 2 + 4 * H * 2
    assert inter == 8 * I * 2
    bf, _, interf = bench.touched_bytes(cfg, counts, fused=True)
    assert bf == 2 * 3 * I * H * 2 + 4 * H * 2
    assert interf == 8 * I * 2 + 8 * I * 2 + 8 * H * 4
    g8, d8 = bench.q_bytes(cfg, counts, "fp8_row")
    assert g8 == 2 * 2 * I * (H + 4) + 4 * (H + 4)
    assert d8 == 2 * H * (I + 4) + 8 * (I + 4)
    gm, dm = bench.q_bytes(cfg, counts, "mxfp8")
    g4, d4 = bench.q_bytes(cfg, counts, "w4a8")
    # E2M1 weights take half the code bytes of E4M3; scales and tokens equal
    assert gm - g4 == 2 * 2 * I * H * 0.5
    assert dm - d4 == 2 * H * I * 0.5
    assert gm == 2 * 2 * I * (H + H / 32) + 4 * (H + H / 32)
    assert dm == 2 * H * (I + I / 32) + 8 * (I + I / 32)


def test_traffic_profile_covers_every_roofline_kernel():
    """Every roofline the bench line reports has a DRAM-traffic entry, all
    taken on one kernel source, each a scaled-up measurement that reads the
    algorithmic bytes at least about once (ratios below 1 would mean the
    twin's traffic was not the launch's)."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    keys = ["expert_mlp_fused/decode", "gemm_gateup/prefill", "expert_mlp_fused/hash",
            "gemm_gateup/skew"]
    keys += [f"{k}_gateup/{w}" for k in ("fp8_row", "mxfp8", "w4a8") for w in ("decode", "prefill")]
    hashes = set()
    for k in keys:
        assert k in d, k
        e = d[k]
        hashes.add(e["source_hash"])
        assert e["bytes_per_launch"] > 0
        assert 0.98 <= e["ratio"] <= 1.25, (k, e["ratio"])
        scaled = e["measured_small_case_bytes"] * e["full_case_algorithmic_bytes"] / \
            e["small_case_algorithmic_bytes"]
        assert abs(scaled - e["bytes_per_launch"]) <= 1e-6 * scaled + 1, k
    assert len(hashes) == 1, hashes
