"""The oracle still reproduces the stored tiny-workload fixture."""
import json
import os

import numpy as np

import oracle
import synth

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_tiny():
    with open(os.path.join(HERE, "tiny.json")) as f:
        g = json.load(f)
    g["weights"] = np.array([[int(h, 16) for h in r] for r in g["weights_f32_hex"]],
                            dtype=np.uint32).view(np.float32)
    g["out"] = np.array([[int(r[i:i + 4], 16) for i in range(0, len(r), 4)]
                         for r in g["out_bf16_hex"]], dtype=np.uint16)
    return g


def test_oracle_reproduces_tiny_fixture():
    g = load_tiny()
    o = oracle.run_config(synth.CONFIGS["tiny"], nthreads=2)
    assert np.array_equal(o["ids_log"], np.array(g["ids_log"]))
    assert np.array_equal(o["counts"], np.array(g["counts"]))
    assert np.array_equal(o["flat_to_row"], np.array(g["flat_to_row"]))
    assert np.array_equal(o["weights"], g["weights"])
    assert np.array_equal(o["out"], g["out"])
