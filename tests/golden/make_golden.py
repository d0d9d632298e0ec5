"""Writes tests/golden/tiny.json: the oracle's outputs on the tiny workload
(T=64, H=256, E=8, I=128, top-2, softmax, renormalise, scaling 1.0, seed 0).

The pages print no worked example, so this file is a regression anchor for
the oracle (and a stored expectation for the GPU tests), written only by
calling oracle/ on synth/ inputs:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    cfg = synth.CONFIGS["tiny"]
    o = oracle.run_config(cfg, nthreads=1)
    doc = {
        "workload": "tiny routed MoE: T=64 H=256 E=8 I=128 top-2 softmax renormalise "
                    "routed_scaling=1.0 seed=0 (synth generator)",
        "source": "oracle/ on synth/ inputs; the pages print no numeric example",
        "ids_log": o["ids_log"].tolist(),
        "ids_phys": o["ids_phys"].tolist(),
        "weights_f32_hex": [[f"{int(v):08x}" for v in row] for row in o["weights"].view(np.uint32)],
        "counts": o["counts"].tolist(),
        "offsets": o["offsets"].tolist(),
        "flat_to_row": o["flat_to_row"].tolist(),
        "out_bf16_hex": ["".join(f"{int(v):04x}" for v in row) for row in o["out"]],
    }
    with open(os.path.join(HERE, "tiny.json"), "w") as f:
        json.dump(doc, f, indent=0)


if __name__ == "__main__":
    main()
