"""Writes tests/golden/oracle_tiny_layer.json from the oracle alone.

A regression fixture of the oracle on the tiny MoE workload (T=64, H=256,
I=512, E=8, top-2, seed 0): routing of the first tokens, a few output rows as
bf16 bit patterns, and whole-tensor sums.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import inputs  # noqa: E402
import oracle  # noqa: E402
from helpers import moe_experts, moe_host_inputs  # noqa: E402


def compute():
    cfg = inputs.WORKLOADS["tiny"]
    x_bits, logits = moe_host_inputs(0, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    w13, w2 = moe_experts(0, cfg)
    r = oracle.moe_layer(x, logits, cfg["k"], w13.w, w13.s, w2.w, w2.s)
    rows = [0, 17, 63]
    return {
        "workload": "tiny MoE layer T=64 H=256 I=512 E=8 top-2, seed 0",
        "ids_first4": r["ids"][:4].tolist(),
        "seg_indptr": r["seg"].tolist(),
        "out_rows": {str(t): oracle.bf16_bits(r["out"][t]).tolist() for t in rows},
        "out_sum": float(r["out"].sum()),
        "out_abs_sum": float(np.abs(r["out"]).sum()),
        "y13_abs_sum": float(np.abs(r["y13"]).sum()),
        "hq_code_sum": int(r["hq"].astype(np.int64).sum()),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny_layer.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
