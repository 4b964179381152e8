"""Writes tests/golden/oracle_tiny_layer.json and oracle_tiny_shard.json from the oracle alone.

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


def compute_shard():
    """Shard 1 of 2 of the same layer (experts 1, 3, 5, 7 as local ids 0-3)."""
    cfg = inputs.WORKLOADS["tiny"]
    x_bits, logits = moe_host_inputs(0, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    w13, w2 = moe_experts(0, cfg)
    experts = [1, 3, 5, 7]
    emap = [-1] * cfg["E"]
    for l, e in enumerate(experts):
        emap[e] = l
    r = oracle.moe_layer(x, logits, cfg["k"], lambda l: w13.w(experts[l]), lambda l: w13.s(experts[l]),
                         lambda l: w2.w(experts[l]), lambda l: w2.s(experts[l]), expert_map=emap)
    rows = [0, 17, 63]
    return {
        "workload": "tiny MoE layer T=64 H=256 I=512 E=8 top-2, seed 0; expert-parallel shard of experts 1, 3, 5, 7",
        "seg_indptr": r["seg"].tolist(),
        "src2dst_first8": r["src2dst"][:8].tolist(),
        "out_rows": {str(t): oracle.bf16_bits(r["out"][t]).tolist() for t in rows},
        "out_sum": float(r["out"].sum()),
        "out_abs_sum": float(np.abs(r["out"]).sum()),
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny_layer.json"), "w") as f:
        json.dump(compute(), f, indent=1)
        f.write("\n")
    with open(os.path.join(HERE, "oracle_tiny_shard.json"), "w") as f:
        json.dump(compute_shard(), f, indent=1)
        f.write("\n")
