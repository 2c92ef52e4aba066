"""Write oracle_tiny_f32.json: sampled oracle outputs for the tiny fp32 workload.

Calls only oracle/ (and the seeded input generators); never the CUDA path.
Run from the repository root:  python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import attn_workloads as W  # noqa: E402
from oracle import attn as OA  # noqa: E402


def main():
    w = W.WORKLOADS["tiny_f32"]
    q, k, v = W.make_prefill_inputs(w)
    out = OA.attention(q, k, v, causal=True, rope_base=w.rope_base, scale=w.scale,
                       operand_dtype="f32")
    rng = np.random.default_rng(2024)
    idx = [(0, h, t, c) for h in range(w.Hq) for t in (0, 1, 31, 63) for c in (0, 15)]
    idx += [tuple(int(x) for x in (0, rng.integers(w.Hq), rng.integers(w.T), rng.integers(w.d)))
            for _ in range(16)]
    doc = {
        "workload": "tiny_f32 (B=1, Hq=Hkv=2, T=64, d=16, RoPE base 1e4, scale 1/4, seed 0)",
        "written_by": "tests/golden/make_oracle_golden.py (oracle.attn.attention, operand_dtype f32)",
        "index": [list(i) for i in idx],
        "value": [float(out[i]) for i in idx],
    }
    with open(os.path.join(os.path.dirname(__file__), "oracle_tiny_f32.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
