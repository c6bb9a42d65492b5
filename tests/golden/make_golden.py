"""Writes tests/golden/tiny_attention.json.  Calls only ``oracle/``.

The stored cases are small enough to read by eye; they pin the oracle
against later changes to itself and check that x86-64 and aarch64 hosts
compute the same values.  Inputs are fixed short decimals (exactly
representable in bf16), so they are reproducible without a generator.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

CASES = [
    dict(q=[[1.0, 0.5], [-0.25, 2.0], [0.75, -1.5]],
         k=[[0.5, -1.0], [1.25, 0.25], [-2.0, 0.5]],
         v=[[1.0, 2.0], [-0.5, 0.125], [3.0, -1.0]], alpha=0.5, causal=False),
    dict(q=[[1.0, 0.5], [-0.25, 2.0], [0.75, -1.5]],
         k=[[0.5, -1.0], [1.25, 0.25], [-2.0, 0.5]],
         v=[[1.0, 2.0], [-0.5, 0.125], [3.0, -1.0]], alpha=0.5, causal=True),
    dict(q=[[2.0, -1.0, 0.5, 0.25]], k=[[1.0, 1.0, -1.0, 0.5], [0.0, -2.0, 1.5, 1.0]],
         v=[[0.5, -0.5, 1.0, 2.0], [-1.0, 0.25, 0.75, -3.0]], alpha=0.5, causal=True),
]


def main():
    out = []
    for c in CASES:
        o, lse = oracle.attention_head(c["q"], c["k"], c["v"], c["alpha"], c["causal"])
        out.append(dict(c, o=o.tolist(), lse=lse.tolist()))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_attention.json")
    with open(path, "w") as f:
        json.dump({"generator": "tests/golden/make_golden.py (oracle only)",
                   "cases": out}, f, indent=1)


if __name__ == "__main__":
    main()
