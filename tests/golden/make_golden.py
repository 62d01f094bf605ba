"""Write tests/golden/tiny_fp32_oracle.json from the fp64 oracle (and nothing else).

Workload: 1 request, 1 head, D=64, fp32, RoPE base 1e4, docs of 16 tokens at logical offsets 0
and 16, 8 question tokens at 32..39 attending causally to themselves and fully to both docs
(the tiny CPU-checkable case). Source of the arithmetic: the oracle's form A, i.e. attention over
keys materialised at absolute positions, which the LazyAttention summaries ("Mathematical
equivalence") state the deferred form reproduces exactly.

Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workload as W  # noqa: E402


def main():
    wl = W.tiny_fp32()
    out, lse = oracle.attend_request(wl, 0)
    doc = {
        "workload": "tiny_fp32 (seed 0)",
        "source": "oracle form A (fp64), written by tests/golden/make_golden.py",
        "out": out.tolist(),
        "lse": lse.tolist(),
    }
    with open(os.path.join(HERE, "tiny_fp32_oracle.json"), "w") as f:
        json.dump(doc, f)


if __name__ == "__main__":
    main()
