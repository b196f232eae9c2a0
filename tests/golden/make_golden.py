"""Writes tiny_mixed_oracle.json: a regression fixture of the float64 oracle on
the tiny mixed batch (seed 0). Calls only `oracle` and the input generator.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_attention_07_gb300 import workloads as W  # noqa: E402


def main():
    seed = 0
    batch = W.make_batch(W.spec_tiny(seed))
    Hq = batch.spec.num_q_heads
    T = batch.q.shape[0]
    # first and last token of every request, all heads
    toks = sorted({int(batch.query_start_loc[r]) for r in range(batch.spec.num_reqs)}
                  | {int(batch.query_start_loc[r + 1]) - 1 for r in range(batch.spec.num_reqs)})
    rows = [t * Hq + h for t in toks for h in range(Hq)]
    assert max(toks) < T
    out, lse = oracle.batch_reference(batch, rows=np.array(rows, dtype=np.int64))
    doc = {
        "about": "float64 oracle on the tiny mixed batch (seed 0); first 8 output dims per row",
        "seed": seed,
        "rows": rows,
        "out": [[float(x) for x in o[:8]] for o in out],
        "lse": [float(x) for x in lse],
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_mixed_oracle.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
