"""Writes tests/golden/tiny_topk.json from the float64 oracle (and nothing else).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import dsa_workloads as W  # noqa: E402
import oracle  # noqa: E402


def main():
    wl = W.make_workload(W.SPECS["tiny"])
    res = oracle.dsa_forward(wl)
    out = {"workload": "tiny (1 x 512, 16 queries, k=64, seed 0)",
           "written_by": "tests/golden/make_golden.py (oracle only)",
           "idx": [res.idx[t].tolist() for t in range(wl.total_q)]}
    with open(os.path.join(ROOT, "tests", "golden", "tiny_topk.json"), "w") as f:
        json.dump(out, f)


if __name__ == "__main__":
    main()
