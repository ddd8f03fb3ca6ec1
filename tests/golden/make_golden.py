"""Writes the oracle regression fixture in this folder.

It calls only the oracle (fp64) on inputs drawn from a fixed numpy seed; the
values pin the oracle against accidental change, not the GPU path.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def main():
    B, T, Hq, Hkv, D, theta = 1, 5, 4, 2, 4, 10000.0
    rng = np.random.default_rng(20261202)
    q = rng.standard_normal((B, T, Hq, D)).round(6)
    k = rng.standard_normal((B, T, Hkv, D)).round(6)
    v = rng.standard_normal((B, T, Hkv, D)).round(6)
    dO = rng.standard_normal((B, T, Hq, D)).round(6)
    o, lse = oracle.attn_fwd(q, k, v, theta)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, theta)
    out = {
        "what": "fp64 oracle on a tiny GQA case (B1 T5 Hq4 Hkv2 D4, theta 1e4); regression pin",
        "theta": theta,
        "arrays": {n: a.tolist() for n, a in
                   (("q", q), ("k", k), ("v", v), ("dO", dO), ("o", o), ("lse", lse),
                    ("dq", dq), ("dk", dk), ("dv", dv))},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny_B1_T5_Hq4_Hkv2_D4.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
