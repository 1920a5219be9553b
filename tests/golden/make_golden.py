"""Writes the oracle regression fixtures in this folder.  Calls only oracle/
(and the seeded input generator): the pages print no worked numeric example
for the attention forward, so these fixtures freeze the pinned fp64 oracle's
own output on small seeded cases, to catch drift across compilers and hosts.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_forward_11_gb300 import inputs  # noqa: E402

CASES = [
    # name, B, Sq, Skv, Hq, Hkv, D, causal, scale, seed, q_sigma
    ("small_causal_gqa", 1, 5, 7, 4, 2, 16, 1, 0.25, 101, 1.0),
    ("small_noncausal", 2, 3, 9, 2, 2, 16, 0, 0.25, 102, 1.0),
    ("small_sharp", 1, 4, 6, 2, 1, 16, 0, 0.25, 103, 4.0),
    ("small_fully_masked", 1, 6, 3, 1, 1, 16, 1, 0.25, 104, 1.0),
]


def main():
    for (name, B, Sq, Skv, Hq, Hkv, D, causal, scale, seed, qs) in CASES:
        q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=seed, q_sigma=qs)
        o, lse = oracle.attn_full(q, k, v, int(causal), scale)
        rec = {"case": name, "B": B, "Sq": Sq, "Skv": Skv, "Hq": Hq, "Hkv": Hkv, "D": D,
               "causal": causal, "scale": scale, "seed": seed, "q_sigma": qs,
               "source": "oracle/oracle.c via tests/golden/make_golden.py",
               "o": [float.hex(float(x)) for x in o.ravel()],
               "lse": [float.hex(float(x)) for x in lse.ravel()]}
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(rec, f, indent=0)
            f.write("\n")


if __name__ == "__main__":
    main()
