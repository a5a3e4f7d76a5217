"""Write tests/golden/oracle_small.json: small attention cases and the fp64 oracle's outputs.

Calls nothing but ``oracle/`` (and the seeded input generator).  The stored outputs are a
regression record of the oracle itself: tests/test_oracle.py recomputes them and fails if the
oracle's arithmetic changes.  They are not an independent pin; the pins are the closed forms,
brute force and invariants in that test file.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from oracle import rope as orope  # noqa: E402
from fa_workloads import bf16_bits  # noqa: E402

CASES = [
    # name, lq, lk, hq, hkv, d, causal, window, alibi, rope
    ("causal_square", 6, 6, 2, 2, 8, True, 0, False, False),
    ("noncausal_q_lt_k", 4, 7, 2, 1, 8, False, 0, False, False),
    ("causal_window_gqa", 7, 9, 4, 2, 8, True, 3, False, False),
    ("alibi_causal", 5, 5, 2, 2, 8, True, 0, True, False),
    ("rope_causal", 5, 6, 2, 2, 8, True, 0, False, True),
]


def run_case(name, lq, lk, hq, hkv, d, causal, window, alibi, rope, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(lq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(lk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(lk, hkv, d, generator=g).to(torch.bfloat16)
    slopes = np.array([2.0 ** -(i + 1) for i in range(hq)]) if alibi else None
    if rope:
        cos_t, sin_t = orope.tables(16, d)
        q = orope.rotate_bf16(q, np.arange(lq) + lk - lq, cos_t, sin_t, d)
        k = orope.rotate_bf16(k, np.arange(lk), cos_t, sin_t, d)
    rows = oracle.all_rows([lq], hq)
    o, lse = oracle.attention_rows(bf16_bits(q), bf16_bits(k), bf16_bits(v), [0], [lq], [0], [lk],
                                   1.0 / np.sqrt(d), causal, window, rows, alibi_slopes=slopes)
    return {"name": name, "lq": lq, "lk": lk, "hq": hq, "hkv": hkv, "d": d, "causal": causal,
            "window": window, "alibi": alibi, "rope": rope, "seed": seed,
            "o": [float(x) for x in o.reshape(-1)], "lse": [float(x) for x in lse.reshape(-1)]}


def build():
    return [run_case(*c, seed=1000 + i) for i, c in enumerate(CASES)]


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(out, "w") as f:
        json.dump({"cases": build()}, f, indent=0)
    print("wrote", out)
