"""Writes oracle_small_cases.json: frozen oracle outputs for a few small seeded cases.

Calls only the oracle and the seeded input generator. The file is a regression
guard for the oracle (a change to the oracle's arithmetic shows up as a diff here);
the independent pins are the tests in test_oracle_rounding.py and
test_oracle_attention.py.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from bf16_forward_attention_gb300 import inputs  # noqa: E402
from oracle import attention_fp64, bf16_bits_to_f64, round_bf16  # noqa: E402

CASES = [
    dict(name="bhsd_1x1_5x7", layout="bhsd", B=1, H=1, Sq=5, Sk=7, seed=101),
    dict(name="bshd_1x2_3x130", layout="bshd", B=1, H=2, Sq=3, Sk=130, seed=102),
    dict(name="bhsd_wide_2x1_4x9", layout="bhsd", B=2, H=1, Sq=4, Sk=9, seed=103, qk_std=8.0,
         v_dist="uniform"),
]


def compute(case):
    w = inputs.Workload(case["name"], case["layout"], case["B"], case["H"], case["Sq"], case["Sk"],
                        seed=case["seed"], qk_std=case.get("qk_std", 1.0),
                        v_dist=case.get("v_dist", "normal"))
    q, k, v = (bf16_bits_to_f64(t.view(__import__("torch").int16).numpy()) for t in inputs.make_qkv(w))
    o = attention_fp64(q, k, v, inputs.default_scale(), w.layout)
    return {m: "".join(format(int(b), "04X") for b in round_bf16(o, m).reshape(-1))
            for m in ("rtne", "rtna", "rtz")}


def main():
    out = {"source": "written by tests/golden/make_golden.py from oracle/ only", "cases": []}
    for c in CASES:
        out["cases"].append(dict(c, expected=compute(c)))
    with open(os.path.join(HERE, "oracle_small_cases.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
