"""Writes tests/golden/page_example.json from the fp64 oracle only.

The FAG-V2 page's call example (section "调用示例", call example) runs the
backward on a TND problem of shape {256, 1, 128} in FLOAT32 with every
element of query, key, value, dy and attentionIn equal to 1,
softmaxMax = softmaxSum = 3.0 in every lane of their {256, 1, 8} tensors,
scaleValue = 0.088388, keepProb = 1, preTokens = nextTokens = 65536,
headNum = 1, sparseMode 0, actual lengths {256} / {256}.  The page prints no
output values, so the expected values here are the oracle's, and the test
also checks them against the closed form that the inputs force:
dP_ij = D_i = 128 so dS = 0 and dQ = dK = 0 exactly, while every P_ij equals
exp(0.088388 * 128 - 3) / 3 and dV = 256 * that value in every element.

Run:  python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def page_example():
    t, n, d = 256, 1, 128
    ones = np.ones((t, n, d))
    stats = np.full((t, n, 8), 3.0)
    dq, dk, dv = oracle.varlen_backward(ones, ones, ones, ones, ones, stats, stats,
                                        [256], [256], 0.088388, 65536, 65536)
    assert np.all(dv == dv.flat[0])
    return {
        "source": ("FAG-V2 page, section 调用示例 (call example): TND {256,1,128} FLOAT32 all-ones "
                   "query/key/value/dy/attentionIn, softmaxMax = softmaxSum = 3.0, scaleValue 0.088388, "
                   "keepProb 1, preTokens = nextTokens = 65536, headNum 1, sparseMode 0, "
                   "actualSeqQLen = actualSeqKvLen = {256}. The page prints no outputs; values written "
                   "by tests/golden/make_golden.py from the oracle."),
        "shape": [t, n, d],
        "scale": 0.088388,
        "stat_value": 3.0,
        "pre_tokens": 65536,
        "next_tokens": 65536,
        "lens": [256],
        "dq_max_abs": float(np.abs(dq).max()),
        "dk_max_abs": float(np.abs(dk).max()),
        "dv_value": float(dv.flat[0]),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "page_example.json")
    with open(out, "w") as f:
        json.dump(page_example(), f, indent=1)
        f.write("\n")
    print("wrote", out)
