"""Writes tests/golden/decode_two_keys.json: a two-key attention example whose
LSE and output follow in closed form (no oracle, no GPU code involved).

Run from the repository root:  python tests/golden/make_closed_forms.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    # q = [2, 0, 1]; k0 = [1, 0, 0]; k1 = [0, 0, 1]; sm_scale = 1/2
    # s0 = 1, s1 = 1/2; lse = 1 + ln(1 + e^-1/2); w0 = 1/(1+e^-1/2), w1 = 1 - w0
    v0, v1 = [1.0, -2.0], [3.0, 0.5]
    e = math.exp(-0.5)
    w0, w1 = 1 / (1 + e), e / (1 + e)
    d = {
        "_source": ("Worked by hand from the definition of single-head softmax "
                    "attention with LSE (DCP + FP8 KV MLA decode digest, "
                    "§关键源码片段 mla_attention.py: forward_mqa returns attn_out "
                    "and lse). s_j = sm_scale*q.k_j: s0 = 0.5*2 = 1, s1 = 0.5*1 = 0.5; "
                    "lse = ln(e + e^0.5) = 1 + ln(1 + e^-0.5); w0 = 1/(1+e^-0.5), "
                    "w1 = e^-0.5/(1+e^-0.5); out = w0*v0 + w1*v1."),
        "q": [2.0, 0.0, 1.0],
        "keys": [[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]],
        "values": [v0, v1],
        "sm_scale": "0.5",
        "lse": repr(1.0 + math.log1p(e)),
        "out": [w0 * v0[c] + w1 * v1[c] for c in range(2)],
    }
    with open(os.path.join(HERE, "decode_two_keys.json"), "w") as f:
        json.dump(d, f, indent=1)


if __name__ == "__main__":
    main()
