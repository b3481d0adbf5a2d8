"""Writes rope_example.json: a rotary embedding worked by hand with the
math module only (no oracle code), width 4, base 10000.

Pair i turns by position * 10000^(-2i/4): pair 0 by position rad, pair 1 by
position / 100 rad.  Interleaved layout: pairs are dims (0,1) and (2,3);
rotate-half layout: pairs are dims (0,2) and (1,3).
"""

import json
import math
import os

x = [1.0, -2.0, 0.5, 3.0]
out = {"base": 10000.0, "x": x, "cases": []}
for pos in [0, 1, 7, 1000]:
    t0, t1 = pos * 1.0, pos / 100.0
    c0, s0, c1, s1 = math.cos(t0), math.sin(t0), math.cos(t1), math.sin(t1)
    inter = [x[0] * c0 - x[1] * s0, x[0] * s0 + x[1] * c0,
             x[2] * c1 - x[3] * s1, x[2] * s1 + x[3] * c1]
    half = [x[0] * c0 - x[2] * s0, x[1] * c1 - x[3] * s1,
            x[0] * s0 + x[2] * c0, x[1] * s1 + x[3] * c1]
    out["cases"].append({"position": pos, "interleaved": inter, "rotate_half": half})
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "rope_example.json"), "w") as f:
    json.dump(out, f, indent=1)
