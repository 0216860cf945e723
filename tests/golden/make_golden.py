"""Writes closed_forms.json: small attention cases whose results follow from
closed forms worked out by hand (no oracle, no library).  Run it from the
repository root: python tests/golden/make_golden.py

Cases (the formulas are in each case's "derivation"):
  three_keys      forward, the online softmax of the shader pages reduced to
                  three scores 0, 1, 2 (meganeura attention.wgsl, fn main:
                  out = sum_t e^(s_t - m) v_t / sum_t e^(s_t - m), lse = (m, log l))
  rope_d4         the same with rotary embedding on half-split pairs, D = 4, base 100
  backward_d1     the plain gradient for one query over two keys, D = 1
  empty_cross     cross attention over zero keys (attention.wgsl: zeros, lse -1e30)
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def three_keys():
    e = math.e
    z = 1 + e + e * e
    return {
        "call": "forward", "mask": 2, "H": 1, "G": 1, "D": 4, "q_seq": 1, "kv_seq": 3,
        "q": [[2, 0, 0, 0]], "k": [[0, 5, -1, 2], [1, 0, 7, 0], [2, -3, 0, 1]], "v": [[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0]],
        "out": [[1 / z, e / z, e * e / z, 0.0]], "lse": [[[2.0, math.log(1 + 1 / e + 1 / (e * e))]]],
        "derivation": "scale 1/2, scores q.k_t/2 = k_t[0] = 0, 1, 2; weights e^0, e^1, e^2 over 1 + e + e^2; "
                      "V rows are unit vectors; lse = (max 2, log(1 + e^-1 + e^-2))",
    }


def rope_d4():
    s = [math.sin(2.0) / 2, (math.cos(1.0) + math.sin(0.1)) / 2]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    l = sum(w)
    return {
        "call": "forward_rope", "mask": 2, "H": 1, "G": 1, "D": 4, "q_seq": 3, "kv_seq": 2, "base": 100.0, "row": 2,
        "q": [[0, 0, 0, 0], [0, 0, 0, 0], [1, 1, 0, 0]], "k": [[0, 0, 1, 0], [1, 0, 0, 1]], "v": [[1, 0, 0, 0], [0, 1, 0, 0]],
        "out_row": [w[0] / l, w[1] / l, 0.0, 0.0], "lse_row": [m, math.log(l)],
        "derivation": "pairs (0,2) turn by 1 rad per position, (1,3) by 100^(-1/2) = 0.1; q row 2 -> "
                      "(cos 2, cos 0.2, sin 2, sin 0.2), k0 at 0 stays e2, k1 at 1 -> (cos 1, -sin 0.1, sin 1, cos 0.1); "
                      "scores (scale 1/2) sin(2)/2 and (cos 1 + sin 0.1)/2",
    }


def backward_d1():
    a, k1, k2, v1, v2, g = 0.5, 1.0, -2.0, 3.0, -1.0, 2.0
    s1, s2 = a * k1, a * k2  # scale 1/sqrt(1) = 1
    p1 = 1 / (1 + math.exp(s2 - s1))
    p2 = 1 - p1
    out = p1 * v1 + p2 * v2
    ds1, ds2 = p1 * (g * v1 - g * out), p2 * (g * v2 - g * out)
    return {
        "call": "backward", "mask": 2, "H": 1, "G": 1, "D": 1, "q_seq": 1, "kv_seq": 2,
        "q": [[a]], "k": [[k1], [k2]], "v": [[v1], [v2]], "dout": [[g]],
        "dq": [[ds1 * k1 + ds2 * k2]], "dk": [[ds1 * a], [ds2 * a]], "dv": [[p1 * g], [p2 * g]],
        "derivation": "p1 = 1/(1 + e^(a(k2 - k1))), out = p1 v1 + p2 v2, ds_i = p_i g (v_i - out), "
                      "dq = sum ds_i k_i, dk_i = ds_i a, dv_i = p_i g",
    }


def empty_cross():
    return {
        "call": "forward", "mask": 2, "H": 2, "G": 1, "D": 4, "q_seq": 2, "kv_seq": 0,
        "q": [[1, 2, 3, 4, 5, 6, 7, 8], [-1, 0, 1, 0, 2, 0, 3, 0]], "k": [], "v": [],
        "out": [[0.0] * 8, [0.0] * 8], "lse": [[[-1e30, -1e30], [-1e30, -1e30]]] * 2,
        "derivation": "no keys: the pages' zero-sum guard writes zeros, and the LSE pair keeps its -1e30 start",
    }


if __name__ == "__main__":
    cases = {"three_keys": three_keys(), "rope_d4": rope_d4(), "backward_d1": backward_d1(),
             "empty_cross": empty_cross()}
    with open(os.path.join(HERE, "closed_forms.json"), "w") as f:
        json.dump(cases, f, indent=1)
        f.write("\n")
