"""Scalar brute-force twin of the oracle for tiny inputs: Python floats (IEEE float64) and plain loops.

TEST INFRASTRUCTURE ONLY. It reads codes one byte at a time, sorts every logit in full and sums every product
in a loop, so that it shares no vectorised step with moe_oracle.py. Sources as in moe_oracle.py.
"""
from __future__ import annotations

import math


def weight_int4(q_packed, s, b, r, c, group=64):
    byte = int(q_packed[r][c // 2])
    code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
    return float(s[r][c // group]) * code + float(b[r][c // group])


def weight_int8(q, s, b, r, c, group=64):
    return float(s[r][c // group]) * int(q[r][c]) + float(b[r][c // group])


def matvec(weight_fn, n_rows, n_cols, x):
    out = []
    for r in range(n_rows):
        acc = 0.0
        for c in range(n_cols):
            acc += weight_fn(r, c) * float(x[c])
        out.append(acc)
    return out


def silu(z):
    return z / (1.0 + math.exp(-z))


def block_token(w, x, top_k, group=64):
    """One token through the block, loop by loop. Returns (out list, ids sorted, weights, sigmoid gate)."""
    H = len(x)
    E = len(w["router_q"]) - 1
    logits = matvec(lambda r, c: weight_int8(w["router_q"], w["router_s"], w["router_b"], r, c, group),
                    E + 1, H, x)
    m = max(logits[:E])
    ex = [math.exp(v - m) for v in logits[:E]]
    z = sum(ex)
    p = [v / z for v in ex]
    order = sorted(range(E), key=lambda e: (-logits[e], e))
    ids = sorted(order[:top_k])
    zs = sum(p[e] for e in ids)
    wts = [p[e] / zs for e in ids]
    sg = 1.0 / (1.0 + math.exp(-logits[E]))

    def mlp(gate, up, down, n_inter):
        a = matvec(gate, n_inter, H, x)
        u = matvec(up, n_inter, H, x)
        h = [silu(a[i]) * u[i] for i in range(n_inter)]
        return matvec(down, H, n_inter, h)

    out = [0.0] * H
    for e, wt in zip(ids, wts):
        I = len(w["exp_gate_q"][e])
        y = mlp(lambda r, c: weight_int4(w["exp_gate_q"][e], w["exp_gate_s"][e], w["exp_gate_b"][e], r, c, group),
                lambda r, c: weight_int4(w["exp_up_q"][e], w["exp_up_s"][e], w["exp_up_b"][e], r, c, group),
                lambda r, c: weight_int4(w["exp_down_q"][e], w["exp_down_s"][e], w["exp_down_b"][e], r, c, group),
                I)
        for i in range(H):
            out[i] += wt * y[i]
    Is = len(w["sh_gate_q"])
    ys = mlp(lambda r, c: weight_int8(w["sh_gate_q"], w["sh_gate_s"], w["sh_gate_b"], r, c, group),
             lambda r, c: weight_int8(w["sh_up_q"], w["sh_up_s"], w["sh_up_b"], r, c, group),
             lambda r, c: weight_int8(w["sh_down_q"], w["sh_down_s"], w["sh_down_b"], r, c, group),
             Is)
    for i in range(H):
        out[i] += sg * ys[i]
    return out, ids, wts, sg
