"""Pure-Python scalar-loop attention for tiny inputs (a pin for the oracle).

Written independently of ``oracle/``: plain nested loops over the textbook
definition of causal scaled-dot-product attention with GQA head sharing,
no numpy in the arithmetic.
"""

import math


def brute_forward(q, k, v, scale):
    """q: [n][hq][d], k/v: [n][hkv][d] nested lists -> (o [n][hq][d], lse [n][hq])."""
    n, hq, d = len(q), len(q[0]), len(q[0][0])
    hkv = len(k[0])
    grp = hq // hkv
    o = [[[0.0] * d for _ in range(hq)] for _ in range(n)]
    lse = [[0.0] * hq for _ in range(n)]
    for h in range(hq):
        g = h // grp
        for i in range(n):
            scores = []
            for j in range(i + 1):
                acc = 0.0
                for x in range(d):
                    acc += q[i][h][x] * k[j][g][x]
                scores.append(scale * acc)
            m = max(scores)
            ex = [math.exp(s - m) for s in scores]
            tot = sum(ex)
            for x in range(d):
                acc = 0.0
                for j in range(i + 1):
                    acc += ex[j] / tot * v[j][g][x]
                o[i][h][x] = acc
            lse[i][h] = m + math.log(tot)
    return o, lse


def brute_backward(q, k, v, do, scale):
    """Gradients by the chain rule written out per scalar."""
    n, hq, d = len(q), len(q[0]), len(q[0][0])
    hkv = len(k[0])
    grp = hq // hkv
    o, lse = brute_forward(q, k, v, scale)
    dq = [[[0.0] * d for _ in range(hq)] for _ in range(n)]
    dk = [[[0.0] * d for _ in range(hkv)] for _ in range(n)]
    dv = [[[0.0] * d for _ in range(hkv)] for _ in range(n)]
    for h in range(hq):
        g = h // grp
        for i in range(n):
            delta = sum(do[i][h][x] * o[i][h][x] for x in range(d))
            for j in range(i + 1):
                s = scale * sum(q[i][h][x] * k[j][g][x] for x in range(d))
                p = math.exp(s - lse[i][h])
                dp = sum(do[i][h][x] * v[j][g][x] for x in range(d))
                ds = p * (dp - delta)
                for x in range(d):
                    dq[i][h][x] += scale * ds * k[j][g][x]
                    dk[j][g][x] += scale * ds * q[i][h][x]
                    dv[j][g][x] += p * do[i][h][x]
    return dq, dk, dv
