"""Pure-Python brute force of the fused loss -- TEST INFRASTRUCTURE ONLY.

Triple loops with ``math.exp`` / ``math.log`` on Python floats, for tiny
inputs (n, d <= 8, V <= 50).  The tests use it as one independent check of
the C oracle; it follows the same definitions ("Loss functions and
resident-context kernels", lossk function table; "Fuse distillation + z-loss
in the triton monolithic path", section "What it does") without any of the C
code's structure (no chunk buffer, no max shift reuse, no blocking).
"""
import math


def _logits(H, W):
    return [[sum(H[t][k] * W[v][k] for k in range(len(H[t]))) for v in range(len(W))]
            for t in range(len(H))]


def _lse(row):
    m = max(row)
    return m + math.log(sum(math.exp(x - m) for x in row))


def ce(H, W, y, mask=None, wz=0.0, grad_scale=1.0):
    """Returns (total, lse list, dH, dW) for the label cross-entropy + z-loss."""
    n, d, V = len(H), len(H[0]), len(W)
    mask = mask if mask is not None else [1] * n
    nv = sum(1 for t in range(n) if mask[t])
    S = _logits(H, W)
    total = 0.0
    lses = []
    G = [[0.0] * V for _ in range(n)]
    for t in range(n):
        lse = _lse(S[t])
        lses.append(lse)
        if not mask[t] or nv == 0:
            continue
        total += (lse - S[t][y[t]]) + wz * lse * lse
        a = grad_scale / nv
        for v in range(V):
            G[t][v] = a * ((1 + 2 * wz * lse) * math.exp(S[t][v] - lse) - (1.0 if v == y[t] else 0.0))
    total = total / nv if nv else 0.0
    dH = [[sum(G[t][v] * W[v][k] for v in range(V)) for k in range(d)] for t in range(n)]
    dW = [[sum(G[t][v] * H[t][k] for t in range(n)) for k in range(d)] for v in range(V)]
    return total, lses, dH, dW


def distill(H, W, teacher, direction, T=1.0, mask=None, wz=0.0, grad_scale=1.0):
    """Returns (total, per-token loss list, dH, dW) for distillation + z-loss."""
    n, d, V = len(H), len(H[0]), len(W)
    mask = mask if mask is not None else [1] * n
    nv = sum(1 for t in range(n) if mask[t])
    S = _logits(H, W)
    total = 0.0
    per = []
    G = [[0.0] * V for _ in range(n)]
    for t in range(n):
        a = [x / T for x in S[t]]
        b = [x / T for x in teacher[t]]
        la, lb = _lse(a), _lse(b)
        q = [math.exp(x - la) for x in a]
        p = [math.exp(x - lb) for x in b]
        if direction == "ce":
            L = -sum(p[v] * (a[v] - la) for v in range(V))
        elif direction == "fkl":
            L = sum(p[v] * ((b[v] - lb) - (a[v] - la)) for v in range(V))
        else:
            L = sum(q[v] * ((a[v] - la) - (b[v] - lb)) for v in range(V))
        per.append(L if mask[t] else 0.0)
        if not mask[t] or nv == 0:
            continue
        total += L + wz * la * la
        c = grad_scale / nv
        for v in range(V):
            if direction == "rkl":
                g = q[v] * ((a[v] - la) - (b[v] - lb) - L) / T
            else:
                g = (q[v] - p[v]) / T
            G[t][v] = c * (g + 2 * wz * la * q[v] / T)
    total = total / nv if nv else 0.0
    dH = [[sum(G[t][v] * W[v][k] for v in range(V)) for k in range(d)] for t in range(n)]
    dW = [[sum(G[t][v] * H[t][k] for t in range(n)) for k in range(d)] for v in range(V)]
    return total, per, dH, dW
