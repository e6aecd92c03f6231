"""Literal loop versions of the chunk-step formulas, for tiny shapes only.

Written separately from the oracle (plain Python floats and the ``math``
module, nested loops over t, h, w instead of index arithmetic) so that the two
can pin each other.  Inputs are nested lists or NumPy arrays; outputs are
nested Python lists.
"""
import math


def pairs_per_axis(D):
    # a third of the pairs (rounded down) for each spatial axis, the rest for time
    third = (D // 2) // 3
    return (D // 2) - 2 * third, third, third


def rope_token(vec, t, h, w, base):
    """Rotate one head vector (list of D floats) of a token at (t, h, w)."""
    D = len(vec)
    n_t, n_h, n_w = pairs_per_axis(D)
    out = list(vec)
    pair = 0
    for pos, n_a in ((t, n_t), (h, n_h), (w, n_w)):
        for j in range(n_a):
            ang = pos * math.pow(base, -float(j) / float(n_a))
            a, b = vec[2 * pair], vec[2 * pair + 1]
            out[2 * pair] = a * math.cos(ang) - b * math.sin(ang)
            out[2 * pair + 1] = a * math.sin(ang) + b * math.cos(ang)
            pair += 1
    return out


def rope_block(x, grid_t, grid_h, grid_w, t0, base):
    """x[b][n][h][d] -> rotated copy (lists)."""
    B, H = len(x), len(x[0][0])
    out = [[None] * (grid_t * grid_h * grid_w) for _ in range(B)]
    for b in range(B):
        n = 0
        for tt in range(grid_t):
            for hh in range(grid_h):
                for ww in range(grid_w):
                    out[b][n] = [rope_token([float(e) for e in x[b][n][head]], t0 + tt, hh, ww, base)
                                 for head in range(H)]
                    n += 1
    return out


def attend(q, keys, values, scale):
    """q: list[Nq][H][D]; keys/values: list[Nkv][H][D] -> list[Nq][H][D]."""
    Nq, H, D = len(q), len(q[0]), len(q[0][0])
    out = [[[0.0] * D for _ in range(H)] for _ in range(Nq)]
    for i in range(Nq):
        for head in range(H):
            scores = []
            for j in range(len(keys)):
                acc = 0.0
                for d in range(D):
                    acc += q[i][head][d] * keys[j][head][d]
                scores.append(acc * scale)
            top = max(scores)
            weights = [math.exp(s - top) for s in scores]
            total = sum(weights)
            for d in range(D):
                acc = 0.0
                for j in range(len(keys)):
                    acc += weights[j] * values[j][head][d]
                out[i][head][d] = acc / total
    return out


def linear(rows, weight, bias=None):
    """rows [M][K], weight [N][K] -> rows @ weight^T (+ bias)."""
    out = []
    for r in rows:
        line = []
        for n in range(len(weight)):
            acc = 0.0 if bias is None else float(bias[n])
            for k in range(len(r)):
                acc += float(r[k]) * float(weight[n][k])
            line.append(acc)
        out.append(line)
    return out
