"""Pure-Python loop restatement of the forward pass, for tiny shapes only.

It is written position by position from the definitions (no matrices, no
mask array, no cache): the hidden state of position p in layer l is computed
from the layer-(l-1) states of positions 0..p only. Used to pin the oracle's
vectorised code on tiny inputs.
"""
import math


def _rms(vec, eps):
    ms = sum(v * v for v in vec) / len(vec)
    return [v / math.sqrt(ms + eps) for v in vec]


def _matvec(w, vec):
    # w is row-major [out][in]; y[o] = sum_i w[o][i] * vec[i]
    return [sum(float(w[o][i]) * vec[i] for i in range(len(vec))) for o in range(len(w))]


def _rope(vec, pos, base):
    hd = len(vec)
    h = hd // 2
    out = [0.0] * hd
    for i in range(h):
        ang = pos * base ** (-2.0 * i / hd)
        c, s = math.cos(ang), math.sin(ang)
        out[i] = vec[i] * c - vec[i + h] * s
        out[i + h] = vec[i] * s + vec[i + h] * c
    return out


def forward_positions(cfg, wte, layers, lm_head, tokens):
    """Logits for every position of one sequence ``tokens`` (list of ints)."""
    d, H, Hkv, hd = cfg["d_model"], cfg["n_head"], cfg["n_kv_head"], cfg["head_dim"]
    eps, base = cfg["rms_eps"], cfg["rope_base"]
    T = len(tokens)
    xs = [[float(v) for v in wte[t]] for t in tokens]           # per position residual
    for (wq, wk, wv, wo, w_fc, w_proj) in layers:
        ks, vs, qs = [], [], []
        for p in range(T):
            xn = _rms(xs[p], eps)
            q, k, v = _matvec(wq, xn), _matvec(wk, xn), _matvec(wv, xn)
            qs.append([_rms(_rope(q[h * hd:(h + 1) * hd], p, base), eps) for h in range(H)])
            ks.append([_rms(_rope(k[g * hd:(g + 1) * hd], p, base), eps) for g in range(Hkv)])
            vs.append([v[g * hd:(g + 1) * hd] for g in range(Hkv)])
        new_xs = []
        for p in range(T):
            att = []
            for h in range(H):
                g = h * Hkv // H
                scores = [sum(qs[p][h][i] * ks[s][g][i] for i in range(hd)) / math.sqrt(hd)
                          for s in range(p + 1)]
                m = max(scores)
                e = [math.exp(sc - m) for sc in scores]
                z = sum(e)
                att.extend(sum(e[s] / z * vs[s][g][i] for s in range(p + 1)) for i in range(hd))
            x = [a + b for a, b in zip(xs[p], _matvec(wo, att))]
            hmid = [max(u, 0.0) ** 2 for u in _matvec(w_fc, _rms(x, eps))]
            x = [a + b for a, b in zip(x, _matvec(w_proj, hmid))]
            new_xs.append(x)
        xs = new_xs
    return [_matvec(lm_head, _rms(x, eps)) for x in xs]
