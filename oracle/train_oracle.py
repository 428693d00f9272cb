"""fp64 CPU oracle of the training step: the mean next-token loss of a batch, its
gradient with respect to every parameter (the backward pass), and the Adam update.

TEST INFRASTRUCTURE. Only the tests may import this module; the product path never
calls it and shares no code with it.

The Microgpt summary (telegra.ph) describes the training loop (section 训练过程): run
the forward pass and the cross-entropy loss against the true next tokens (item 2),
then backpropagate to get the gradient of the loss for every parameter (item 3). Its
section 自动微分 says how: the chain rule applied from the loss back through the
computation graph (item 2). Here that is written out by hand, one rule per operation
of the forward pass in `gpt_oracle` (the same model, the same readings), in reverse
order:

* cross-entropy: d loss / d z = (softmax(z) - onehot(target)) / (rows counted), 0 for
  a row whose target is negative (left out, as in `gpt_oracle.cross_entropy`);
* y = x W^T: dW += dy^T x, dx = dy W;
* RMSNorm y = x r, r = (mean(x^2) + eps)^(-1/2): dx = r dy - (r^3 / n) x sum(dy x);
* RoPE, a rotation of each pair (i, i + hd/2) by +theta: dx is dy rotated by -theta;
* ReLU^2, h = max(a, 0)^2: da = 2 max(a, 0) dh;
* attention, S = q k^T / sqrt(hd) masked to s <= t, P = softmax(S), O = P V:
  dV = P^T dO, dP = dO V^T, dS = P (dP - rowsum(dP P)), dq = dS k / sqrt(hd),
  dk = dS^T q / sqrt(hd); the query heads of one KV head add into its dk and dv;
* residual x + f(x): the gradient passes to both;
* embedding lookup: each position's dx is added into its token's row of d wte.

The update (训练过程 item 4) is Adam with bias-corrected moment estimates
(`adam_update`); `train_step` chains the three. Nothing is blocked or fused; numpy
matmuls are the only library steps.
"""
from __future__ import annotations

import numpy as np

from oracle import gpt_oracle as G

F64 = np.float64


def _rms(x, eps):
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r, r


def _rms_back(x, r, dy):
    n = x.shape[-1]
    return r * dy - (r ** 3 / n) * x * np.sum(dy * x, axis=-1, keepdims=True)


def _rope_back(dy, cos, sin):
    half = dy.shape[-1] // 2
    d1, d2 = dy[..., :half], dy[..., half:]
    return np.concatenate([d1 * cos + d2 * sin, -d1 * sin + d2 * cos], axis=-1)


def loss_and_grads(cfg, wte, layers, lm_head, tokens, targets):
    """Mean next-token loss of tokens [B, n] (positions 0..n-1 of each sequence)
    against targets [B, n], and the gradient of that mean with respect to wte,
    each layer's (wq, wk, wv, wo, w_fc, w_proj) and lm_head, as float64 arrays of
    the parameters' shapes. Returns (loss, {"wte": ..., "layers": [...],
    "lm_head": ...})."""
    cfg = G._cfg(cfg)
    G._check_weights(cfg, wte, layers, lm_head)
    H, Hkv, hd, eps = cfg["n_head"], cfg["n_kv_head"], cfg["head_dim"], cfg["rms_eps"]
    group = H // Hkv
    scale = 1.0 / np.sqrt(F64(hd))
    tokens = np.asarray(tokens)
    targets = np.asarray(targets)
    B, n = tokens.shape
    count = int(np.sum(targets >= 0))
    wte64 = np.asarray(wte, dtype=F64)
    lm = np.asarray(lm_head, dtype=F64)
    lw = [tuple(np.asarray(m, dtype=F64) for m in mats) for mats in layers]
    d_wte = np.zeros_like(wte64)
    d_lm = np.zeros_like(lm)
    d_layers = [[np.zeros_like(m) for m in mats] for mats in lw]
    cos, sin = G.rope_tables(n, hd, cfg["rope_base"])
    allowed = np.arange(n)[None, :] <= np.arange(n)[:, None]
    loss_sum = 0.0
    for b in range(B):
        # ---------------------------------------------------------------- forward
        x = wte64[tokens[b]]
        saved = []
        for wq, wk, wv, wo, w_fc, w_proj in lw:
            x_in = x
            xn1, r1 = _rms(x_in, eps)
            q = G._split_heads(xn1 @ wq.T, H, hd)
            k = G._split_heads(xn1 @ wk.T, Hkv, hd)
            v = G._split_heads(xn1 @ wv.T, Hkv, hd)
            qr, kr = G.apply_rope(q, cos, sin), G.apply_rope(k, cos, sin)
            qn, rq = _rms(qr, eps)
            kn, rk = _rms(kr, eps)
            P = np.empty((H, n, n))
            O = np.empty((H, n, hd))
            for h in range(H):
                s = np.where(allowed, (qn[h] @ kn[h // group].T) * scale, -np.inf)
                P[h] = G.softmax_rows(s)
                O[h] = P[h] @ v[h // group]
            att = G._merge_heads(O)
            x_mid = x_in + att @ wo.T
            xn2, r2 = _rms(x_mid, eps)
            a = xn2 @ w_fc.T
            hmid = np.square(np.maximum(a, 0.0))
            x = x_mid + hmid @ w_proj.T
            saved.append((x_in, xn1, r1, qr, kr, qn, kn, rq, rk, v, P, att, x_mid, xn2, r2, a,
                          hmid))
        xnf, rf = _rms(x, eps)
        z = xnf @ lm.T
        # ------------------------------------------------------------------- loss
        t = targets[b]
        keep = t >= 0
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        lse = np.log(e.sum(axis=1)) + m[:, 0]
        rows = np.nonzero(keep)[0]
        loss_sum += float(np.sum(lse[rows] - z[rows, t[rows]]))
        dz = e / e.sum(axis=1, keepdims=True)
        dz[rows, t[rows]] -= 1.0
        dz[~keep] = 0.0
        dz /= count
        # --------------------------------------------------------------- backward
        d_lm += dz.T @ xnf
        dx = _rms_back(x, rf, dz @ lm)
        for li in range(len(lw) - 1, -1, -1):
            wq, wk, wv, wo, w_fc, w_proj = lw[li]
            dq_, dk_, dv_, do_, dfc_, dproj_ = d_layers[li]
            (x_in, xn1, r1, qr, kr, qn, kn, rq, rk, v, P, att, x_mid, xn2, r2, a,
             hmid) = saved[li]
            dproj_ += dx.T @ hmid
            da = (dx @ w_proj) * 2.0 * np.maximum(a, 0.0)
            dfc_ += da.T @ xn2
            dx_mid = dx + _rms_back(x_mid, r2, da @ w_fc)
            do_ += dx_mid.T @ att
            dO = G._split_heads(dx_mid @ wo, H, hd)
            dqn = np.empty_like(qn)
            dkn = np.zeros_like(kn)
            dv = np.zeros_like(v)
            for h in range(H):
                g = h // group
                dv[g] += P[h].T @ dO[h]
                dP = dO[h] @ v[g].T
                dS = P[h] * (dP - np.sum(dP * P[h], axis=-1, keepdims=True))
                dqn[h] = scale * (dS @ kn[g])
                dkn[g] += scale * (dS.T @ qn[h])
            dq = G._merge_heads(_rope_back(_rms_back(qr, rq, dqn), cos, sin))
            dk = G._merge_heads(_rope_back(_rms_back(kr, rk, dkn), cos, sin))
            dvm = G._merge_heads(dv)
            dq_ += dq.T @ xn1
            dk_ += dk.T @ xn1
            dv_ += dvm.T @ xn1
            dx = dx_mid + _rms_back(x_in, r1, dq @ wq + dk @ wk + dvm @ wv)
        np.add.at(d_wte, tokens[b], dx)
    loss = loss_sum / count if count else float("nan")
    return loss, {"wte": d_wte, "layers": [tuple(m) for m in d_layers], "lm_head": d_lm}


def adam_update(w, g, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8):
    """One Adam step (Kingma and Ba, "Adam: A Method for Stochastic Optimization",
    Algorithm 1) for parameter w with gradient g, moment estimates m, v and step
    count t >= 1 (this step's). The Microgpt summary (训练过程 item 4) says only that
    Adam keeps the mean of the gradients and the mean of their squares; the
    constants are the paper's defaults, a reading. Returns (w, m, v), new arrays:
      m = beta1 m + (1 - beta1) g,  v = beta2 v + (1 - beta2) g^2,
      w = w - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)."""
    g = np.asarray(g, dtype=F64)
    m = beta1 * np.asarray(m, dtype=F64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=F64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    return np.asarray(w, dtype=F64) - lr * m_hat / (np.sqrt(v_hat) + eps), m, v


def train_step(cfg, params, state, tokens, targets, lr):
    """One iteration of the summary's training loop (训练过程 items 2-4): forward
    pass and mean loss, gradients by backpropagation, one Adam step for every
    parameter. params: {"wte", "layers" (list of 6-tuples), "lm_head"}; state: None
    for the first step, else what the previous call returned. Returns (loss before
    the step, new params, new state)."""
    loss, g = loss_and_grads(cfg, params["wte"], params["layers"], params["lm_head"], tokens,
                             targets)
    flat_p = [params["wte"], params["lm_head"]] + [m for mats in params["layers"] for m in mats]
    flat_g = [g["wte"], g["lm_head"]] + [m for mats in g["layers"] for m in mats]
    if state is None:
        state = {"t": 0, "m": [np.zeros_like(p, dtype=F64) for p in flat_p],
                 "v": [np.zeros_like(p, dtype=F64) for p in flat_p]}
    t = state["t"] + 1
    new_p, new_m, new_v = [], [], []
    for p, gp, m, v in zip(flat_p, flat_g, state["m"], state["v"]):
        w, m, v = adam_update(p, gp, m, v, t, lr)
        new_p.append(w)
        new_m.append(m)
        new_v.append(v)
    n_l = len(params["layers"])
    out = {"wte": new_p[0], "lm_head": new_p[1],
           "layers": [tuple(new_p[2 + 6 * l: 8 + 6 * l]) for l in range(n_l)]}
    return loss, out, {"t": t, "m": new_m, "v": new_v}
