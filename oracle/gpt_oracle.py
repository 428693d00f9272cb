"""fp64 CPU oracle of the nanochat-style GPT forward pass (prefill and decode).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline may import this module. The product path (the CUDA library and its
Python binding) never calls it, and it shares no code with that path.

What it computes, in the order the pages give it:

* token embedding lookup, no position table -- rotary embeddings carry the
  position instead (Microgpt summary, telegra.ph, section 核心架构 item 3, and
  section 与生产级模型的区别 item 3 naming RoPE);
* RMSNorm without gain or bias (Microgpt summary, 核心架构 opening sentence;
  模型参数 item 1 lists only matrices as parameters);
* separate Q, K, V linear layers (復刻 ChatGPT 有多難？, jxzklqfsx.com, section
  為什么可以訓練如此之快, the causal self-attention paragraph);
* rotary embedding that splits each head vector into two halves and rotates
  them as pairs, with cos/sin tables computed ahead of time (same section, the
  RoPE paragraph and the precomputed rotary embedding paragraph);
* QK normalisation (8000行手写代码！nanochat, hongdingcd.com, the paragraph on
  the model architecture: dense Transformer, rotary embeddings, QK norm);
* causal attention with multi-query / grouped-query head sharing
  (Microgpt summary, 核心架构 item 4; hongdingcd.com, the MQA/KV-cache
  paragraph);
* softmax into probabilities in [0, 1] summing to 1 (核心架构 item 2);
* output projection plus residual (核心架构 item 6);
* two-layer MLP with ReLU^2 (jxzklqfsx.com, the ReLU2 paragraph; 核心架构
  item 5) plus residual;
* final norm and an untied LM head (模型参数 item 1: embedding table and final
  output projection are separate matrices);
* KV cache: decode appends one position and attends over the cache
  (jxzklqfsx.com, the KV cache paragraph; CSDN nanochat article,
  wap.jaobe.com, the Engine paragraph with prefill and decode);
* greedy next token: argmax of the logits, lowest index on ties (Microgpt
  summary, 推理 section; greedy is the zero-temperature limit);
* the training step's loss: the cross-entropy between each position's predicted
  distribution and the true next token (Microgpt summary, 训练过程 item 2).

Readings where the pages are silent: eps = cfg["rms_eps"] (1e-5 in the
workloads); attention scale 1/sqrt(head_dim); RoPE rotates the pair
(i, i + hd/2) by +theta with theta = pos * base^(-2i/hd), positions from 0;
RoPE is applied before the QK norm; query head h reads KV head
h // (H / Hkv); the cache holds K after RoPE and norm and V as projected.

Weights arrive as float arrays (bf16 values are exact in float32); every
product here is evaluated in float64. A matmul from numpy is used as a step;
nothing is blocked, fused or reordered beyond the definitions above.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def rmsnorm(x, eps):
    """x / sqrt(mean(x^2) + eps) along the last axis; no learned gain."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def rope_tables(n_pos, head_dim, base):
    """cos and sin of theta[t, i] = t * base^(-2 i / head_dim), i < head_dim/2.

    Parameter-free tables that the pages say are computed once ahead of time.
    """
    half = head_dim // 2
    i = np.arange(half, dtype=F64)
    inv_freq = np.power(F64(base), -2.0 * i / head_dim)
    theta = np.arange(n_pos, dtype=F64)[:, None] * inv_freq[None, :]
    return np.cos(theta), np.sin(theta)


def apply_rope(x, cos, sin):
    """Rotate the two halves of each head vector as pairs (i, i + hd/2).

    x: [..., n, hd]; cos, sin: [n, hd/2] for the n positions of x.
    y_i = x_i cos - x_{i+h} sin ;  y_{i+h} = x_i sin + x_{i+h} cos.
    """
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x1 * sin + x2 * cos], axis=-1)


def softmax_rows(s):
    """Two-pass softmax along the last axis (max, then exp and sum).

    Entries equal to -inf get probability 0.
    """
    m = np.max(s, axis=-1, keepdims=True)
    p = np.exp(s - m)
    return p / np.sum(p, axis=-1, keepdims=True)


def attend(q, q_pos, k, v, return_probs=False):
    """Causal attention of one sequence.

    q: [H, n, hd] queries at absolute positions q_pos [n];
    k, v: [Hkv, S, hd] keys / values at positions 0..S-1.
    Query at position t sees keys s <= t. Query head h reads KV head
    h // (H // Hkv) (contiguous groups).
    Returns o [H, n, hd] (and the probabilities [H, n, S] if asked).
    """
    H, n, hd = q.shape
    Hkv, S, _ = k.shape
    group = H // Hkv
    allowed = np.arange(S)[None, :] <= np.asarray(q_pos)[:, None]      # [n, S]
    o = np.empty((H, n, hd), dtype=F64)
    probs = np.empty((H, n, S), dtype=F64) if return_probs else None
    for h in range(H):
        g = h // group
        s = (q[h] @ k[g].T) / np.sqrt(F64(hd))
        s = np.where(allowed, s, -np.inf)
        p = softmax_rows(s)
        o[h] = p @ v[g]
        if return_probs:
            probs[h] = p
    return (o, probs) if return_probs else o


def linear(x, w):
    """y = x W^T for a row-major [out, in] weight."""
    return np.asarray(x, dtype=F64) @ np.asarray(w, dtype=F64).T


def relu2(x):
    return np.square(np.maximum(x, 0.0))


def _split_heads(y, n_heads, hd):
    """[n, n_heads*hd] -> [n_heads, n, hd]; head j owns columns [j*hd, (j+1)*hd)."""
    return y.reshape(y.shape[0], n_heads, hd).transpose(1, 0, 2)


def _merge_heads(o):
    """[n_heads, n, hd] -> [n, n_heads*hd]."""
    return o.transpose(1, 0, 2).reshape(o.shape[1], -1)


class KVCache:
    """fp64 cache, per layer k/v of shape [B, Hkv, T_cap, hd]; ``length`` positions filled."""

    def __init__(self, cfg, batch, t_cap):
        shp = (batch, cfg["n_kv_head"], t_cap, cfg["head_dim"])
        self.k = [np.zeros(shp, dtype=F64) for _ in range(cfg["n_layer"])]
        self.v = [np.zeros(shp, dtype=F64) for _ in range(cfg["n_layer"])]
        self.length = 0


def _block(cfg, layer_w, x, positions, k_all, v_all, cos, sin, trace=None):
    """One transformer block for one sequence.

    x: [n, d] residual stream at absolute ``positions`` [n]; k_all/v_all
    [Hkv, S, hd] are this sequence's cache arrays for the layer, already holding
    positions < positions[0]; the block writes its own K/V rows into them and
    attends over positions 0..positions[-1].
    """
    wq, wk, wv, wo, w_fc, w_proj = layer_w
    H, Hkv, hd, eps = cfg["n_head"], cfg["n_kv_head"], cfg["head_dim"], cfg["rms_eps"]
    xn = rmsnorm(x, eps)
    q = _split_heads(linear(xn, wq), H, hd)
    k = _split_heads(linear(xn, wk), Hkv, hd)
    v = _split_heads(linear(xn, wv), Hkv, hd)
    q = rmsnorm(apply_rope(q, cos, sin), eps)        # RoPE, then QK norm
    k = rmsnorm(apply_rope(k, cos, sin), eps)
    k_all[:, positions, :] = k
    v_all[:, positions, :] = v
    S = int(positions[-1]) + 1
    o = attend(q, positions, k_all[:, :S], v_all[:, :S])
    x = x + linear(_merge_heads(o), wo)
    hmid = relu2(linear(rmsnorm(x, eps), w_fc))
    x = x + linear(hmid, w_proj)
    if trace is not None:
        trace.append(x.copy())
    return x


def _cfg(shape):
    """Accept a dict or any object with the shape attributes."""
    if isinstance(shape, dict):
        return shape
    keys = ("vocab", "d_model", "n_layer", "n_head", "n_kv_head", "head_dim",
            "d_mlp", "rope_base", "rms_eps")
    return {k: getattr(shape, k) for k in keys}


def _check_weights(cfg, wte, layers, lm_head):
    d, H, Hkv, hd, F = (cfg[k] for k in ("d_model", "n_head", "n_kv_head", "head_dim", "d_mlp"))
    assert wte.shape == (cfg["vocab"], d) and lm_head.shape == (cfg["vocab"], d)
    assert len(layers) == cfg["n_layer"]
    want = ((H * hd, d), (Hkv * hd, d), (Hkv * hd, d), (d, H * hd), (F, d), (d, F))
    for mats in layers:
        assert tuple(m.shape for m in mats) == want
    assert H % Hkv == 0 and hd % 2 == 0


def forward(cfg, wte, layers, lm_head, tokens, cache=None, start=0, logit_positions=None,
            trace=None):
    """Run ``tokens`` [B, n] at positions start..start+n-1 through the model.

    With ``start`` = 0 this is the prefill; with n = 1 and ``start`` = pos it is
    one decode step. ``cache`` (a KVCache) receives every position's K/V and
    supplies the earlier ones. ``logit_positions`` (indices into 0..n-1) limits
    the LM head to those rows. Returns logits [B, n or len(logit_positions), V].
    """
    cfg = _cfg(cfg)
    _check_weights(cfg, wte, layers, lm_head)
    tokens = np.asarray(tokens)
    B, n = tokens.shape
    if cache is None:
        cache = KVCache(cfg, B, start + n)
    assert cache.length == start and start + n <= cache.k[0].shape[2]
    positions = np.arange(start, start + n)
    cos, sin = rope_tables(start + n, cfg["head_dim"], cfg["rope_base"])
    cos, sin = cos[positions], sin[positions]
    rows = np.arange(n) if logit_positions is None else np.asarray(logit_positions)
    out = np.empty((B, len(rows), cfg["vocab"]), dtype=F64)
    lm = np.asarray(lm_head, dtype=F64)
    for b in range(B):
        x = np.asarray(wte[tokens[b]], dtype=F64)           # embedding rows [n, d]
        tr = [] if trace is not None else None
        for l, layer_w in enumerate(layers):
            x = _block(cfg, layer_w, x, positions, cache.k[l][b], cache.v[l][b], cos, sin, tr)
        out[b] = rmsnorm(x[rows], cfg["rms_eps"]) @ lm.T
        if trace is not None:
            trace.append(tr)
    cache.length = start + n
    return out


def prefill(cfg, wte, layers, lm_head, tokens, t_cap=None, logit_positions=None, trace=None):
    """Full-sequence forward from position 0; returns (logits, cache)."""
    cfg = _cfg(cfg)
    B, T = np.asarray(tokens).shape
    cache = KVCache(cfg, B, T if t_cap is None else t_cap)
    logits = forward(cfg, wte, layers, lm_head, tokens, cache, 0, logit_positions, trace)
    return logits, cache


def decode_step(cfg, wte, layers, lm_head, tokens, cache):
    """One token per sequence at position cache.length; returns logits [B, V]."""
    tokens = np.asarray(tokens).reshape(-1, 1)
    return forward(cfg, wte, layers, lm_head, tokens, cache, cache.length)[:, 0, :]


def greedy_next(logits):
    """Index of the largest logit in each row; ties go to the lowest index."""
    return np.argmax(np.asarray(logits), axis=-1)


def sample_temperature(logits, temperature, u):
    """One draw per row from the softmax of logits / temperature, by inverse CDF.

    Follows the Microgpt summary, section 推理（生成）: item 1 draws the next token
    from the predicted distribution, item 2 divides by a temperature (lower values
    sharpen the distribution, higher ones flatten it). The random number is an
    input: u[b] in [0, 1) selects the smallest index k whose cumulative
    probability exceeds u[b] (the last index if rounding leaves the total below
    u[b]). A temperature <= 0 is the zero-temperature limit: the greedy index.
    """
    logits = np.asarray(logits, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64).reshape(-1)
    if temperature <= 0:
        return greedy_next(logits)
    p = softmax_rows(logits / float(temperature))
    cdf = np.cumsum(p, axis=-1)
    out = np.empty(logits.shape[0], dtype=np.int64)
    for b in range(logits.shape[0]):
        k = int(np.searchsorted(cdf[b], u[b], side="right"))
        out[b] = min(k, logits.shape[1] - 1)
    return out


def cross_entropy(logits, targets):
    """Next-token loss of each row and their mean (Microgpt summary, 训练过程
    item 2: the cross-entropy between the model's prediction and the true token,
    a measure of how surprised the model is).

    loss[r] = -log p_r[targets[r]] with p_r = softmax(logits[r]) (核心架构 item 2),
    written as log(sum_v exp(z[r, v] - m_r)) + m_r - z[r, targets[r]] with m_r the
    row max, so that no exponential overflows. Reading where the pages are
    silent: a row whose target is negative is ignored (loss 0, not counted in the
    mean). Returns (loss [R], mean over counted rows; NaN if none counts).
    """
    z = np.asarray(logits, dtype=F64)
    t = np.asarray(targets).reshape(-1)
    assert z.ndim == 2 and z.shape[0] == t.shape[0]
    keep = t >= 0
    assert np.all(t[keep] < z.shape[1])
    m = z.max(axis=1)
    lse = np.log(np.sum(np.exp(z - m[:, None]), axis=1)) + m
    loss = np.zeros(z.shape[0], dtype=F64)
    rows = np.nonzero(keep)[0]
    loss[rows] = lse[rows] - z[rows, t[rows]]
    mean = float(np.sum(loss[rows]) / len(rows)) if len(rows) else float("nan")
    return loss, mean
