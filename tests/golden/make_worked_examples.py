"""Writes worked_examples.json: hand-derived closed forms, evaluated with math only.

Each entry states the passage it follows and the derivation. Nothing here
calls the oracle or the CUDA path.
"""
import json
import math
import os

s13, s25, s15 = math.sqrt(13.0), math.sqrt(2.5), math.sqrt(1.5)
c2, s2, c02, s02 = math.cos(2.0), math.sin(2.0), math.cos(0.02), math.sin(0.02)

examples = {
    "rmsnorm": {
        "cite": "Microgpt summary (telegra.ph), 核心架构: RMSNorm replaces LayerNorm; no gain (模型参数 item 1)",
        "derivation": "x=[3,4], eps=0.5: mean(x^2)+eps = 12.5+0.5 = 13, y = x/sqrt(13)",
        "x": [3.0, 4.0], "eps": 0.5, "y": [3 / s13, 4 / s13],
    },
    "rope": {
        "cite": "復刻 ChatGPT 有多難？ (jxzklqfsx.com), 為什么可以訓練如此之快: split the vector in two halves, rotate, concatenate",
        "derivation": "hd=4, base=1e4, pos=2: theta_0 = 2, theta_1 = 2*1e4^(-1/2) = 0.02; pairs (x0,x2) and (x1,x3) rotated by +theta",
        "x": [1.0, 2.0, 3.0, 4.0], "pos": 2, "base": 10000.0,
        "y": [1 * c2 - 3 * s2, 2 * c02 - 4 * s02, 1 * s2 + 3 * c2, 2 * s02 + 4 * c02],
    },
    "attention": {
        "cite": "Microgpt summary, 核心架构 items 2 and 4: softmax weights over the current and earlier positions",
        "derivation": "hd=2 (scale 1/sqrt2); q1=[sqrt2 ln3,0], k0=0, k1=[1,0]: scores of position 1 are [0, ln3] -> p=[1/4,3/4]; o1 = v0/4 + 3 v1/4; position 0 sees only k0",
        "q": [[0.0, 0.0], [math.sqrt(2.0) * math.log(3.0), 0.0]],
        "k": [[0.0, 0.0], [1.0, 0.0]],
        "v": [[4.0, 0.0], [0.0, 8.0]],
        "probs": [[1.0, 0.0], [0.25, 0.75]],
        "o": [[4.0, 0.0], [1.0, 6.0]],
    },
    "residual_only_logits": {
        "cite": "Microgpt summary, 核心架构 item 6 (residual) and 模型参数 item 1 (untied output projection)",
        "derivation": "with W_o = W_proj = 0 the residual stream stays the embedding row; logits = rmsnorm(row) . lm_head^T, eps=0.5",
        "eps": 0.5,
        "wte": [[3.0, 4.0], [1.0, -1.0], [0.0, 2.0]],
        "lm_head": [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]],
        "tokens": [0, 2, 1],
        "logits": [[3 / s13, 4 / s13, 7 / s13], [0.0, 2 / s25, 2 / s25], [1 / s15, -1 / s15, 0.0]],
    },
}

if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_examples.json")
    with open(out, "w") as f:
        json.dump(examples, f, indent=1, ensure_ascii=False)
