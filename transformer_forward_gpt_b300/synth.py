"""Seeded synthetic workloads: model shapes, random weights and token ids.

This module only describes and draws inputs. It holds none of the forward
pass's arithmetic, so both the CUDA path and the CPU oracle can be fed from it
without sharing any computation.

Shapes follow the nanochat-style GPT described on the pages (d_model = 64 x
depth, head_dim 128, 4x ReLU^2 MLP, vocabulary 65,536) and the microgpt summary
(vocabulary 27, width 16, one layer, four heads, block size 16).

Recipe:
  * numpy ``default_rng(seed)`` (PCG64); every matrix W[rows, cols] is drawn as
    float32 standard normals times 1/sqrt(cols) (std = 1/sqrt(fan_in)).
  * bf16 workloads round each draw to bfloat16 (round to nearest even); the
    fp32 workload keeps the float32 draw.
  * draw order: wte, then per layer wq, wk, wv, wo, w_fc, w_proj, then lm_head.
  * token ids: ``default_rng(seed + 1).integers(0, vocab, size=(B, T))``.
"""
from __future__ import annotations

import dataclasses
import numpy as np


@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    vocab: int
    d_model: int
    n_layer: int
    n_head: int
    n_kv_head: int
    head_dim: int
    d_mlp: int
    dtype: str                 # "f32" or "bf16": storage type of weights and activations
    rope_base: float = 10000.0
    rms_eps: float = 1e-5
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic job: a model shape plus batch / sequence sizes."""
    shape: ModelShape
    batch: int
    seq: int                   # prefill length
    decode_steps: int = 0      # greedy KV-cache decode steps after the prefill


TINY = ModelShape("tiny", vocab=27, d_model=16, n_layer=1, n_head=4, n_kv_head=4,
                  head_dim=4, d_mlp=64, dtype="f32", seed=0)
D12 = ModelShape("d12", vocab=65536, d_model=768, n_layer=12, n_head=6, n_kv_head=6,
                 head_dim=128, d_mlp=3072, dtype="bf16", seed=12)
D20 = ModelShape("d20", vocab=65536, d_model=1280, n_layer=20, n_head=10, n_kv_head=10,
                 head_dim=128, d_mlp=5120, dtype="bf16", seed=20)
D20_MQA = ModelShape("d20_mqa", vocab=65536, d_model=1280, n_layer=20, n_head=10, n_kv_head=1,
                     head_dim=128, d_mlp=5120, dtype="bf16", seed=2001)
D26 = ModelShape("d26", vocab=65536, d_model=1664, n_layer=26, n_head=13, n_kv_head=13,
                 head_dim=128, d_mlp=6656, dtype="bf16", seed=26)

SHAPES = {s.name: s for s in (TINY, D12, D20, D20_MQA, D26)}

WORKLOADS = {
    "tiny_prefill": Workload(TINY, batch=1, seq=16),
    "d12_prefill": Workload(D12, batch=8, seq=2048),
    "d20_prefill": Workload(D20, batch=4, seq=2048),
    "d20_mqa_decode": Workload(D20_MQA, batch=32, seq=1024, decode_steps=128),
    "d26_prefill": Workload(D26, batch=4, seq=2048),
    "d26_decode": Workload(D26, batch=64, seq=2048, decode_steps=64),
}


def with_changes(shape: ModelShape, **kw) -> ModelShape:
    """A copy of ``shape`` with some fields replaced (reduced test shapes)."""
    return dataclasses.replace(shape, **kw)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u = u + np.uint32(0x7FFF) + lsb
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> the exactly equal float32 values."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Weights:
    """Weights of one model, every matrix row-major [out, in].

    ``f32`` holds the values as float32 (exact for bf16 models). ``bits`` holds
    the bf16 bit patterns (uint16) for bf16 models, else None.
    Per layer: (wq [H*hd, d], wk [Hkv*hd, d], wv [Hkv*hd, d], wo [d, H*hd],
    w_fc [F, d], w_proj [d, F]).
    """
    shape: ModelShape
    wte: np.ndarray
    layers: list
    lm_head: np.ndarray
    bits: dict | None = None

    def matrices(self):
        """(name, array) pairs in draw order."""
        yield "wte", self.wte
        for l, mats in enumerate(self.layers):
            for n, m in zip(LAYER_MATRIX_NAMES, mats):
                yield f"layers.{l}.{n}", m
        yield "lm_head", self.lm_head


LAYER_MATRIX_NAMES = ("wq", "wk", "wv", "wo", "w_fc", "w_proj")


def layer_matrix_shapes(s: ModelShape):
    qd, kvd = s.n_head * s.head_dim, s.n_kv_head * s.head_dim
    return ((qd, s.d_model), (kvd, s.d_model), (kvd, s.d_model), (s.d_model, qd),
            (s.d_mlp, s.d_model), (s.d_model, s.d_mlp))


def _draw(rng, rows, cols, bf16):
    w = rng.standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(1.0 / np.sqrt(cols))
    if not bf16:
        return w, None
    b = round_to_bf16_bits(w)
    return bf16_bits_to_f32(b), b


def make_weights(s: ModelShape, seed: int | None = None) -> Weights:
    rng = np.random.default_rng(s.seed if seed is None else seed)
    bf16 = s.dtype == "bf16"
    bits = {} if bf16 else None
    wte, b = _draw(rng, s.vocab, s.d_model, bf16)
    if bf16:
        bits["wte"] = b
    layers = []
    for l in range(s.n_layer):
        mats = []
        for n, (r, c) in zip(LAYER_MATRIX_NAMES, layer_matrix_shapes(s)):
            w, b = _draw(rng, r, c, bf16)
            mats.append(w)
            if bf16:
                bits[f"layers.{l}.{n}"] = b
        layers.append(tuple(mats))
    lm, b = _draw(rng, s.vocab, s.d_model, bf16)
    if bf16:
        bits["lm_head"] = b
    return Weights(s, wte, layers, lm, bits)


def make_tokens(s: ModelShape, batch: int, seq: int, seed: int | None = None) -> np.ndarray:
    rng = np.random.default_rng((s.seed if seed is None else seed) + 1)
    return rng.integers(0, s.vocab, size=(batch, seq), dtype=np.int64).astype(np.int32)


def param_count(s: ModelShape) -> int:
    """Number of weight values of a shape (no gains, no biases, untied head)."""
    per_layer = sum(r * c for r, c in layer_matrix_shapes(s))
    return 2 * s.vocab * s.d_model + s.n_layer * per_layer
