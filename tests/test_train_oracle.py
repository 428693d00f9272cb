"""Pins of the backward-pass oracle (oracle/train_oracle.py) against facts that do not
come from its own code: the pinned forward oracle's loss, central finite differences
of that forward loss for entries of every parameter matrix, and the closed form of
the gradient when the LM head is zero."""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from oracle import train_oracle as TR
from transformer_forward_gpt_b300 import synth

SMALL_GQA = synth.ModelShape("small_gqa", vocab=61, d_model=32, n_layer=2, n_head=4,
                             n_kv_head=2, head_dim=8, d_mlp=128, dtype="f32", seed=5)


def _setup(shape, B, n, seed):
    W = synth.make_weights(shape)
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, shape.vocab, size=(B, n))
    tgt = rng.integers(0, shape.vocab, size=(B, n))
    tgt[0, 2] = -1                      # left out
    return W, toks, tgt


def _forward_loss(shape, wte, layers, lm, toks, tgt):
    logits, _ = O.prefill(shape, wte, layers, lm, toks)
    return O.cross_entropy(logits.reshape(-1, shape.vocab), tgt.reshape(-1))[1]


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_GQA])
def test_loss_is_the_forward_oracles(shape):
    W, toks, tgt = _setup(shape, 2, 7, 1)
    loss, _ = TR.loss_and_grads(shape, W.wte, W.layers, W.lm_head, toks, tgt)
    assert abs(loss - _forward_loss(shape, W.wte, W.layers, W.lm_head, toks, tgt)) < 1e-12


@pytest.mark.parametrize("shape,B,n", [(synth.TINY, 2, 8), (SMALL_GQA, 2, 6)])
def test_gradients_match_central_differences(shape, B, n):
    """Eight entries of every parameter matrix: (L(w + h) - L(w - h)) / 2h of the
    forward oracle's loss, h = 1e-5, against the analytic gradient."""
    W, toks, tgt = _setup(shape, B, n, 2)
    wte = W.wte.astype(np.float64)
    layers = [[m.astype(np.float64) for m in mats] for mats in W.layers]
    lm = W.lm_head.astype(np.float64)
    _, g = TR.loss_and_grads(shape, wte, layers, lm, toks, tgt)
    rng = np.random.default_rng(3)
    used = np.unique(toks)
    unused = np.setdiff1d(np.arange(shape.vocab), used)
    assert len(unused) and np.all(g["wte"][unused] == 0.0)

    def check(arr, grad, rows=None):
        for _ in range(8):
            r = int(rng.choice(rows)) if rows is not None else int(rng.integers(arr.shape[0]))
            c = int(rng.integers(arr.shape[1]))
            keep = arr[r, c]
            arr[r, c] = keep + 1e-5
            up = _forward_loss(shape, wte, layers, lm, toks, tgt)
            arr[r, c] = keep - 1e-5
            dn = _forward_loss(shape, wte, layers, lm, toks, tgt)
            arr[r, c] = keep
            fd = (up - dn) / 2e-5
            assert abs(fd - grad[r, c]) <= 1e-8 + 1e-5 * abs(fd), (arr.shape, r, c, fd, grad[r, c])

    check(wte, g["wte"], rows=used)
    check(lm, g["lm_head"])
    for l in range(shape.n_layer):
        for i in range(6):
            check(layers[l][i], g["layers"][l][i])


def test_zero_lm_head_gradient_in_closed_form():
    """With lm_head = 0 every logit is 0, so d loss / d z = (1/V - onehot) / count
    and d lm_head = sum over rows of that times the final-norm output. Nothing
    reaches the blocks or the embedding (d xn = d z lm_head = 0). The final-norm
    output is read off the forward oracle with an identity head (V >= d)."""
    shape = synth.TINY
    W, toks, tgt = _setup(shape, 2, 8, 4)
    V, d = shape.vocab, shape.d_model
    zero = np.zeros_like(W.lm_head)
    loss, g = TR.loss_and_grads(shape, W.wte, W.layers, zero, toks, tgt)
    assert abs(loss - np.log(V)) < 1e-12
    eye = np.zeros((V, d))
    eye[:d] = np.eye(d)
    xnf = O.prefill(shape, W.wte, W.layers, eye, toks)[0][..., :d].reshape(-1, d)
    t = tgt.reshape(-1)
    keep = t >= 0
    dz = np.full((len(t), V), 1.0 / V)
    dz[np.nonzero(keep)[0], t[keep]] -= 1.0
    dz[~keep] = 0.0
    dz /= keep.sum()
    assert np.allclose(g["lm_head"], dz.T @ xnf, rtol=0, atol=1e-14)
    assert not np.any(g["wte"]) and not any(np.any(m) for mats in g["layers"] for m in mats)


def test_adam_first_step_is_lr_times_sign():
    """At t = 1 the bias-corrected moments are g and g^2, so the step is
    lr g / (|g| + eps): lr times the sign of g up to eps."""
    g = np.array([3.0, -0.5, 1e-3, 0.0])
    w, m, v = TR.adam_update(np.zeros(4), g, np.zeros(4), np.zeros(4), 1, 0.01)
    assert np.allclose(w, -0.01 * g / (np.abs(g) + 1e-8), rtol=1e-15, atol=0)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)
    assert w[3] == 0.0


def test_adam_constant_gradient_takes_equal_steps():
    """With the same gradient every step, m_hat = g and v_hat = g^2 at every t."""
    g = np.array([0.7, -2.0])
    w, m, v = np.zeros(2), np.zeros(2), np.zeros(2)
    prev = w
    for t in range(1, 30):
        w, m, v = TR.adam_update(w, g, m, v, t, 0.05)
        assert np.allclose(w - prev, -0.05 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=0)
        prev = w


def test_adam_minimises_a_quadratic():
    w, m, v = np.array([0.0]), np.zeros(1), np.zeros(1)
    for t in range(1, 3001):
        w, m, v = TR.adam_update(w, w - 3.0, m, v, t, 0.01)   # gradient of (w - 3)^2 / 2
    assert abs(w[0] - 3.0) < 1e-3


def test_training_steps_lower_the_loss():
    """A few steps of the loop on the tiny model and one batch: the loss falls at
    each step, and the parameters move only where the gradient is nonzero."""
    shape = synth.TINY
    W, toks, tgt = _setup(shape, 2, 8, 6)
    params = {"wte": W.wte, "layers": W.layers, "lm_head": W.lm_head}
    state = None
    losses = []
    for _ in range(5):
        loss, new, state = TR.train_step(shape, params, state, toks, tgt, 1e-2)
        losses.append(loss)
        unused = np.setdiff1d(np.arange(shape.vocab), np.unique(toks))
        assert np.array_equal(new["wte"][unused], np.asarray(params["wte"], np.float64)[unused])
        params = new
    assert all(b < a for a, b in zip(losses, losses[1:])), losses
