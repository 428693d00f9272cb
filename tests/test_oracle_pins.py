"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test names the passage it follows. Together they are chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign, a wrong head or
pair index, a transposed weight, a missing scale or eps) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import gpt_oracle as O
from transformer_forward_gpt_b300 import synth
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cfg(shape):
    return O._cfg(shape)


def _weights(shape, seed=None):
    w = synth.make_weights(shape, seed)
    return w.wte, w.layers, w.lm_head


def _small(**kw):
    """A reduced shape for invariants (few layers, small vocab)."""
    base = dict(name="small", vocab=61, d_model=32, n_layer=2, n_head=4, n_kv_head=2,
                head_dim=8, d_mlp=128, dtype="f32", seed=5)
    base.update(kw)
    return synth.ModelShape(**base)


# ---------------------------------------------------------------- worked examples
def test_golden_worked_examples():
    """Hand-derived values (tests/golden/worked_examples.json), each cited there."""
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        g = json.load(f)
    r = g["rmsnorm"]
    np.testing.assert_allclose(O.rmsnorm(np.array(r["x"]), r["eps"]), r["y"], rtol=0, atol=1e-12)
    r = g["rope"]
    cos, sin = O.rope_tables(r["pos"] + 1, len(r["x"]), r["base"])
    y = O.apply_rope(np.array([r["x"]], dtype=float), cos[r["pos"]:r["pos"] + 1],
                     sin[r["pos"]:r["pos"] + 1])[0]
    np.testing.assert_allclose(y, r["y"], rtol=0, atol=1e-12)
    a = g["attention"]
    q = np.array(a["q"], dtype=float)[None]
    k = np.array(a["k"], dtype=float)[None]
    v = np.array(a["v"], dtype=float)[None]
    o, p = O.attend(q, np.arange(q.shape[1]), k, v, return_probs=True)
    np.testing.assert_allclose(p[0], a["probs"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[0], a["o"], rtol=0, atol=1e-12)
    m = g["residual_only_logits"]
    cfg = dict(vocab=3, d_model=2, n_layer=1, n_head=1, n_kv_head=1, head_dim=2, d_mlp=8,
               rope_base=10000.0, rms_eps=m["eps"])
    wte = np.array(m["wte"], dtype=float)
    lm = np.array(m["lm_head"], dtype=float)
    rng = np.random.default_rng(0)
    layer = (rng.standard_normal((2, 2)), rng.standard_normal((2, 2)),
             rng.standard_normal((2, 2)), np.zeros((2, 2)),
             rng.standard_normal((8, 2)), np.zeros((2, 8)))
    logits, _ = O.prefill(cfg, wte, [layer], lm, np.array([m["tokens"]]))
    np.testing.assert_allclose(logits[0], m["logits"], rtol=0, atol=1e-12)


def test_rmsnorm_zero_row_is_zero():
    """x = 0 gives 0 (the eps keeps the denominator positive)."""
    assert np.all(O.rmsnorm(np.zeros((2, 8)), 1e-5) == 0)


# ------------------------------------------------------------------------- RoPE
def test_rope_preserves_norm_and_is_identity_at_zero():
    """Rotation of pairs keeps each head vector's length (RoPE paragraph)."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 50, 128))
    cos, sin = O.rope_tables(50, 128, 10000.0)
    y = O.apply_rope(x, cos, sin)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])


def test_rope_scores_depend_only_on_offset():
    """<R(m) q, R(n) k> is a function of m - n only."""
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    cos, sin = O.rope_tables(300, 64, 10000.0)

    def rot(x, t):
        return O.apply_rope(x[None], cos[t:t + 1], sin[t:t + 1])[0]
    for m, n, c in [(7, 3, 100), (40, 40, 250), (0, 5, 17)]:
        assert abs(rot(q, m) @ rot(k, n) - rot(q, m + c) @ rot(k, n + c)) < 1e-11


# -------------------------------------------------------------------- attention
def test_softmax_rows_are_probabilities():
    """Probabilities lie in [0, 1] and each row sums to 1 (核心架构 item 2)."""
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((4, 33, 16)) * 3 for _ in range(3))
    _, p = O.attend(q, np.arange(33), k, v, return_probs=True)
    assert np.all(p >= 0) and np.all(p <= 1)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-13)
    assert np.all(np.triu(p, 1) == 0)          # no weight on later positions


def test_length_one_attention_returns_v():
    """One key: its softmax weight is 1, so the output is that position's V."""
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((6, 1, 8)), rng.standard_normal((3, 1, 8)), rng.standard_normal((3, 1, 8))
    o = O.attend(q, np.array([0]), k, v)
    for h in range(6):
        np.testing.assert_array_equal(o[h], v[h // 2])


def test_grouped_query_heads_share_contiguous_kv_heads():
    """Query heads 0,1 read KV head 0 and heads 2,3 read KV head 1 (GQA)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 5, 8))
    k = rng.standard_normal((2, 5, 8))
    v = np.stack([np.full((5, 8), 1.0), np.full((5, 8), -1.0)])
    o = O.attend(q, np.arange(5), k, v)
    np.testing.assert_allclose(o[:2], 1.0, atol=1e-14)
    np.testing.assert_allclose(o[2:], -1.0, atol=1e-14)


# ----------------------------------------------------------------- whole model
@pytest.mark.parametrize("shape", [synth.TINY, _small(), _small(n_kv_head=1, seed=6)])
def test_bruteforce_loops_match_oracle(shape):
    """Position-by-position pure-Python loops agree with the vectorised oracle."""
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    toks = synth.make_tokens(shape, 1, 9)[0].tolist()
    ref = np.array(bruteforce.forward_positions(cfg, wte, layers, lm, toks))
    got, _ = O.prefill(cfg, wte, layers, lm, np.array([toks]))
    np.testing.assert_allclose(got[0], ref, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("shape", [synth.TINY, _small()])
def test_causality_future_tokens_do_not_change_earlier_logits(shape):
    """Each position sees only itself and earlier positions (核心架构 item 4)."""
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    toks = synth.make_tokens(shape, 1, 12)
    a, _ = O.prefill(cfg, wte, layers, lm, toks)
    toks2 = toks.copy()
    toks2[0, 7:] = (toks2[0, 7:] + 1) % shape.vocab
    b, _ = O.prefill(cfg, wte, layers, lm, toks2)
    np.testing.assert_array_equal(a[0, :7], b[0, :7])
    assert np.abs(a[0, 7:] - b[0, 7:]).max() > 1e-3


@pytest.mark.parametrize("shape", [synth.TINY, _small(),
                                   synth.with_changes(synth.D20_MQA, n_layer=2, vocab=257)])
def test_decode_with_cache_equals_prefill(shape):
    """Decode at position p with the KV cache gives prefill's logits at p
    (KV cache paragraph; Engine with prefill and decode)."""
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    T0, steps = 5, 4
    toks = synth.make_tokens(shape, 2, T0 + steps)
    full, _ = O.prefill(cfg, wte, layers, lm, toks)
    pre, cache = O.prefill(cfg, wte, layers, lm, toks[:, :T0], t_cap=T0 + steps)
    np.testing.assert_allclose(pre, full[:, :T0], rtol=0, atol=1e-12)
    for j in range(steps):
        lg = O.decode_step(cfg, wte, layers, lm, toks[:, T0 + j], cache)
        np.testing.assert_allclose(lg, full[:, T0 + j], rtol=0, atol=1e-11)
    assert cache.length == T0 + steps


def test_mqa_equals_mha_with_replicated_kv_heads():
    """One shared KV head (MQA) == MHA whose K/V weights repeat that head."""
    mqa = _small(n_kv_head=1, seed=8)
    cfg = _cfg(mqa)
    wte, layers, lm = _weights(mqa)
    hd, H = mqa.head_dim, mqa.n_head
    mha_layers = [(wq, np.tile(wk, (H, 1)), np.tile(wv, (H, 1)), wo, wf, wp)
                  for (wq, wk, wv, wo, wf, wp) in layers]
    cfg_mha = dict(cfg, n_kv_head=H)
    toks = synth.make_tokens(mqa, 2, 10)
    a, _ = O.prefill(cfg, wte, layers, lm, toks)
    b, _ = O.prefill(cfg_mha, wte, mha_layers, lm, toks)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_batch_rows_are_independent():
    shape = _small()
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    toks = synth.make_tokens(shape, 3, 8)
    a, _ = O.prefill(cfg, wte, layers, lm, toks)
    for b in range(3):
        one, _ = O.prefill(cfg, wte, layers, lm, toks[b:b + 1])
        np.testing.assert_array_equal(one[0], a[b])


def test_cached_k_is_unit_rms_and_v_is_layer0_projection():
    """QK norm leaves each cached key head with mean square ~1; V is cached as
    projected (layer 0: V = rmsnorm(embedding) W_v^T)."""
    shape = _small()
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    toks = synth.make_tokens(shape, 1, 6)
    _, cache = O.prefill(cfg, wte, layers, lm, toks)
    for l in range(shape.n_layer):
        ms = np.mean(cache.k[l] ** 2, axis=-1)
        assert np.all(np.abs(ms - 1) < 1e-3)
    xn = O.rmsnorm(wte[toks[0]].astype(float), shape.rms_eps)
    v0 = xn @ layers[0][2].astype(float).T
    np.testing.assert_allclose(cache.v[0][0].transpose(1, 0, 2).reshape(6, -1), v0, atol=1e-13)


def test_relu2_mlp_closed_form():
    """With attention output zeroed, one block adds W2 relu(W1 n(x))^2 to x
    (ReLU2 paragraph; 核心架构 items 5 and 6). Selector weights make it exact:
    h = [relu(a)^2, relu(-a)^2] for a = n(x)_0, added back to coordinates 0, 1."""
    cfg = dict(vocab=2, d_model=2, n_layer=1, n_head=1, n_kv_head=1, head_dim=2, d_mlp=2,
               rope_base=10000.0, rms_eps=0.0)
    wte = np.array([[3.0, 4.0], [-1.0, 0.0]])
    lm = np.eye(2)
    z = np.zeros((2, 2))
    layer = (np.eye(2), np.eye(2), np.eye(2), z, np.array([[1.0, 0.0], [-1.0, 0.0]]), np.eye(2))
    logits, _ = O.prefill(cfg, wte, [layer], lm, np.array([[0, 1]]))
    for pos, row in enumerate(wte):
        n = row / math.sqrt(np.mean(row ** 2))
        x = row + np.array([max(n[0], 0) ** 2, max(-n[0], 0) ** 2])
        want = x / math.sqrt(np.mean(x ** 2))
        np.testing.assert_allclose(logits[0, pos], want, atol=1e-13)


def test_microgpt_parameter_count():
    """The microgpt summary (模型参数 item 2) counts 4,192 parameters for vocab 27,
    width 16, one layer, four heads, MLP 64, block size 16. The tiny shape is that
    model with the learned position table (16 x 16) replaced by RoPE."""
    assert synth.param_count(synth.TINY) == 4192 - 16 * 16
    cfg = _cfg(synth.TINY)
    wte, layers, lm = _weights(synth.TINY)
    O._check_weights(cfg, wte, layers, lm)        # the oracle consumes exactly these
    n = wte.size + lm.size + sum(m.size for mats in layers for m in mats)
    assert n == 3936


def test_uniform_prediction_cross_entropy_is_ln27():
    """A zeroed LM head gives equal logits; the loss of uniform guessing over 27
    tokens is ln 27 = 3.2958, the microgpt summary's "about 3.3" (训练过程)."""
    shape = synth.TINY
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    logits, _ = O.prefill(cfg, wte, layers, np.zeros_like(lm), synth.make_tokens(shape, 1, 16))
    assert np.all(logits == 0)
    lse = np.log(np.sum(np.exp(logits[0]), axis=-1))
    targets = synth.make_tokens(shape, 1, 16)[0, 1:]
    ce = np.mean(lse[:15] - logits[0, np.arange(15), targets])
    assert abs(ce - math.log(27)) < 1e-12 and round(ce, 1) == 3.3


def test_greedy_ties_go_to_lowest_index():
    lg = np.array([[0.0, 2.0, 2.0, 1.0], [5.0, 5.0, 5.0, 5.0]])
    assert O.greedy_next(lg).tolist() == [1, 0]


def test_bf16_rounding_of_inputs():
    """Input generator rounds to nearest even bf16 (ties to even, exact values kept)."""
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3], dtype=np.float32)
    y = synth.bf16_bits_to_f32(synth.round_to_bf16_bits(x))
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == 1.0 + 2 ** -6 and y[3] == -2.5
    assert abs(y[4] - 1e-3) <= 1e-3 * 2 ** -8


# ---------------------------------------------------------- temperature sampling
# Microgpt summary, section 推理（生成）: draw from the predicted distribution;
# the temperature sharpens (low) or flattens (high) it.

def test_sampling_two_classes_closed_form():
    """Two logits a, b: P(first) = 1 / (1 + e^((b - a) / T)), so u just below that
    probability picks index 0 and u just above picks index 1."""
    for a, b, T in [(0.3, -1.2, 0.7), (2.0, 2.5, 1.0), (-1.0, 3.0, 2.5)]:
        p0 = 1.0 / (1.0 + math.exp((b - a) / T))
        lo, hi = p0 * (1 - 1e-9), p0 * (1 + 1e-9)
        ks = O.sample_temperature(np.array([[a, b], [a, b]]), T, np.array([lo, hi]))
        assert ks.tolist() == [0, 1]


def test_sampling_uniform_logits_picks_floor_u_times_v():
    """Equal logits at any temperature: every index has probability 1/V, so u
    selects floor(u V) (u placed mid-interval, away from the boundaries)."""
    V = 97
    j = np.arange(V)
    u = (j + 0.5) / V
    ks = O.sample_temperature(np.full((V, V), 1.25), 0.8, u)
    assert (ks == j).all()


def test_sampling_inverse_cdf_frequencies():
    """A uniform grid of N values of u lands in class k about p_k N times (within
    one), the defining property of inverse-CDF sampling."""
    rng = np.random.default_rng(11)
    logits = rng.standard_normal(12) * 2.0
    T = 1.3
    z = np.exp((logits - logits.max()) / T)
    p = z / z.sum()
    N = 20000
    u = (np.arange(N) + 0.5) / N
    ks = O.sample_temperature(np.tile(logits, (N, 1)), T, u)
    counts = np.bincount(ks, minlength=12)
    assert np.all(np.abs(counts - p * N) <= 1.0)


def test_sampling_low_temperature_is_greedy_and_zero_is_greedy():
    """As T -> 0 the distribution concentrates on the largest logit; T <= 0 is
    the greedy limit itself (lowest index on ties)."""
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((6, 50))
    u = rng.random(6)
    assert (O.sample_temperature(logits, 1e-4, u) == np.argmax(logits, axis=1)).all()
    tied = np.array([[1.0, 3.0, 3.0, 0.0]])
    assert O.sample_temperature(tied, 0.0, np.array([0.9])).tolist() == [1]


def test_prefill_in_chunks_equals_one_prefill():
    """Running a prompt in pieces through the KV cache gives the one-shot prefill's
    logits and cache (KV cache paragraph: earlier positions are read back, not
    recomputed)."""
    shape = _small(n_kv_head=1)
    cfg = _cfg(shape)
    wte, layers, lm = _weights(shape)
    toks = synth.make_tokens(shape, 2, 9)
    full, fcache = O.prefill(cfg, wte, layers, lm, toks)
    cache = O.KVCache(cfg, 2, 9)
    parts = []
    for a, b in [(0, 3), (3, 7), (7, 9)]:
        parts.append(O.forward(cfg, wte, layers, lm, toks[:, a:b], cache, a))
    np.testing.assert_allclose(np.concatenate(parts, axis=1), full, rtol=0, atol=1e-11)
    for l in range(cfg["n_layer"]):
        np.testing.assert_allclose(cache.k[l], fcache.k[l], rtol=0, atol=1e-12)
        np.testing.assert_allclose(cache.v[l], fcache.v[l], rtol=0, atol=1e-12)
    assert cache.length == 9


# ----------------------------------------------------------- cross-entropy loss
def test_cross_entropy_two_classes_by_hand():
    """z = (0, ln 3): p = (1/4, 3/4), so the loss is ln 4 for target 0 and
    ln(4/3) for target 1."""
    z = np.array([[0.0, math.log(3.0)], [0.0, math.log(3.0)]])
    loss, mean = O.cross_entropy(z, np.array([0, 1]))
    assert abs(loss[0] - math.log(4.0)) < 1e-15
    assert abs(loss[1] - math.log(4.0 / 3.0)) < 1e-15
    assert abs(mean - (math.log(4.0) + math.log(4.0 / 3.0)) / 2) < 1e-15


def test_cross_entropy_of_uniform_logits_is_ln_v():
    for V in (2, 27, 1000, 65536):
        z = np.full((3, V), 1.7)
        loss, _ = O.cross_entropy(z, np.array([0, V // 2, V - 1]))
        assert np.allclose(loss, math.log(V), rtol=0, atol=1e-12)


def test_cross_entropy_matches_minus_log_probability_brute_force():
    """Pure-Python loops: p = exp(z_t) / sum exp(z_v), loss = -log p."""
    rng = np.random.default_rng(31)
    z = rng.standard_normal((6, 9)) * 3
    t = rng.integers(0, 9, size=6)
    loss, mean = O.cross_entropy(z, t)
    want = []
    for r in range(6):
        den = sum(math.exp(float(v)) for v in z[r])
        want.append(-math.log(math.exp(float(z[r, t[r]])) / den))
    assert np.allclose(loss, want, rtol=1e-13, atol=0)
    assert abs(mean - sum(want) / 6) < 1e-13


def test_cross_entropy_shift_invariance_and_no_overflow():
    rng = np.random.default_rng(32)
    z = rng.standard_normal((4, 50))
    t = rng.integers(0, 50, size=4)
    a, _ = O.cross_entropy(z, t)
    b, _ = O.cross_entropy(z + np.array([[1000.0], [-1000.0], [3.5], [0.0]]), t)
    assert np.allclose(a, b, rtol=0, atol=1e-10)
    # a dominant logit: about 0 for its own target, about the gap for another
    big, _ = O.cross_entropy(np.array([[1000.0, 0.0], [1000.0, 0.0]]), np.array([0, 1]))
    assert big[0] == 0.0 and big[1] == 1000.0


def test_cross_entropy_ignores_negative_targets():
    z = np.array([[0.0, math.log(3.0)], [5.0, -2.0], [1.0, 1.0]])
    loss, mean = O.cross_entropy(z, np.array([1, -1, 0]))
    assert loss[1] == 0.0
    assert abs(mean - (math.log(4.0 / 3.0) + math.log(2.0)) / 2) < 1e-15
    _, none = O.cross_entropy(z, np.array([-1, -1, -1]))
    assert math.isnan(none)
