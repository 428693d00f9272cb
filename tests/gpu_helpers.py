"""Shared pieces of the GPU parity tests: running the CUDA path through the
C ABI, running the oracle on the same seeded inputs, and the tolerance checks."""
import numpy as np

from oracle import gpt_oracle as O
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

POISON = -1536.0   # planted in unwritten cache slots (exact in bf16 and fp16); must survive exactly


def tol_for(shape):
    """max |delta logit| <= tol * RMS(oracle logits): 1e-4 for fp32, 2e-2 for bf16."""
    return 1e-4 if shape.dtype == "f32" else 2e-2


def rel_err(got, ref):
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.abs(np.asarray(got, dtype=np.float64) - ref).max() / rms)


def assert_close(got, ref, tol, what):
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|delta|/rms = {e:.3g} > {tol}"
    return e


def to_np(t):
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_weights(W):
    return W.wte, W.layers, W.lm_head


def argmax_agreement(got_idx, ref_logits, tol):
    """Argmax must agree wherever the oracle's top-1 margin exceeds tol * RMS.
    Returns (rows checked, rows with margin > 2 tol * RMS)."""
    ref_logits = np.asarray(ref_logits)
    rms = np.sqrt(np.mean(ref_logits ** 2))
    top2 = np.sort(ref_logits, axis=-1)[..., -2:]
    margin = top2[..., 1] - top2[..., 0]
    want = ref_logits.argmax(-1)
    sure = margin > tol * rms
    assert np.array_equal(np.asarray(got_idx)[sure], want[sure]), "argmax differs on a decided row"
    return int(sure.sum()), int((margin > 2 * tol * rms).sum())


def poison_cache(cache):
    import torch
    k, v = cache.tensors()
    k.fill_(POISON)
    v.fill_(POISON)
    torch.cuda.synchronize()


def check_cache(cache, ocache, shape, seqs, length, tol):
    """Filled slots match the oracle's K/V within tol * RMS; slots >= length keep
    the poison value exactly (cache indexing)."""
    k, v = cache.tensors()
    for name, dev, orc in (("K", k, ocache.k), ("V", v, ocache.v)):
        for l in range(shape.n_layer):
            for j, b in enumerate(seqs):
                got = to_np(dev[l, b, :, :length])
                assert_close(got, orc[l][j][:, :length], tol, f"{name} cache layer {l} seq {b}")
        tail = dev[:, :, :, length:]
        if tail.numel():
            assert bool((tail.float() == POISON).all()), f"{name} cache written beyond length"
