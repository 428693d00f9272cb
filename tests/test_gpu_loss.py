"""The training step's loss (nc_prefill_loss, nc_op_cross_entropy) on the GPU.

Each position's loss is lse(z) - z[target], so its error is at most twice the
largest logit error.
- Op level (nc_op_cross_entropy, the fused LM-head reduction alone): against the
  oracle's cross-entropy of the fp64 product of the same 16-bit operands, within
  fp32 accumulation and exponential rounding (1e-4), at ragged sizes and at the
  full d20 LM head (8192 x 65536 x 1280, sampled rows).
- Model level (nc_prefill_loss): the prefill's bar of 2e-2 x RMS on the logits
  gives 4e-2 x RMS against the oracle's cross-entropy of its own logits. Where the
  whole prefill is deterministic (B*T <= 128: split-K sums in a fixed order), the
  loss also matches the fp64 cross-entropy of the library's own logits from
  nc_prefill within 1e-4. Above that, two prefills differ through the run-dependent
  order of the projections' fp32 sums (rounded to fp16 in between), so the check
  against the own logits at the full d20 size uses the bound of two runs each
  within 2e-2 x RMS of the oracle: 8e-2 x RMS.
- The mean is the mean of the counted rows; negative targets are left out; a
  target past the vocabulary is left out and flagged; a zero LM head gives ln V at
  every position of the full d20 size; fp32 models are refused.
"""
import math

import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import oracle_weights, to_np
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu


def _targets(shape, toks, rng):
    """Position t predicts token t + 1; the last position of each sequence gets a
    fresh draw (its next token lies outside the window)."""
    t = np.empty_like(toks)
    t[:, :-1] = toks[:, 1:]
    t[:, -1] = rng.integers(0, shape.vocab, size=toks.shape[0])
    return t


def _loss(model, cache, tok_d, tgt_d, B, T):
    import torch
    loss = torch.full((B * T,), float("nan"), device="cuda")
    mean = torch.full((1,), float("nan"), device="cuda")
    nc.nc_prefill_loss(model.handle, tok_d, tgt_d, B, T, loss, mean, cache.handle)
    torch.cuda.synchronize()
    return to_np(loss), float(mean.item())


@pytest.mark.parametrize("base,B,T,vocab", [(synth.D20, 3, 150, 1000),
                                            (synth.D20_MQA, 2, 129, 2048),
                                            (synth.D12, 1, 40, 300)])
def test_loss_matches_oracle_and_own_logits(cuda_device, base, B, T, vocab):
    import torch
    shape = synth.with_changes(base, name=base.name + "_loss", n_layer=2, vocab=vocab)
    W = synth.make_weights(shape)
    rng = np.random.default_rng(B * T)
    toks = synth.make_tokens(shape, B, T)
    tgt = _targets(shape, toks, rng)
    tgt.reshape(-1)[rng.choice(B * T, size=7, replace=False)] = -1   # left out
    ref_logits, _ = O.prefill(shape, *oracle_weights(W), toks)
    ref_logits = ref_logits.reshape(B * T, vocab)
    ref_loss, ref_mean = O.cross_entropy(ref_logits, tgt.reshape(-1))
    model = nc.Model(W, max_seq=T, max_batch=B)
    cache = model.cache(B, T)
    tok_d = torch.from_numpy(toks).cuda()
    tgt_d = torch.from_numpy(tgt).cuda()
    got, mean = _loss(model, cache, tok_d, tgt_d, B, T)
    keep = tgt.reshape(-1) >= 0
    rms = np.sqrt(np.mean(ref_logits ** 2))
    assert np.all(got[~keep] == 0.0)
    err = np.abs(got - ref_loss).max()
    assert err <= 4e-2 * rms, f"loss vs oracle: {err:.3g} > 4e-2 x {rms:.3g}"
    assert abs(mean - ref_mean) <= 4e-2 * rms
    if B * T <= 128:   # deterministic prefill: the library's own logits, reduced in fp64
        lg = torch.empty(B, T, vocab, device="cuda")
        nc.nc_prefill(model.handle, tok_d, B, T, lg, cache.handle)
        torch.cuda.synchronize()
        own, _ = O.cross_entropy(to_np(lg).reshape(B * T, vocab), tgt.reshape(-1))
        assert np.abs(got - own).max() <= 1e-4
    assert abs(mean - np.mean(got[keep])) <= 1e-6 * abs(mean)
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    cache.close()
    model.close()


def test_target_past_the_vocabulary_is_left_out_and_flagged(cuda_device):
    import torch
    shape = synth.with_changes(synth.D20, name="d20_loss_bad", n_layer=1, vocab=512)
    W = synth.make_weights(shape)
    B, T = 2, 64
    toks = synth.make_tokens(shape, B, T)
    tgt = _targets(shape, toks, np.random.default_rng(3))
    tgt[1, 5] = shape.vocab
    model = nc.Model(W, max_seq=T, max_batch=B)
    cache = model.cache(B, T)
    got, mean = _loss(model, cache, torch.from_numpy(toks).cuda(), torch.from_numpy(tgt).cuda(),
                      B, T)
    assert got[T + 5] == 0.0
    keep = np.ones(B * T, dtype=bool)
    keep[T + 5] = False
    assert abs(mean - np.mean(got[keep])) <= 1e-6 * abs(mean)
    assert nc.nc_model_check(model.handle) == nc.NC_ERR_BOUNDS
    assert nc.nc_model_check(model.handle) == nc.NC_OK      # the check clears the word
    # every target left out: the mean is NaN
    _, none = _loss(model, cache, torch.from_numpy(toks).cuda(),
                    torch.full((B, T), -1, dtype=torch.int32, device="cuda"), B, T)
    assert math.isnan(none)
    cache.close()
    model.close()


def test_full_size_d20(cuda_device):
    """B 4 x T 2048 at d20: 64 sampled positions against the cross-entropy of the
    library's own logits (a second prefill), the mean against the rows; then a zero
    LM head, whose logits are all 0, gives ln 65536 at every position."""
    import torch
    wl = synth.WORKLOADS["d20_prefill"]
    shape, B, T = wl.shape, wl.batch, wl.seq
    W = synth.make_weights(shape)
    rng = np.random.default_rng(9)
    toks = synth.make_tokens(shape, B, T)
    tgt = _targets(shape, toks, rng)
    tok_d = torch.from_numpy(toks).cuda()
    tgt_d = torch.from_numpy(tgt).cuda()
    model = nc.Model(W, max_seq=T, max_batch=B)
    cache = model.cache(B, T)
    got, mean = _loss(model, cache, tok_d, tgt_d, B, T)
    assert np.all(np.isfinite(got))
    rows = np.sort(rng.choice(B * T, size=64, replace=False))
    lg = torch.empty(B * T, shape.vocab, device="cuda")
    nc.nc_prefill(model.handle, tok_d, B, T, lg, cache.handle)
    torch.cuda.synchronize()
    sel = to_np(lg[torch.from_numpy(rows).cuda()])
    del lg
    own, _ = O.cross_entropy(sel, tgt.reshape(-1)[rows])
    assert np.abs(got[rows] - own).max() <= 8e-2 * np.sqrt(np.mean(sel ** 2))
    assert abs(mean - np.mean(got)) <= 1e-6 * abs(mean)
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    cache.close()
    model.close()
    W.lm_head[:] = 0.0
    W.bits["lm_head"][:] = 0
    model = nc.Model(W, max_seq=T, max_batch=B)
    cache = model.cache(B, T)
    got, mean = _loss(model, cache, tok_d, tgt_d, B, T)
    assert np.abs(got - math.log(shape.vocab)).max() <= 2e-6
    assert abs(mean - math.log(shape.vocab)) <= 2e-6
    cache.close()
    model.close()


def test_fp32_model_is_refused(cuda_device):
    import torch
    shape = synth.TINY
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=16, max_batch=1, act_dtype=nc.NC_F32)
    cache = model.cache(1, 16)
    tok = torch.from_numpy(synth.make_tokens(shape, 1, 16)).cuda()
    mean = torch.empty(1, device="cuda")
    with pytest.raises(nc.NcError):
        nc.nc_prefill_loss(model.handle, tok, tok, 1, 16, None, mean, cache.handle)
    with pytest.raises(nc.NcError):
        nc.nc_prefill_loss(model.handle, tok, None, 1, 16, None, mean, cache.handle)
    cache.close()
    model.close()


@pytest.mark.parametrize("dt", [nc.NC_BF16, nc.NC_F16])
@pytest.mark.parametrize("M,N,K", [(300, 1000, 256), (37, 384, 768), (1, 256, 64),
                                   (129, 65536, 1280), (8192, 65536, 1280)])
def test_op_cross_entropy_matches_oracle(cuda_device, M, N, K, dt):
    import torch
    tt = torch.bfloat16 if dt == nc.NC_BF16 else torch.float16
    g = torch.Generator().manual_seed(M + N + K)
    A = (torch.randn(M, K, generator=g) * 2.0).to(tt)
    Bm = (torch.randn(N, K, generator=g) / math.sqrt(K)).to(tt)
    tgt = torch.randint(0, N, (M,), generator=g, dtype=torch.int32)
    if M > 4:
        tgt[1] = -1          # left out
        tgt[3] = N + 5       # left out
    A_d, B_d, t_d = A.cuda(), Bm.cuda(), tgt.cuda()
    loss = torch.full((M,), float("nan"), device="cuda")
    mean = torch.full((1,), float("nan"), device="cuda")
    nbytes = nc.nc_op_cross_entropy_scratch_bytes(M, N)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_cross_entropy(A_d, B_d, t_d, M, N, K, dt, loss, mean, scratch, nbytes)
    torch.cuda.synchronize()
    got = to_np(loss)
    t_np = tgt.numpy().astype(np.int64)
    t_np[t_np >= N] = -1
    rows = np.arange(M) if M <= 512 else np.sort(np.random.default_rng(M).choice(M, 64, replace=False))
    a64, b64 = A.double().numpy()[rows], Bm.double().numpy()
    z = a64 @ b64.T
    want, _ = O.cross_entropy(z, t_np[rows])
    # fp32 accumulation over K (random-walk size, 4 sigma) in the two logits a loss
    # depends on most, plus fp32 rounding of the exponentials and the logarithm
    tol = 1e-4 + 8 * math.sqrt(K) * 2.0 ** -24 * float((np.abs(a64) @ np.abs(b64).T).max())
    assert np.abs(got[rows] - want).max() <= tol
    keep = t_np >= 0
    assert np.all(got[~keep] == 0.0)
    if M <= 512:
        _, want_mean = O.cross_entropy(z, t_np)
        assert abs(float(mean.item()) - want_mean) <= tol
    assert abs(float(mean.item()) - np.mean(got[keep])) <= 1e-6 * abs(float(mean.item()))


def test_op_cross_entropy_argument_checks(cuda_device):
    import torch
    A = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(4, dtype=torch.int32, device="cuda")
    mean = torch.empty(1, device="cuda")
    nbytes = nc.nc_op_cross_entropy_scratch_bytes(4, 256)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(nc.NcError):      # scratch too small
        nc.nc_op_cross_entropy(A, B, t, 4, 256, 64, nc.NC_BF16, None, mean, scratch, nbytes - 1)
    with pytest.raises(nc.NcError):      # fp32 operands
        nc.nc_op_cross_entropy(A, B, t, 4, 256, 64, nc.NC_F32, None, mean, scratch, nbytes)
    with pytest.raises(nc.NcError):      # K not a multiple of 64
        nc.nc_op_cross_entropy(A, B, t, 4, 256, 48, nc.NC_BF16, None, mean, scratch, nbytes)
    nc.nc_op_cross_entropy(A, B, t, 4, 256, 64, nc.NC_BF16, None, mean, scratch, nbytes)
    torch.cuda.synchronize()
    assert abs(float(mean.item()) - math.log(256)) <= 2e-6     # zero logits: ln N
