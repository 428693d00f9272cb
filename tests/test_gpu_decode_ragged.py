"""Decode with a position per sequence (nc_decode_step_ragged) against the oracle
run on each sequence alone (GPU).

B sequences are prefilled together to a common length T, then cut back to their
own prompt lengths with nc_kv_cache_set_lengths; every decode step then feeds
each sequence its next token at its own position. The oracle runs each
sequence's own prompt and steps on its own, so the check is exact per sequence:
logits within 2e-2 x RMS, the greedy token wherever the oracle's margin exceeds
the tolerance, the cached K/V of every filled slot within tolerance, and the
slots past the prefill that no step wrote still holding the poison value.
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import POISON, argmax_agreement, assert_close, oracle_weights, poison_cache, to_np
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _small(base, **kw):
    return synth.with_changes(base, name=base.name + "_ragged", **kw)


def _run(shape, prompt_lens, steps):
    import torch
    B = len(prompt_lens)
    T = max(prompt_lens)
    t_cap = T + steps + 4
    W = synth.make_weights(shape)
    toks = synth.make_tokens(shape, B, t_cap)
    model = nc.Model(W, max_seq=t_cap, max_batch=B)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    tok_d = torch.from_numpy(toks).cuda()
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, tok_d[:, :T].contiguous(), B, T, None, am, cache.handle)
    nc.nc_kv_cache_set_lengths(cache.handle, prompt_lens)
    assert nc.nc_kv_cache_lengths(cache.handle, B) == list(prompt_lens)
    # the oracle: each sequence alone, its own prompt, then its own steps
    ocaches, orefs = [], []
    for b, n in enumerate(prompt_lens):
        _, oc = O.prefill(shape, *oracle_weights(W), toks[b:b + 1, :n], t_cap=t_cap,
                          logit_positions=[n - 1])
        refs = [O.decode_step(shape, *oracle_weights(W), toks[b:b + 1, n + j], oc)[0]
                for j in range(steps)]
        ocaches.append(oc)
        orefs.append(refs)
    lg = torch.empty(B, shape.vocab, device="cuda")
    for j in range(steps):
        pos = [n + j for n in prompt_lens]
        step_tok = torch.tensor([toks[b, p] for b, p in enumerate(pos)], dtype=torch.int32,
                                device="cuda")
        nc.nc_decode_step_ragged(model.handle, step_tok, pos, B, lg, am, cache.handle)
        torch.cuda.synchronize()
        got = to_np(lg)
        ref = np.stack([orefs[b][j] for b in range(B)])
        for b in range(B):
            assert_close(got[b], ref[b], TOL, f"{shape.name} seq {b} step {j} (pos {pos[b]})")
        argmax_agreement(am.cpu().numpy(), ref, TOL)
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    final = [n + steps for n in prompt_lens]
    assert nc.nc_kv_cache_lengths(cache.handle, B) == final
    k, v = cache.tensors()
    for name, dev, attr in (("K", k, "k"), ("V", v, "v")):
        for l in range(shape.n_layer):
            for b in range(B):
                got = to_np(dev[l, b, :, :final[b]])
                assert_close(got, getattr(ocaches[b], attr)[l][0][:, :final[b]], TOL,
                             f"{name} cache layer {l} seq {b}")
                # past both the prefill and this sequence's steps: never written
                tail = dev[l, b, :, max(T, final[b]):]
                assert bool((tail.float() == POISON).all()), f"{name} cache seq {b} written past its end"
    cache.close()
    model.close()


@pytest.mark.parametrize("lens", [(40, 17, 33, 64), (1, 95, 32, 33, 64, 2)])
def test_ragged_mqa(cuda_device, lens):
    _run(_small(synth.D20_MQA, n_layer=2, vocab=512), list(lens), 3)


def test_ragged_gqa(cuda_device):
    _run(_small(synth.D20, n_layer=2, vocab=512, n_kv_head=2), [70, 9, 31], 3)


def test_ragged_many_sequences_uneven_blocks(cuda_device):
    """36 sequences (two launches of up to 32), lengths from 1 to 300: pairs get
    CTA blocks in proportion to their tiles."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 300, size=36)]
    lens[3] = 300
    _run(_small(synth.D20_MQA, n_layer=1, vocab=256), lens, 2)


def test_ragged_argument_checks(cuda_device):
    import torch
    shape = _small(synth.D20_MQA, n_layer=1, vocab=256)
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=40, max_batch=3)
    cache = model.cache(3, 40)
    tok = torch.from_numpy(synth.make_tokens(shape, 3, 20)).cuda()
    am = torch.empty(3, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, tok, 3, 20, None, am, cache.handle)
    with pytest.raises(nc.NcError) as e:      # longer than the sequence holds
        nc.nc_kv_cache_set_lengths(cache.handle, [20, 21, 5])
    assert e.value.code == nc.NC_ERR_INVALID_ARG
    assert nc.nc_kv_cache_lengths(cache.handle, 3) == [20, 20, 20]
    nc.nc_kv_cache_set_lengths(cache.handle, [20, 7, 12])
    with pytest.raises(nc.NcError) as e:      # a position that is not the sequence's length
        nc.nc_decode_step_ragged(model.handle, am, [20, 8, 12], 3, None, am, cache.handle)
    assert e.value.code == nc.NC_ERR_INVALID_ARG
    with pytest.raises(nc.NcError) as e:      # the uniform call needs equal lengths
        nc.nc_decode_step(model.handle, am, 3, 20, None, am, cache.handle)
    assert e.value.code == nc.NC_ERR_INVALID_ARG
    nc.nc_decode_step_ragged(model.handle, am, [20, 7, 12], 3, None, am, cache.handle)
    torch.cuda.synchronize()
    assert nc.nc_kv_cache_lengths(cache.handle, 3) == [21, 8, 13]
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    cache.close()
    model.close()
