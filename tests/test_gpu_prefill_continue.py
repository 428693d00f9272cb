"""Prefill continued from a non-empty cache (nc_prefill_continue) against the
oracle's one-shot prefill (GPU).

A prompt run in pieces must give, for every piece, the logits the oracle gives at
those positions of the whole prompt, and at the end the whole prompt's K/V (slots
past the length still poisoned). The pieces cover a start that is not a multiple
of the 128-row attention tile (so the causal boundary splits key tiles), tile-aligned
starts, a one-token piece (one decode step through the per-kernel path), MQA and
MHA shapes.
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import (argmax_agreement, assert_close, check_cache, oracle_weights,
                               poison_cache, to_np)
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu


def _small(base, **kw):
    return synth.with_changes(base, name=base.name + "_small", **kw)


def _run(shape, B, cuts, act=nc.NC_F16, tol=2e-2):
    import torch
    W = synth.make_weights(shape)
    T = cuts[-1]
    t_cap = T + 3
    toks = synth.make_tokens(shape, B, T)
    full, ocache = O.prefill(shape, *oracle_weights(W), toks, t_cap=t_cap)
    model = nc.Model(W, max_seq=t_cap, max_batch=B, act_dtype=act)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    tok_d = torch.from_numpy(toks).cuda()
    a = 0
    for b in cuts:
        n = b - a
        lg = torch.empty(B, n, shape.vocab, device="cuda")
        piece = tok_d[:, a:b].contiguous()
        if a == 0:
            nc.nc_prefill(model.handle, piece, B, n, lg, cache.handle)
        else:
            nc.nc_prefill_continue(model.handle, piece, B, n, lg, cache.handle)
        torch.cuda.synchronize()
        ref = full[:, a:b]
        assert_close(to_np(lg), ref, tol, f"{shape.name} positions {a}..{b - 1}")
        argmax_agreement(lg.argmax(-1).cpu().numpy().reshape(-1), ref.reshape(-1, shape.vocab), tol)
        a = b
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    check_cache(cache, ocache, shape, list(range(B)), T, tol)
    cache.close()
    model.close()


def test_mqa_start_inside_a_tile(cuda_device):
    _run(_small(synth.D20_MQA, n_layer=2, vocab=1000), 3, [100, 300])


def test_mha_tile_aligned_then_short_piece(cuda_device):
    _run(_small(synth.D20, n_layer=2, vocab=1000), 2, [128, 256, 260])


def test_gqa_one_token_piece_and_several_pieces(cuda_device):
    _run(_small(synth.D20, n_layer=2, vocab=768, n_kv_head=2), 2, [37, 38, 170, 171, 300])


def test_fp32_model_rejects_a_continued_multi_token_piece(cuda_device):
    import torch
    shape = synth.TINY
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=16, max_batch=1, act_dtype=nc.NC_F32)
    cache = model.cache(1, 16)
    toks = torch.from_numpy(synth.make_tokens(shape, 1, 8)).cuda()
    lg = torch.empty(1, 8, shape.vocab, device="cuda")
    nc.nc_prefill(model.handle, toks[:, :4].contiguous(), 1, 4, lg, cache.handle)
    with pytest.raises(RuntimeError):
        nc.nc_prefill_continue(model.handle, toks[:, 4:8].contiguous(), 1, 4, lg, cache.handle)
    cache.close()
    model.close()
