"""The five workloads at their full sizes, in the launch configuration the
benchmark times, checked against the oracle on sampled sequences (GPU).

Sequences never interact, so the oracle's run on a subset of the batch is an
exact reference for those rows of the GPU's full-batch run. Every position's
logits of the sampled sequences are compared, plus their KV-cache rows, and for
decode every step's logits and greedy token.
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import (argmax_agreement, assert_close, check_cache, oracle_weights,
                               poison_cache, to_np)
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.mark.parametrize("name,seqs", [("d12_prefill", [0, 7]), ("d20_prefill", [0, 3]),
                                       ("d26_prefill", [1])])
def test_full_prefill(cuda_device, name, seqs):
    import torch
    wl = synth.WORKLOADS[name]
    shape, B, T = wl.shape, wl.batch, wl.seq
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=T, max_batch=B)
    cache = model.cache(B, T)
    poison_cache(cache)
    toks = synth.make_tokens(shape, B, T)
    logits = torch.empty(B, T, shape.vocab, device="cuda")
    nc.nc_prefill(model.handle, torch.from_numpy(toks).cuda(), B, T, logits, cache.handle)
    torch.cuda.synchronize()
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    ref, ocache = O.prefill(shape, *oracle_weights(W), toks[seqs])
    for j, b in enumerate(seqs):
        assert_close(to_np(logits[b]), ref[j], TOL, f"{name} seq {b} logits")
    check_cache(cache, ocache, shape, seqs, T, TOL)


@pytest.mark.parametrize("name,seqs", [("d20_mqa_decode", [0, 31]), ("d26_decode", [5])])
def test_full_decode(cuda_device, name, seqs):
    """Prefill to the workload's context, then greedy decode. The sampled
    sequences are fed the oracle's greedy tokens (teacher forcing, so one
    near-tie cannot change the rest of the run); the others feed back their own
    GPU argmax."""
    import torch
    wl = synth.WORKLOADS[name]
    shape, B, T0, steps = wl.shape, wl.batch, wl.seq, wl.decode_steps
    t_cap = T0 + steps
    W = synth.make_weights(shape)
    toks = synth.make_tokens(shape, B, T0)
    # oracle greedy run of the sampled sequences
    o_logits, oc = O.prefill(shape, *oracle_weights(W), toks[seqs], t_cap=t_cap,
                             logit_positions=[T0 - 1])
    o_steps = [o_logits[:, 0]]
    fed = []
    for j in range(steps):
        nxt = O.greedy_next(o_steps[-1])
        fed.append(nxt)
        o_steps.append(O.decode_step(shape, *oracle_weights(W), nxt, oc))

    model = nc.Model(W, max_seq=t_cap, max_batch=B)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    lg = torch.empty(B, shape.vocab, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, torch.from_numpy(toks).cuda(), B, T0, lg, am, cache.handle)
    torch.cuda.synchronize()
    idx = torch.tensor(seqs, device="cuda")
    decided = 0
    for j in range(steps + 1):
        got = to_np(lg[idx])
        assert_close(got, o_steps[j], TOL, f"{name} step {j} logits")
        decided += argmax_agreement(am[idx].cpu().numpy(), o_steps[j], TOL)[0]
        if j == steps:
            break
        nxt = am.clone()
        nxt[idx] = torch.from_numpy(fed[j].astype(np.int32)).cuda()
        nc.nc_decode_step(model.handle, nxt, B, T0 + j, lg, am, cache.handle)
        torch.cuda.synchronize()
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    assert decided >= (steps + 1) * len(seqs) // 2
    check_cache(cache, oc, shape, seqs, t_cap, TOL)
