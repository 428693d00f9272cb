"""The persistent single-launch decode step against the oracle (GPU).

Each case prefills B sequences to T0 positions, then runs decode steps through
nc_decode_step with the persistent path forced on, and compares every step's
logits with the oracle (max |delta| <= 2e-2 x RMS), the greedy token wherever
the oracle's top-1 margin exceeds the tolerance, and the KV cache (filled slots
within tolerance, slots past the length still holding the poison value).

The shapes cover: every N-tile width of the kernel (B = 1, 5, 12, 20, 32) and
batches above 32 (several launches), MQA / GQA / MHA (one query head per KV
head), contexts whose last 32-position tile is partial, long contexts where
one (sequence, KV head) spans several CTAs (the O projection merges their
partial softmax states), d_model 768 / 1280 / 1664, and bf16 storage.
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import (argmax_agreement, assert_close, check_cache, oracle_weights,
                               poison_cache, to_np)
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu


def _run(shape, B, T0, steps, path=nc.NC_DECODE_PERSISTENT, act=nc.NC_F16, tol=2e-2, seqs=None):
    import torch
    W = synth.make_weights(shape)
    t_cap = T0 + steps
    seqs = list(range(B)) if seqs is None else seqs
    toks = synth.make_tokens(shape, B, t_cap)
    full, ocache = O.prefill(shape, *oracle_weights(W), toks[seqs])
    model = nc.Model(W, max_seq=t_cap, max_batch=B, act_dtype=act)
    nc.nc_model_set_decode_path(model.handle, path)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    tok_d = torch.from_numpy(toks).cuda()
    lg = torch.empty(B, shape.vocab, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, tok_d[:, :T0].contiguous(), B, T0, lg, am, cache.handle)
    errs = []
    idx = torch.tensor(seqs, device="cuda")
    for j in range(steps):
        nc.nc_decode_step(model.handle, tok_d[:, T0 + j].contiguous(), B, T0 + j, lg, am,
                          cache.handle)
        torch.cuda.synchronize()
        ref = full[:, T0 + j]
        errs.append(assert_close(to_np(lg[idx]), ref, tol, f"{shape.name} B{B} step {j}"))
        argmax_agreement(am[idx].cpu().numpy(), ref, tol)
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    check_cache(cache, ocache, shape, seqs, t_cap, tol)
    cache.close()
    model.close()
    return max(errs)


def _small(base, **kw):
    return synth.with_changes(base, name=base.name + "_small", **kw)


@pytest.mark.parametrize("B", [1, 5, 12, 20, 32])
def test_batch_widths_mqa(cuda_device, B):
    _run(_small(synth.D20_MQA, n_layer=2, vocab=1000), B, 45, 3)


@pytest.mark.parametrize("kv", [10, 2])
def test_gqa_and_mha(cuda_device, kv):
    _run(_small(synth.D20, n_layer=2, vocab=1000, n_kv_head=kv), 6, 37, 3)


def test_batch_above_32_runs_in_chunks(cuda_device):
    _run(_small(synth.D20_MQA, n_layer=2, vocab=512), 45, 20, 2, seqs=[0, 31, 32, 44])


def test_long_context_spans_ctas(cuda_device):
    # 2 sequences x 1 KV head x 63 tiles: each (sequence, KV head) covers ~74 CTAs
    _run(_small(synth.D20_MQA, n_layer=2, vocab=1000), 2, 1000, 3)


def test_shares_spanning_two_pairs(cuda_device):
    """20 sequences x 32 tiles = 640 tiles over the SMs: shares of 4-5 tiles, many
    of them ending in one (sequence, KV head) pair and starting in the next. Those
    CTAs prepare and compute both pairs in one round, one tile per warp, and add each
    pair's sums to its own accumulators; the new k / v rows land in whichever CTA
    holds a pair's last tile."""
    _run(_small(synth.D20_MQA, n_layer=2, vocab=512), 20, 1000, 2, seqs=[0, 7, 13, 19])


def test_tiles_shared_evenly_over_many_laps(cuda_device):
    """More (sequence, KV head) pairs than CTAs: the tiles of all pairs are shared
    evenly, about 50 per CTA, so the ring of stages turns over many times within
    one attention phase and the CTAs hold pieces of several pairs."""
    _run(_small(synth.D26, n_layer=1, vocab=512), 12, 1500, 2, seqs=[0, 5, 11])


@pytest.mark.parametrize("base", [synth.D12, synth.D26])
def test_other_widths(cuda_device, base):
    _run(_small(base, n_layer=2, vocab=768), 4, 70, 2)


def test_bf16_storage(cuda_device):
    _run(_small(synth.D20_MQA, n_layer=2, vocab=1000), 8, 50, 2, act=nc.NC_BF16, tol=6e-2)


def test_paths_agree(cuda_device):
    """The persistent path and the per-kernel path on the same inputs."""
    shape = _small(synth.D20_MQA, n_layer=3, vocab=2048)
    a = _run(shape, 7, 60, 3, path=nc.NC_DECODE_PERSISTENT)
    b = _run(shape, 7, 60, 3, path=nc.NC_DECODE_KERNELS)
    assert a < 2e-2 and b < 2e-2


def test_many_steps_keep_barrier_state(cuda_device):
    """Forty steps in a row: the grid barrier counter carries over between launches."""
    _run(_small(synth.D20_MQA, n_layer=1, vocab=512), 3, 16, 40)


def test_phase_trace_is_ordered(cuda_device):
    """nc_decode_trace: barrier arrivals and exits of CTA 0 are in time order, the
    producer marks precede the phases they load for, and a too-small buffer is
    left untouched."""
    import torch
    shape = _small(synth.D20_MQA, n_layer=2, vocab=512)
    W = synth.make_weights(shape)
    B, T0 = 4, 40
    model = nc.Model(W, max_seq=T0 + 2, max_batch=B)
    nc.nc_model_set_decode_path(model.handle, nc.NC_DECODE_PERSISTENT)
    cache = model.cache(B, T0 + 2)
    toks = torch.from_numpy(synth.make_tokens(shape, B, T0 + 1)).cuda()
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, toks[:, :T0].contiguous(), B, T0, None, am, cache.handle)
    n = nc.nc_decode_trace_entries(model.cfg)
    nbar = 5 * shape.n_layer + 3
    assert n >= 2 * nbar + 2
    small = torch.full((n - 1,), -7, dtype=torch.int64, device="cuda")
    nc.nc_decode_trace(model.handle, small)
    nc.nc_decode_step(model.handle, toks[:, T0].contiguous(), B, T0, None, am, cache.handle)
    torch.cuda.synchronize()
    assert bool((small == -7).all()), "a buffer below the required size must not be written"
    buf = torch.zeros(n, dtype=torch.int64, device="cuda")
    nc.nc_decode_trace(model.handle, buf)
    nc.nc_kv_cache_set_length(cache.handle, T0)
    nc.nc_decode_step(model.handle, toks[:, T0].contiguous(), B, T0, None, am, cache.handle)
    torch.cuda.synchronize()
    nc.nc_decode_trace(model.handle, None)
    t = buf.cpu().numpy()
    main = t[: 2 * nbar + 2]
    assert (np.diff(main) >= 0).all(), "barrier timestamps must be non-decreasing"
    assert main[-1] > main[0]
    marks = t[2 * nbar + 2: 8 * nbar + 2].reshape(-1, 6)
    for k in range(2, nbar):   # producer started each streamed phase before it ended
        if marks[k - 1, 4]:
            assert marks[k - 1, 4] <= main[2 * k - 1]
    # per CTA and barrier: arrival <= exit, and no CTA leaves before the last arrives
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per = t[8 * nbar + 2:].reshape(nbar, 256, 2)[:, :min(sms, 256)]
    assert (per[:, :, 0] > 0).all() and (per[:, :, 0] <= per[:, :, 1]).all()
    assert (per[:, :, 1].min(axis=1) >= per[:, :, 0].max(axis=1)).all()
    assert nc.nc_model_check(model.handle) == nc.NC_OK
