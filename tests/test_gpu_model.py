"""Whole forward pass (prefill, decode, greedy generation) through the C ABI
against the oracle on the same seeded inputs (GPU).

Small shapes span several tiles and ragged tails; the full workloads run at
their real sizes on the GPU and are checked on the sequences the oracle can
afford (sequences are independent, so a subset is an exact check of them).
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import (argmax_agreement, assert_close, check_cache, oracle_weights,
                               poison_cache, to_np, tol_for)
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu


def _prefill_case(shape, B, T, t_cap, seqs, positions=None, check_kv=True):
    import torch
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=t_cap, max_batch=B)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    toks = synth.make_tokens(shape, B, T)
    tok_d = torch.from_numpy(toks).cuda()
    logits = torch.empty(B, T, shape.vocab, device="cuda")
    nc.nc_prefill(model.handle, tok_d, B, T, logits, cache.handle)
    torch.cuda.synchronize()
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    assert cache.length == T
    ref, ocache = O.prefill(shape, *oracle_weights(W), toks[seqs], logit_positions=positions)
    got = logits[seqs] if positions is None else logits[seqs][:, positions]
    tol = tol_for(shape)
    err = assert_close(to_np(got), ref, tol, f"{shape.name} prefill logits")
    if check_kv:
        check_cache(cache, ocache, shape, seqs, T, tol)
    return err


def _small(base, **kw):
    return synth.with_changes(base, name=base.name + "_small", **kw)


# ------------------------------------------------------------------ tiny fp32
def test_tiny_prefill(cuda_device):
    _prefill_case(synth.TINY, 1, 16, 16, [0])


def test_tiny_decode_equals_oracle(cuda_device):
    import torch
    shape = synth.TINY
    W = synth.make_weights(shape)
    T0, steps = 6, 10
    model = nc.Model(W, max_seq=16, max_batch=1)
    cache = model.cache(1, 16)
    poison_cache(cache)
    toks = synth.make_tokens(shape, 1, T0 + steps)
    full, ocache = O.prefill(shape, *oracle_weights(W), toks)
    tok_d = torch.from_numpy(toks).cuda()
    lg = torch.empty(1, shape.vocab, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, tok_d[:, :T0].contiguous(), 1, T0, lg, am, cache.handle)
    assert_close(to_np(lg), full[:, T0 - 1], 1e-4, "prefill_last")
    for j in range(steps):
        step_tok = tok_d[:, T0 + j].contiguous()
        nc.nc_decode_step(model.handle, step_tok, 1, T0 + j, lg, am, cache.handle)
        torch.cuda.synchronize()
        assert_close(to_np(lg), full[:, T0 + j], 1e-4, f"decode step {j}")
        argmax_agreement(am.cpu().numpy(), full[:, T0 + j], 1e-4)
    check_cache(cache, ocache, shape, [0], T0 + steps, 1e-4)


def test_tiny_generate_host_greedy(cuda_device):
    import torch
    shape = synth.TINY
    W = synth.make_weights(shape)
    T, steps = 5, 10
    model = nc.Model(W, max_seq=16, max_batch=1)
    cache = model.cache(1, 16)
    prompt = torch.from_numpy(synth.make_tokens(shape, 1, T)).pin_memory()
    out = torch.empty(steps + 1, 1, dtype=torch.int32).pin_memory()
    nc.nc_generate_host(model.handle, prompt, 1, T, steps, out, cache.handle)
    # oracle greedy, fed its own tokens
    logits, oc = O.prefill(shape, *oracle_weights(W), prompt.numpy(), t_cap=16)
    want = [int(O.greedy_next(logits[0, -1]))]
    lgs = [logits[0, -1]]
    for _ in range(steps):
        lg = O.decode_step(shape, *oracle_weights(W), np.array([want[-1]]), oc)[0]
        lgs.append(lg)
        want.append(int(O.greedy_next(lg)))
    got = out[:, 0].numpy().tolist()
    rms = np.sqrt(np.mean(np.square(lgs)))
    for j in range(steps + 1):
        top2 = np.sort(lgs[j])[-2:]
        if top2[1] - top2[0] <= 1e-4 * rms:
            break   # near tie: later tokens may legitimately differ
        assert got[j] == want[j], f"greedy token {j}"


def test_bad_token_is_flagged_not_faulted(cuda_device):
    import torch
    shape = synth.TINY
    W = synth.make_weights(shape)
    model = nc.Model(W, max_seq=16, max_batch=1)
    cache = model.cache(1, 16)
    toks = torch.tensor([[1, 2, 27, -3]], dtype=torch.int32, device="cuda")
    logits = torch.empty(1, 4, 27, device="cuda")
    nc.nc_prefill(model.handle, toks, 1, 4, logits, cache.handle)
    assert nc.nc_model_check(model.handle) == nc.NC_ERR_BOUNDS
    assert nc.nc_model_check(model.handle) == nc.NC_OK    # cleared after reading


def _scale_pow2(W, name, k):
    """Multiplies one matrix of W by 2^k (exact, also for its bf16 bits)."""
    if name == "wte":
        W.wte = W.wte * np.float32(2.0 ** k)
        arr = W.wte
    else:
        l, n = name.split(".")[1], name.split(".")[2]
        mats = list(W.layers[int(l)])
        i = synth.LAYER_MATRIX_NAMES.index(n)
        mats[i] = mats[i] * np.float32(2.0 ** k)
        W.layers[int(l)] = tuple(mats)
        arr = mats[i]
    if W.bits is not None:
        W.bits[name] = synth.round_to_bf16_bits(arr)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("case", ["relu2", "residual"])
def test_fp16_overflow_is_flagged(cuda_device, act, case):
    """Values stored in fp16 that exceed its range latch NC_ERR_RANGE instead of
    silently becoming inf. 'relu2': W_fc x 2^9 puts the ReLU^2 activations near
    2^18 (the prefill's FC epilogue and the decode step's PROJ staging). 'residual':
    wte x 2^20 puts the residual near 3e4 RMS, which only the decode step stages
    un-normalised. bf16 has fp32's range: no flag."""
    import torch
    shape = synth.with_changes(synth.D20_MQA, name="range", n_layer=1, vocab=512)
    W = synth.make_weights(shape)
    if case == "relu2":
        _scale_pow2(W, "layers.0.w_fc", 9)
    else:
        _scale_pow2(W, "wte", 20)
    adt = nc.NC_F16 if act == "f16" else nc.NC_BF16
    model = nc.Model(W, max_seq=48, max_batch=2, act_dtype=adt)
    nc.nc_model_set_decode_path(model.handle, nc.NC_DECODE_PERSISTENT)
    cache = model.cache(2, 48)
    toks = torch.from_numpy(synth.make_tokens(shape, 2, 33)).cuda()
    am = torch.empty(2, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, toks[:, :32].contiguous(), 2, 32, None, am, cache.handle)
    want_prefill = nc.NC_ERR_RANGE if (act == "f16" and case == "relu2") else nc.NC_OK
    assert nc.nc_model_check(model.handle) == want_prefill
    nc.nc_decode_step(model.handle, toks[:, 32].contiguous(), 2, 32, None, am, cache.handle)
    want_decode = nc.NC_ERR_RANGE if act == "f16" else nc.NC_OK
    assert nc.nc_model_check(model.handle) == want_decode
    assert nc.nc_model_check(model.handle) == nc.NC_OK   # cleared after reading
    cache.close()
    model.close()


def test_host_argument_errors(cuda_device):
    import torch
    shape = synth.TINY
    model = nc.Model(synth.make_weights(shape), max_seq=16, max_batch=1)
    cache = model.cache(1, 8)
    toks = torch.zeros(1, 9, dtype=torch.int32, device="cuda")
    logits = torch.empty(1, 9, 27, device="cuda")
    with pytest.raises(nc.NcError):        # T > cache t_max
        nc.nc_prefill(model.handle, toks, 1, 9, logits, cache.handle)
    with pytest.raises(nc.NcError):        # decode before prefill (pos != len)
        nc.nc_decode_step(model.handle, toks, 1, 3, logits, None, cache.handle)
    with pytest.raises(nc.NcError):
        nc.nc_kv_cache_alloc(model.handle, 1, 17)   # beyond max_seq


# ------------------------------------------------------- bf16, reduced sizes
@pytest.mark.parametrize("kv", [10, 2, 1])
def test_bf16_prefill_tile_mode(cuda_device, kv):
    shape = _small(synth.D20, n_layer=2, vocab=1000, n_kv_head=kv)
    _prefill_case(shape, 2, 300, 320, [0, 1])


def test_bf16_prefill_swap_mode(cuda_device):
    shape = _small(synth.D26, n_layer=2, vocab=700)
    _prefill_case(shape, 3, 37, 40, [0, 1, 2])


def test_bf16_storage_mode_prefill(cuda_device):
    """bf16 activations / KV cache (act_dtype NC_BF16): the same kernels with bf16
    rounding at every GEMM input. Its logits drift ~0.03-0.045 x RMS (max) from
    exact arithmetic by rounding alone, so it is held to 6e-2, not the fp16 bar."""
    import torch
    shape = _small(synth.D20, n_layer=2, vocab=1000, n_kv_head=2)
    W = synth.make_weights(shape)
    B, T = 2, 300
    model = nc.Model(W, max_seq=T, max_batch=B, act_dtype=nc.NC_BF16)
    cache = model.cache(B, T)
    toks = synth.make_tokens(shape, B, T)
    logits = torch.empty(B, T, shape.vocab, device="cuda")
    nc.nc_prefill(model.handle, torch.from_numpy(toks).cuda(), B, T, logits, cache.handle)
    torch.cuda.synchronize()
    ref, _ = O.prefill(shape, *oracle_weights(W), toks)
    assert_close(to_np(logits), ref, 6e-2, "bf16-storage prefill logits")


def test_bf16_decode_steps(cuda_device):
    import torch
    shape = _small(synth.D20_MQA, n_layer=3, vocab=2048)
    W = synth.make_weights(shape)
    B, T0, steps = 5, 200, 6
    t_cap = T0 + steps
    model = nc.Model(W, max_seq=t_cap, max_batch=B)
    cache = model.cache(B, t_cap)
    poison_cache(cache)
    toks = synth.make_tokens(shape, B, t_cap)
    full, ocache = O.prefill(shape, *oracle_weights(W), toks)
    tok_d = torch.from_numpy(toks).cuda()
    lg = torch.empty(B, shape.vocab, device="cuda")
    am = torch.empty(B, dtype=torch.int32, device="cuda")
    nc.nc_prefill_last(model.handle, tok_d[:, :T0].contiguous(), B, T0, lg, am, cache.handle)
    torch.cuda.synchronize()
    assert_close(to_np(lg), full[:, T0 - 1], 2e-2, "prefill_last")
    for j in range(steps):
        nc.nc_decode_step(model.handle, tok_d[:, T0 + j].contiguous(), B, T0 + j, lg, am,
                          cache.handle)
        torch.cuda.synchronize()
        assert_close(to_np(lg), full[:, T0 + j], 2e-2, f"decode step {j}")
        argmax_agreement(am.cpu().numpy(), full[:, T0 + j], 2e-2)
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    check_cache(cache, ocache, shape, list(range(B)), t_cap, 2e-2)
