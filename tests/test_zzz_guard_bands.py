"""Outputs stay inside their buffers (GPU).

Each output, and one KV cache, is a view into a larger buffer whose 16 KB margins on
both sides hold the byte 0xA5. After the call and a synchronize the margins must
still hold it, byte for byte. The inputs and shapes are those of the parity tests;
every output's last tile is partial. Covered:
- the tcgen05 GEMM (tile mode, fp32 tiles stored by TMA) and the fp32 CUDA-core GEMM;
- the cross-entropy reduction;
- prefill logits and loss rows;
- the KV cache written by prefill and by a decode step;
- decode logits and argmax;
- prefill and decode attention;
- RMSNorm, argmax, sampling and the fp8 GEMV.

The file runs last, so that a failure here leaves the parity tests' results intact.
"""
import numpy as np
import pytest

from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu

MARGIN = 16384   # bytes on each side


def _guarded(n, dtype):
    """(whole buffer, view of n elements at a 16 KB offset)."""
    import torch
    elem = torch.empty(0, dtype=dtype).element_size()
    g = MARGIN // elem
    whole = torch.empty(n + 2 * g, dtype=dtype, device="cuda")
    whole.view(torch.uint8).fill_(0xA5)
    return whole, whole[g:g + n]


def _intact(whole, n, what):
    import torch
    torch.cuda.synchronize()
    b = whole.view(torch.uint8)
    g = MARGIN
    lo, hi = b[:g], b[g + n * whole.element_size():]
    assert bool((lo == 0xA5).all()), f"{what}: bytes written before the buffer"
    assert bool((hi == 0xA5).all()), f"{what}: bytes written past the buffer"


@pytest.mark.parametrize("M,N,K", [(37, 384, 768), (300, 1664, 1280)])
def test_gemm_tile_mode(cuda_device, M, N, K):
    import torch
    g = torch.Generator().manual_seed(M)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16).cuda()
    whole, C = _guarded(M * N, torch.float32)
    nc.nc_op_gemm(A, B, C.view(M, N), M, N, K, nc.NC_BF16)
    _intact(whole, M * N, f"gemm {M}x{N}x{K}")
    assert not torch.isnan(C).any()


def test_gemm_f32(cuda_device):
    import torch
    g = torch.Generator().manual_seed(1)
    A = torch.randn(70, 48, generator=g).cuda()
    B = torch.randn(33, 48, generator=g).cuda()
    whole, C = _guarded(70 * 33, torch.float32)
    nc.nc_op_gemm(A, B, C.view(70, 33), 70, 33, 48, nc.NC_F32)
    _intact(whole, 70 * 33, "fp32 gemm")


def test_cross_entropy_op(cuda_device):
    import torch
    M, N, K = 300, 1000, 256
    g = torch.Generator().manual_seed(5)
    A = (torch.randn(M, K, generator=g) * 2).to(torch.bfloat16).cuda()
    B = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16).cuda()
    t = torch.randint(0, N, (M,), generator=g, dtype=torch.int32).cuda()
    wl, loss = _guarded(M, torch.float32)
    wm, mean = _guarded(1, torch.float32)
    nbytes = nc.nc_op_cross_entropy_scratch_bytes(M, N)
    ws, scratch = _guarded(nbytes, torch.uint8)
    nc.nc_op_cross_entropy(A, B, t, M, N, K, nc.NC_BF16, loss, mean, scratch, nbytes)
    _intact(wl, M, "loss rows")
    _intact(wm, 1, "mean")
    _intact(ws, nbytes, "scratch")


def test_model_outputs_and_cache(cuda_device):
    """Prefill logits, the KV cache (caller memory), loss rows, then one decode
    step's logits and argmax."""
    import torch
    shape = synth.with_changes(synth.D20, name="d20_guard", n_layer=2, vocab=1000)
    W = synth.make_weights(shape)
    B, T, V = 3, 150, shape.vocab
    model = nc.Model(W, max_seq=T + 1, max_batch=B)
    cb = nc.nc_kv_cache_bytes(model.cfg, B, T + 1)
    wc, cmem = _guarded(cb, torch.uint8)
    cache = nc.nc_kv_cache_alloc(model.handle, B, T + 1, cmem)
    toks = synth.make_tokens(shape, B, T + 1)
    tok_d = torch.from_numpy(toks[:, :T].copy()).cuda()
    wlg, lg = _guarded(B * T * V, torch.float32)
    nc.nc_prefill(model.handle, tok_d, B, T, lg, cache)
    _intact(wlg, B * T * V, "prefill logits")
    _intact(wc, cb, "KV cache after prefill")
    tgt = torch.from_numpy(toks[:, 1:].copy()).cuda()
    wl, loss = _guarded(B * T, torch.float32)
    wm, mean = _guarded(1, torch.float32)
    nc.nc_prefill_loss(model.handle, tok_d, tgt, B, T, loss, mean, cache)
    _intact(wl, B * T, "loss rows")
    _intact(wm, 1, "mean")
    _intact(wc, cb, "KV cache after the loss pass")
    wd, dl = _guarded(B * V, torch.float32)
    wa, am = _guarded(B, torch.int32)
    step = torch.from_numpy(toks[:, T].copy()).cuda()
    nc.nc_decode_step(model.handle, step, B, T, dl, am, cache)
    _intact(wd, B * V, "decode logits")
    _intact(wa, B, "decode argmax")
    _intact(wc, cb, "KV cache after a decode step")
    assert nc.nc_model_check(model.handle) == nc.NC_OK
    nc.nc_kv_cache_free(cache)
    model.close()


def test_attention(cuda_device):
    import torch
    rng = np.random.default_rng(200)
    B, H, Hkv, T, hd = 2, 4, 2, 200, 128
    t_max = T + 5
    q = torch.from_numpy(rng.standard_normal((B, H, T, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    wo, o = _guarded(B * T * H * hd, torch.bfloat16)
    nc.nc_op_attention_prefill(q, k, v, o.view(B, T, H * hd), B, H, Hkv, T, t_max, hd, nc.NC_BF16)
    _intact(wo, B * T * H * hd, "prefill attention")
    H, Hkv, length = 10, 1, 300
    t_max = length + 3
    q = torch.from_numpy(rng.standard_normal((B, H, 1, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(torch.bfloat16)
    wd, od = _guarded(B * H * hd, torch.bfloat16)
    nbytes = nc.nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_attention_decode(q, k, v, od.view(B, H * hd), B, H, Hkv, length, t_max, hd,
                              nc.NC_BF16, scratch, nbytes)
    _intact(wd, B * H * hd, "decode attention")


def test_rows_argmax_sample_fp8(cuda_device):
    import torch
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((33, 772)).astype(np.float32) * 3).cuda()
    wy, y = _guarded(33 * 772, torch.float16)
    nc.nc_op_rmsnorm(x, y.view(33, 772), nc.NC_F16, 33, 772, 1e-5)
    _intact(wy, 33 * 772, "rmsnorm")
    lg = torch.from_numpy(rng.standard_normal((5, 65536)).astype(np.float32)).cuda()
    wa, am = _guarded(5, torch.int32)
    nc.nc_op_argmax(lg, 5, 65536, am)
    _intact(wa, 5, "argmax")
    sl = torch.from_numpy((rng.standard_normal((9, 1000)) * 2).astype(np.float32)).cuda()
    u = torch.from_numpy(rng.random(9).astype(np.float32)).cuda()
    ws, out = _guarded(9, torch.int32)
    nc.nc_op_sample(sl, 9, 1000, 1.0, u, out)
    _intact(ws, 9, "sample")
    N, K, Bt = 300, 256, 100
    w = torch.from_numpy((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)).cuda()
    wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    wsc = torch.empty(N, dtype=torch.float32, device="cuda")
    nc.nc_op_quantize_e4m3(w, nc.NC_F32, N, K, wq, wsc)
    xa = torch.from_numpy(rng.standard_normal((Bt, K)).astype(np.float32)).cuda()
    wyy, yy = _guarded(Bt * N, torch.float32)
    nbytes = nc.nc_op_gemv_e4m3_scratch_bytes(N, K, Bt)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_gemv_e4m3(wq, wsc, N, K, xa, Bt, yy.view(Bt, N), scratch, nbytes)
    _intact(wyy, Bt * N, "fp8 gemv")
