"""The allocation-free decode attention entry point, for callers that cannot
call cudaMalloc (an engine that owns all device memory through its own pool, a
plugin inside such a host, a loop that cannot take an allocation's implicit
synchronisation). Its partial softmax states live in a fixed array inside the
library; its output must match the scratch-buffer entry point's.

Collected last on purpose, so a stop-at-first-failure run has already run every
other test; it also passes alone in a fresh process (the first call does the
per-device set-up)."""
import numpy as np
import pytest

from transformer_forward_gpt_b300 import binding as nc

pytestmark = pytest.mark.gpu


def _inputs(B, H, Hkv, length, t_max, hd, seed):
    import torch
    rng = np.random.default_rng(seed)
    f = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float32)).cuda().half()
    return f(B, H, hd), f(B, Hkv, t_max, hd), f(B, Hkv, t_max, hd)


@pytest.mark.parametrize("B,H,Hkv,length", [(32, 10, 1, 1100), (4, 13, 13, 2049)])
def test_noalloc_matches_scratch_entry_point_twice(cuda_device, B, H, Hkv, length):
    import torch
    hd, t_max = 128, length + 8
    for call in range(2):      # two calls in a row: the shared array keeps old contents
        q, k, v = _inputs(B, H, Hkv, length - call, t_max, hd, seed=length + call)
        n = length - call
        ref = torch.empty(B, H * hd, device="cuda", dtype=torch.float16)
        nbytes = nc.nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        nc.nc_op_attention_decode(q, k, v, ref, B, H, Hkv, n, t_max, hd, nc.NC_F16, scratch, nbytes)
        got = torch.full((B, H * hd), float("nan"), device="cuda", dtype=torch.float16)
        nc.nc_op_attention_decode_noalloc(q, k, v, got, B, H, Hkv, n, t_max, hd, nc.NC_F16)
        torch.cuda.synchronize()
        # same kernel, same inputs: the tests' fp16 rounding bound is far looser than needed
        d = (got.float() - ref.float()).abs()
        bound = 2.0 ** -11 * ref.float().abs() + 1e-5
        assert bool((d <= bound).all()), f"call {call}: max diff {d.max().item():.3g}"


def test_noalloc_rejects_sizes_beyond_its_array(cuda_device):
    import torch
    # 1024 sequences x 16 heads x 1 split x 130 floats = 8.5 MB > 8 MiB. The
    # buffers are real and large enough, so nothing could read out of bounds.
    B, H, Hkv, length, hd = 1024, 16, 16, 64, 128
    q = torch.zeros(B, H, hd, device="cuda", dtype=torch.float16)
    kv = torch.zeros(B, Hkv, length, hd, device="cuda", dtype=torch.float16)
    o = torch.zeros(B, H * hd, device="cuda", dtype=torch.float16)
    with pytest.raises(nc.NcError) as e:
        nc.nc_op_attention_decode_noalloc(q, kv, kv, o, B, H, Hkv, length, length, hd, nc.NC_F16)
    assert e.value.code == nc.NC_ERR_INVALID_ARG
    assert "fixed array" in str(e.value)
