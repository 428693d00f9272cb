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


def _inputs(B, H, Hkv, t_max, hd, dtype, seed):
    import torch
    rng = np.random.default_rng(seed)
    tt = torch.float16 if dtype == nc.NC_F16 else torch.float32
    f = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float32)).cuda().to(tt)
    return f(B, H, hd), f(B, Hkv, t_max, hd), f(B, Hkv, t_max, hd)


# Each case makes two calls in a row with different lengths. The second call of
# the MHA case is much shorter (5 splits of the key range, then 2), so a result
# that read partials left in the shared array by the first call would differ.
# The fp32 head_dim-64 case runs the CUDA-core kernel instead of the tensor-core one.
@pytest.mark.parametrize("B,H,Hkv,lengths,hd,dtype", [
    (32, 10, 1, (1100, 1099), 128, nc.NC_F16),
    (4, 13, 13, (2049, 100), 128, nc.NC_F16),
    (3, 8, 2, (700, 65), 64, nc.NC_F32),
])
def test_noalloc_matches_scratch_entry_point_twice(cuda_device, B, H, Hkv, lengths, hd, dtype):
    import torch
    tt = torch.float16 if dtype == nc.NC_F16 else torch.float32
    t_max = lengths[0] + 8
    for call, n in enumerate(lengths):   # the shared array keeps the previous call's contents
        q, k, v = _inputs(B, H, Hkv, t_max, hd, dtype, seed=n + call)
        ref = torch.empty(B, H * hd, device="cuda", dtype=tt)
        nbytes = nc.nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        nc.nc_op_attention_decode(q, k, v, ref, B, H, Hkv, n, t_max, hd, dtype, scratch, nbytes)
        got = torch.full((B, H * hd), float("nan"), device="cuda", dtype=tt)
        nc.nc_op_attention_decode_noalloc(q, k, v, got, B, H, Hkv, n, t_max, hd, dtype)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: a bound of one rounding of the output
        # type is far looser than needed
        eps = 2.0 ** -11 if dtype == nc.NC_F16 else 2.0 ** -23
        d = (got.float() - ref.float()).abs()
        bound = eps * ref.float().abs() + 1e-6
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
