"""Single-step kernels through the C ABI against the oracle's steps (GPU)."""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from tests.gpu_helpers import assert_close, to_np
from transformer_forward_gpt_b300 import binding as nc

pytestmark = pytest.mark.gpu


UNIT_ROUNDOFF = {nc.NC_BF16: 2.0 ** -8, nc.NC_F16: 2.0 ** -11, nc.NC_F32: 2.0 ** -24}


def _torch_dt(dt):
    import torch
    return {nc.NC_BF16: torch.bfloat16, nc.NC_F16: torch.float16, nc.NC_F32: torch.float32}[dt]


def _rand(rng, shape, dt, scale=1.0):
    import torch
    return (torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
            .to("cuda").to(_torch_dt(dt)))


def assert_rounding_bound(got, ref, u, extra=0.0, what=""):
    """|got - ref| <= u |ref| + extra elementwise (u = unit roundoff of the stored format)."""
    d = np.abs(got - ref)
    bound = u * np.abs(ref) + extra + 1e-6
    worst = float((d / bound).max())
    assert worst <= 1.0, f"{what}: error reaches {worst:.3g} x the rounding bound"


@pytest.mark.parametrize("dt", [nc.NC_BF16, nc.NC_F16])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 1664, 1280), (37, 384, 768),
                                   (1000, 4992, 1664), (257, 65536, 1280), (8192, 1280, 5120)])
def test_gemm_tcgen05(cuda_device, M, N, K, dt):
    import torch
    rng = np.random.default_rng(M + N + K)
    A, B = _rand(rng, (M, K), dt), _rand(rng, (N, K), dt, 1 / np.sqrt(K))
    C = torch.full((M, N), float("nan"), device="cuda")
    nc.nc_op_gemm(A, B, C, M, N, K, dt)
    torch.cuda.synchronize()
    rows = np.unique(np.linspace(0, M - 1, min(M, 64)).astype(int))
    ref = O.linear(to_np(A[rows]), to_np(B))
    assert_close(to_np(C[rows]), ref, 1e-4, f"gemm {M}x{N}x{K}")
    assert not torch.isnan(C).any()


def test_gemm_f32_simt(cuda_device):
    import torch
    rng = np.random.default_rng(1)
    A = torch.from_numpy(rng.standard_normal((70, 48)).astype(np.float32)).cuda()
    B = torch.from_numpy(rng.standard_normal((33, 48)).astype(np.float32)).cuda()
    C = torch.empty(70, 33, device="cuda")
    nc.nc_op_gemm(A, B, C, 70, 33, 48, nc.NC_F32)
    torch.cuda.synchronize()
    assert_close(to_np(C), O.linear(to_np(A), to_np(B)), 1e-6, "fp32 gemm")


@pytest.mark.parametrize("dt", [nc.NC_F32, nc.NC_BF16, nc.NC_F16])
@pytest.mark.parametrize("M,d", [(77, 1280), (5, 4), (33, 772), (9, 2048), (7, 2052)])
def test_rmsnorm(cuda_device, dt, M, d):
    """Row widths from 4 to 2052, including ones that are not a multiple of 128."""
    import torch
    rng = np.random.default_rng(2)
    x = torch.from_numpy(rng.standard_normal((M, d)).astype(np.float32) * 3).cuda()
    y = torch.empty(M, d, device="cuda", dtype=_torch_dt(dt))
    nc.nc_op_rmsnorm(x, y, dt, M, d, 1e-5)
    torch.cuda.synchronize()
    ref = O.rmsnorm(to_np(x), 1e-5)
    # fp32 arithmetic, then one rounding to the stored format
    assert_rounding_bound(to_np(y), ref, max(UNIT_ROUNDOFF[dt], 2.0 ** -20), what="rmsnorm")


def _attn_inputs(rng, B, H, Hkv, T, t_max, hd, dt):
    import torch
    tdt = _torch_dt(dt)
    q = torch.from_numpy(rng.standard_normal((B, H, T, hd)).astype(np.float32)).cuda().to(tdt)
    k = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(tdt)
    v = torch.from_numpy(rng.standard_normal((B, Hkv, t_max, hd)).astype(np.float32)).cuda().to(tdt)
    k[:, :, T:] = float("nan")   # slots past the sequence must never be read
    v[:, :, T:] = float("nan")
    return q, k, v


@pytest.mark.parametrize("B,H,Hkv,T,dt,qscale", [
    (2, 4, 2, 200, nc.NC_BF16, 1.0), (1, 10, 1, 129, nc.NC_F16, 1.0),
    (3, 2, 2, 64, nc.NC_F16, 1.0), (1, 3, 3, 1, nc.NC_F16, 1.0),
    (2, 13, 13, 300, nc.NC_F16, 1.0), (2, 4, 4, 37, nc.NC_F32, 1.0),
    # more (query tile, head) items than SMs: the persistent kernel runs several
    # items per CTA, with ragged last query / key tiles
    (2, 16, 4, 1037, nc.NC_F16, 1.0), (1, 40, 8, 777, nc.NC_BF16, 1.0),
    # large scores: row maxima keep outgrowing the exponent's reference, so the
    # output rows are rescaled in tensor memory many times
    (1, 24, 2, 900, nc.NC_F16, 6.0)])
def test_attention_prefill(cuda_device, B, H, Hkv, T, dt, qscale):
    """Bound: the output is rounded once (u |o|) and the probabilities are rounded
    to the operand format before P V (u max|v| at most); fp32 elsewhere."""
    import torch
    hd = 8 if dt == nc.NC_F32 else 128
    t_max = T + 5
    rng = np.random.default_rng(T)
    q, k, v = _attn_inputs(rng, B, H, Hkv, T, t_max, hd, dt)
    q *= qscale
    o = torch.empty(B, T, H * hd, device="cuda", dtype=q.dtype)
    nc.nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, t_max, hd, dt)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.attend(to_np(q[b]), np.arange(T), to_np(k[b, :, :T]), to_np(v[b, :, :T]))
        got = to_np(o[b]).reshape(T, H, hd).transpose(1, 0, 2)
        u = UNIT_ROUNDOFF[dt] if dt != nc.NC_F32 else 1e-5
        vmax = float(np.abs(to_np(v[b, :, :T])).max())
        assert_rounding_bound(got, ref, u, u * vmax, f"attention seq {b}")
        if T == 1:   # one position: output is that position's V
            g = np.arange(H) // (H // Hkv)
            assert_close(got[:, 0], to_np(v[b, g, 0]), 1e-2, "length-1 attention")


@pytest.mark.parametrize("B,H,Hkv,length,dt", [(4, 10, 1, 1100, nc.NC_F16), (2, 13, 13, 2049, nc.NC_F16),
                                               (3, 4, 2, 5, nc.NC_F32), (1, 2, 1, 1, nc.NC_BF16),
                                               (2, 10, 1, 300, nc.NC_BF16)])
def test_attention_decode(cuda_device, B, H, Hkv, length, dt):
    import torch
    hd = 8 if dt == nc.NC_F32 else 128
    t_max = length + 3
    rng = np.random.default_rng(length)
    q, k, v = _attn_inputs(rng, B, H, Hkv, length, t_max, hd, dt)
    q = q[:, :, :1].contiguous()
    o = torch.empty(B, H * hd, device="cuda", dtype=q.dtype)
    nbytes = nc.nc_op_attention_decode_scratch_bytes(B, H, t_max, hd)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_attention_decode(q, k, v, o, B, H, Hkv, length, t_max, hd, dt, scratch, nbytes)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.attend(to_np(q[b]), np.array([length - 1]), to_np(k[b, :, :length]),
                       to_np(v[b, :, :length]))[:, 0]
        # 16-bit: probabilities are rounded to the operand format before P V (as in prefill)
        u = UNIT_ROUNDOFF[dt] if dt != nc.NC_F32 else 1e-5
        vmax = float(np.abs(to_np(v[b, :, :length])).max()) if dt != nc.NC_F32 else 0.0
        assert_rounding_bound(to_np(o[b]).reshape(H, hd), ref, u, u * vmax + 1e-5,
                              f"decode attention seq {b}")


def test_argmax_ties_and_sizes(cuda_device):
    import torch
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((5, 65536)).astype(np.float32)).cuda()
    x[1, :] = 0.0
    x[2, 100] = x[2, 70000 % 65536] = 50.0   # tie -> lowest index
    x[3, 65535] = 99.0
    out = torch.empty(5, dtype=torch.int32, device="cuda")
    nc.nc_op_argmax(x, 5, 65536, out)
    torch.cuda.synchronize()
    want = O.greedy_next(to_np(x))
    assert out.cpu().numpy().tolist() == want.tolist()
    assert out[1].item() == 0 and out[2].item() == min(100, 70000 % 65536)


def test_host_errors_enqueue_nothing(cuda_device):
    import torch
    x = torch.zeros(4, 8, device="cuda")
    with pytest.raises(nc.NcError) as e:
        nc.nc_op_rmsnorm(x, x, nc.NC_F32, 4, 6, 1e-5)   # d not a multiple of 4
    assert e.value.code == nc.NC_ERR_INVALID_ARG
    with pytest.raises(nc.NcError) as e:
        nc.nc_op_gemm(x, x, x, 4, 8, 8, nc.NC_BF16)      # K % 64 != 0
    assert e.value.code == nc.NC_ERR_UNSUPPORTED
