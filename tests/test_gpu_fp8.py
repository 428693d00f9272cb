"""fp8 (E4M3) projection variant on the GPU against the oracle: the quantised codes
and scales bit for bit, and the tcgen05 kind::f8f6f4 matrix-vector product within
fp32 accumulation error (the codes and scales being identical, only the order of
the fp32 sums differs from the exact product)."""
import numpy as np
import pytest

from oracle import fp8_oracle as F8
from tests.gpu_helpers import to_np
from transformer_forward_gpt_b300 import binding as nc
from transformer_forward_gpt_b300 import synth

pytestmark = pytest.mark.gpu


def decode_e4m3(codes):
    """Values of E4M3 bytes from the bit layout: sign, 4 exponent bits (bias 7),
    3 mantissa bits; exponent 0 is subnormal; 0x7f / 0xff are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def _quantize_gpu(x_t, dtype):
    import torch
    rows, cols = x_t.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    nc.nc_op_quantize_e4m3(x_t, dtype, rows, cols, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_quantize_codes_and_scales_bit_exact(cuda_device, dtype):
    import torch
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((300, 1280)) * rng.uniform(0.01, 30, size=(300, 1))).astype(np.float32)
    w[7] = 0.0                                 # a zero row: scale 1, all codes 0
    w[9, 3] = 1e-30                            # far below the smallest subnormal after scaling
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    x_t = torch.from_numpy(w).to(tdt).cuda()
    w_in = x_t.float().cpu().numpy()           # the values the kernel sees
    ndt = {"f32": nc.NC_F32, "bf16": nc.NC_BF16, "f16": nc.NC_F16}[dtype]
    q, s = _quantize_gpu(x_t, ndt)
    want_q, want_s = F8.quantize_rows(w_in)
    assert np.array_equal(s, want_s)
    assert np.array_equal(decode_e4m3(q), want_q)
    assert s[7] == 1.0 and not q[7].any()


@pytest.mark.parametrize("N,K,B", [(128, 128, 1), (1280, 1280, 32), (5120, 1280, 32),
                                   (1280, 5120, 7), (300, 256, 100), (65536, 1280, 32)])
def test_gemv_matches_oracle(cuda_device, N, K, B):
    import torch
    rng = np.random.default_rng(N + K + B)
    w = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    x = rng.standard_normal((B, K)).astype(np.float32)
    wq_t = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    ws_t = torch.empty(N, dtype=torch.float32, device="cuda")
    nc.nc_op_quantize_e4m3(torch.from_numpy(w).cuda(), nc.NC_F32, N, K, wq_t, ws_t)
    x_t = torch.from_numpy(x).cuda()
    y_t = torch.full((B, N), float("nan"), device="cuda")
    nbytes = nc.nc_op_gemv_e4m3_scratch_bytes(N, K, B)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_gemv_e4m3(wq_t, ws_t, N, K, x_t, B, y_t, scratch, nbytes)
    torch.cuda.synchronize()
    wq, ws = F8.quantize_rows(w)
    ref = F8.gemv_e4m3(wq, ws, x)
    got = to_np(y_t)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref).max() / rms
    assert err < 1e-4, err


def test_gemv_argument_checks(cuda_device):
    import torch
    wq = torch.zeros(128, 256, dtype=torch.uint8, device="cuda")
    ws = torch.ones(128, device="cuda")
    x = torch.zeros(4, 256, device="cuda")
    y = torch.zeros(4, 128, device="cuda")
    nbytes = nc.nc_op_gemv_e4m3_scratch_bytes(128, 256, 4)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert nc.nc_op_gemv_e4m3_scratch_bytes(128, 256, 129) == 0
    with pytest.raises(nc.NcError):      # K not a multiple of 128
        nc.nc_op_gemv_e4m3(wq, ws, 128, 200, x, 4, y, scratch, nbytes)
    with pytest.raises(nc.NcError):      # more than 128 tokens
        nc.nc_op_gemv_e4m3(wq, ws, 128, 256, x, 129, y, scratch, nbytes)
    with pytest.raises(nc.NcError):      # scratch too small
        nc.nc_op_gemv_e4m3(wq, ws, 128, 256, x, 4, y, scratch, nbytes - 1)
    nc.nc_op_gemv_e4m3(wq, ws, 128, 256, x, 4, y, scratch, nbytes)
    torch.cuda.synchronize()
    assert float(y.abs().max()) == 0.0


def test_fp8_projection_of_a_model_weight(cuda_device):
    """The d20 FC weight (bf16) in fp8: the product stays within the E4M3 rounding
    bound of the 16-bit product (RMS error below 5.1% of RMS, the oracle's bound)."""
    import torch
    shape = synth.with_changes(synth.D20, n_layer=1, vocab=512)
    W = synth.make_weights(shape)
    w_fc = W.layers[0][4]                      # [F, d]
    F_, d = w_fc.shape
    x = np.random.default_rng(2).standard_normal((32, d)).astype(np.float32)
    wq_t = torch.empty(F_, d, dtype=torch.uint8, device="cuda")
    ws_t = torch.empty(F_, dtype=torch.float32, device="cuda")
    w_t = torch.from_numpy(W.bits["layers.0.w_fc"].view(np.int16)).view(torch.bfloat16).cuda()
    nc.nc_op_quantize_e4m3(w_t, nc.NC_BF16, F_, d, wq_t, ws_t)
    y_t = torch.empty(32, F_, device="cuda")
    nbytes = nc.nc_op_gemv_e4m3_scratch_bytes(F_, d, 32)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    nc.nc_op_gemv_e4m3(wq_t, ws_t, F_, d, torch.from_numpy(x).cuda(), 32, y_t, scratch, nbytes)
    torch.cuda.synchronize()
    ref = x.astype(np.float64) @ w_fc.T.astype(np.float64)
    got = to_np(y_t)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.sqrt(np.mean((got - ref) ** 2)) / rms < 0.051
