"""Temperature sampling on the device (nc_op_sample) against the oracle (GPU).

The oracle draws by inverse CDF in fp64 from the same caller-supplied uniforms.
The device sums in fp32, so where u lies within a small tolerance of a cumulative
boundary the two may pick neighbouring indices: there the device's index must be
one the tolerance allows; everywhere else it must equal the oracle's exactly.
"""
import numpy as np
import pytest

from oracle import gpt_oracle as O
from transformer_forward_gpt_b300 import binding as nc

pytestmark = pytest.mark.gpu

TOL = 2e-5   # on cumulative probability: fp32 sums over up to 65,536 terms


def _run(logits, T, u):
    import torch
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    uu = torch.from_numpy(np.asarray(u, dtype=np.float32)).cuda()
    out = torch.full((logits.shape[0],), -1, dtype=torch.int32, device="cuda")
    nc.nc_op_sample(lg, logits.shape[0], logits.shape[1], T, uu, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(logits, T, u):
    got = _run(logits, T, u)
    # the oracle sees the same fp32 inputs (logits and u as the device reads them)
    l32 = logits.astype(np.float32).astype(np.float64)
    u32 = np.asarray(u, dtype=np.float32).astype(np.float64)
    ref = O.sample_temperature(l32, T, u32)
    if T <= 0:
        assert (got == ref).all()
        return
    p = O.softmax_rows(l32 / T)
    cdf = np.cumsum(p, axis=1)
    exact = 0
    for b in range(logits.shape[0]):
        k, r = int(got[b]), int(ref[b])
        lo_r = cdf[b, r - 1] if r > 0 else 0.0
        if abs(cdf[b, r] - u32[b]) > TOL and abs(lo_r - u32[b]) > TOL:
            assert k == r, f"row {b}: device {k}, oracle {r}"
            exact += 1
        else:   # u within TOL of a boundary: any index whose interval reaches u +- TOL
            lo_k = cdf[b, k - 1] if k > 0 else 0.0
            assert lo_k - TOL <= u32[b] <= cdf[b, k] + TOL, f"row {b}: device {k} invalid"
    # with classes wider than the tolerance most draws are away from a boundary;
    # at V = 65,536 a class holds ~1e-5 of the mass and the validity window above
    # (an index within TOL of u) is the check
    if logits.shape[1] <= 4096:
        assert exact >= logits.shape[0] // 2


@pytest.mark.parametrize("B,V", [(16, 65536), (9, 1000), (5, 7), (3, 1)])
@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
def test_sample_matches_oracle(cuda_device, B, V, T):
    rng = np.random.default_rng(B * 1000 + V)
    logits = rng.standard_normal((B, V)) * 2.0
    u = rng.random(B)
    _check(logits, T, u)


def test_sample_greedy_and_ties(cuda_device):
    """Temperature 0 is the greedy index, lowest on ties."""
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((6, 4099))
    logits[2, 17] = logits[2, 4000] = 50.0
    logits[4, :] = 1.0
    _check(logits, 0.0, rng.random(6))


def test_sample_uniform_extremes(cuda_device):
    """u = 0 takes the first index of positive probability; u just below 1 the
    last; values outside [0, 1) are clamped into it."""
    V = 2048
    logits = np.zeros((4, V))
    got = _run(logits, 1.0, [0.0, 0.99999994, -3.0, 7.0])
    assert got[0] == 0 and got[2] == 0
    assert got[1] == V - 1 and got[3] == V - 1


def test_sample_frequencies_follow_the_distribution(cuda_device):
    """A uniform grid of u over many identical rows lands in each class about p_k N
    times (the inverse-CDF property), at a temperature that flattens the logits."""
    rng = np.random.default_rng(9)
    base = rng.standard_normal(40) * 3.0
    N = 4000
    T = 2.5
    u = (np.arange(N) + 0.5) / N
    got = _run(np.tile(base, (N, 1)), T, u)
    p = O.softmax_rows(base.astype(np.float32).astype(np.float64)[None, :] / T)[0]
    counts = np.bincount(got, minlength=40)
    assert np.all(np.abs(counts - p * N) <= 2.0)


def test_sample_never_draws_a_zero_probability_tail(cuda_device):
    """u just below 1 with a tail of -inf logits: u Z can round up to Z in fp32,
    and the draw must then be the last token of nonzero probability, as the
    inverse CDF gives, never one of the masked tail."""
    V, live = 4096, 1000
    logits = np.zeros((4, V))
    logits[:, live:] = -np.inf
    logits[1, :live] = np.linspace(-3.0, 3.0, live)
    u = [0.99999994, 0.99999994, 0.9999999, 0.5]
    got = _run(logits, 1.0, u)
    assert (got < live).all(), got
    ref = O.sample_temperature(logits.astype(np.float32).astype(np.float64), 1.0,
                               np.asarray(u, dtype=np.float32).astype(np.float64))
    assert (ref < live).all()
    assert got[0] == live - 1 and got[1] == live - 1
