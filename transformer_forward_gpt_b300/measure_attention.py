"""Times the tcgen05 prefill attention kernel on its own, through the C ABI.

    python -m transformer_forward_gpt_b300.measure_attention [B H Hkv T]

Defaults to the d20 prefill shape (4 sequences, 10 query heads, 10 KV heads,
2048 positions): seeded N(0, 1) fp16 q, k, v; three warm-up calls, then 20 calls
timed with CUDA events on the current stream. Prints the time per call and the
algorithmic rate (4 * head_dim FLOPs per visible (query, key) pair and head).
"""
import sys

from transformer_forward_gpt_b300 import binding as nc


def main(argv):
    import torch
    B, H, Hkv, T = (int(x) for x in argv) if argv else (4, 10, 10, 2048)
    hd = 128
    torch.manual_seed(0)
    q = torch.randn(B, H, T, hd, device="cuda").half()
    k = torch.randn(B, Hkv, T, hd, device="cuda").half()
    v = torch.randn(B, Hkv, T, hd, device="cuda").half()
    o = torch.empty(B, T, H * hd, device="cuda", dtype=torch.half)
    for _ in range(3):
        nc.nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, T, hd, nc.NC_F16)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 20
    e0.record()
    for _ in range(n):
        nc.nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, T, hd, nc.NC_F16)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    flop = 4.0 * hd * H * B * T * (T + 1) / 2
    print(f"attention B{B} H{H} Hkv{Hkv} T{T}: {ms * 1e3:.1f} us per call, "
          f"{flop / (ms / 1e3) / 1e12:.0f} TFLOP/s")


if __name__ == "__main__":
    main(sys.argv[1:])
