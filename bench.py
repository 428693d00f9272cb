#!/usr/bin/env python
"""Benchmark of the GPT forward pass on B300: d20 prefill tokens/s and d20-MQA
KV-cache decode tokens/s, with their roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole path over one batch of synthetic input:
  (a) prefill of the d20 model, batch 4 x 2048 tokens, every position's logits;
  (b) 128 greedy decode steps of the d20 MQA model, batch 32, over a KV cache
      prefilled (once, before timing) to 1024 positions; each step replays the
      same decode window (cache length set back to 1024, same start tokens).
`value` is (a)'s tokens/s; the decode rate is reported under "decode". Inputs
(weights ~1.1-1.7 GB, logits 2.1 GB, KV cache) are larger than the 126 MB L2.

N > 1 (torchrun): every rank runs an independent replica of the same work on
its own GPU (the path has no cross-sequence exchange); times are the max over
ranks and `value` sums the ranks' tokens. `--impl reference` times the CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "d20 bf16 prefill tok/s & KV-cache decode tok/s on 1 B300; % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}
DECODE_STEPS = 128


# ------------------------------------------------------------------- helpers
def load_peaks():
    """Measured peaks (hbm_gbs, bf16_tflops, bf16_tflops_sustained) if the file is
    present and readable; a key it lacks, or a value that is not a positive number,
    takes the fallback figure and the source says so."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        return dict(PEAKS_FALLBACK), "fallback"
    try:
        with open(path) as f:
            p = json.load(f)
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"
    out, missing = {}, []
    for k, v in PEAKS_FALLBACK.items():
        x = p.get(k) if isinstance(p, dict) else None
        if isinstance(x, (int, float)) and x > 0:
            out[k] = float(x)
        else:
            out[k] = v
            missing.append(k)
    return out, ("measured" if not missing else "measured (fallback for " + ", ".join(missing) + ")")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world, device=None):
    """Element-wise max over ranks (identity for one rank)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def prefill_flops(shape, B, T):
    """Algorithmic FLOPs of one prefill: 2 per multiply-add over the projection
    and LM-head matrices, plus causal attention (4*hd per visible (q, k) pair and head)."""
    d, H, Hkv, hd, F, L, V = (shape.d_model, shape.n_head, shape.n_kv_head, shape.head_dim,
                              shape.d_mlp, shape.n_layer, shape.vocab)
    M = B * T
    per_layer = d * (H + 2 * Hkv) * hd + H * hd * d + 2 * d * F
    gemm = 2 * M * (L * per_layer + d * V)
    attn = 4 * hd * H * (T * (T + 1) // 2) * B * L
    return gemm, attn


def gemm_flops_by_kind(shape, M):
    d, H, Hkv, hd, F, L, V = (shape.d_model, shape.n_head, shape.n_kv_head, shape.head_dim,
                              shape.d_mlp, shape.n_layer, shape.vocab)
    return {"qkv": 2 * M * d * (H + 2 * Hkv) * hd, "oproj": 2 * M * H * hd * d,
            "fc": 2 * M * d * F, "proj": 2 * M * F * d, "lm_head": 2 * M * d * V}


def decode_bytes(shape, B, ctx):
    """Algorithmic HBM bytes of one decode step at context ctx (positions 0..ctx-1
    attended): 16-bit weights read once, K/V of every position read, the new K/V
    row written, fp32 logits written."""
    d, H, Hkv, hd, F, L, V = (shape.d_model, shape.n_head, shape.n_kv_head, shape.head_dim,
                              shape.d_mlp, shape.n_layer, shape.vocab)
    weights = 2 * (L * (d * (H + 2 * Hkv) * hd + H * hd * d + 2 * d * F) + V * d)
    kv = 2 * L * B * Hkv * hd * 2 * (ctx + 1)
    logits = 4 * B * V
    return weights + kv + logits


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        rows = [l.split(",") for l in self.file.read().strip().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import numpy as np
    import torch

    from transformer_forward_gpt_b300 import binding as nc
    from transformer_forward_gpt_b300 import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    # (a) d20 prefill
    wl_p = synth.WORKLOADS["d20_prefill"]
    sp, Bp, Tp = wl_p.shape, wl_p.batch, wl_p.seq
    profiling_aid = (args.phase != "both" or args.prefill_batch is not None
                     or args.decode_steps is not None)
    if args.prefill_batch:
        Bp = args.prefill_batch
    mp = cp = tok_p = logits_p = None
    if args.phase != "decode":
        Wp = synth.make_weights(sp)
        mp = nc.Model(Wp, max_seq=Tp, max_batch=Bp)
        del Wp
        cp = mp.cache(Bp, Tp)
        tok_p = torch.from_numpy(synth.make_tokens(sp, Bp, Tp)).to(dev)
        logits_p = torch.empty(Bp, Tp, sp.vocab, device=dev)

    # (b) d20-MQA decode over a 1024-position cache
    wl_d = synth.WORKLOADS["d20_mqa_decode"]
    sd, Bd, Td = wl_d.shape, wl_d.batch, wl_d.seq
    steps = args.decode_steps or wl_d.decode_steps
    md = cd = tok0 = tok_buf = None
    if args.phase != "prefill":
        Wd = synth.make_weights(sd)
        md = nc.Model(Wd, max_seq=Td + steps, max_batch=Bd)
        del Wd
        cd = md.cache(Bd, Td + steps)
        prompt_d = synth.make_tokens(sd, Bd, Td)
        tok0 = torch.empty(Bd, dtype=torch.int32, device=dev)
        nc.nc_prefill_last(md.handle, torch.from_numpy(prompt_d).to(dev), Bd, Td, None, tok0,
                           cd.handle)
        tok_buf = torch.empty(Bd, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def prefill_phase():
        if args.phase == "decode":
            return
        nc.nc_prefill(mp.handle, tok_p, Bp, Tp, logits_p, cp.handle, stream)

    def decode_phase():
        if args.phase == "prefill":
            return
        nc.nc_kv_cache_set_length(cd.handle, Td)
        tok_buf.copy_(tok0)
        for j in range(steps):
            nc.nc_decode_step(md.handle, tok_buf, Bd, Td + j, None, tok_buf, cd.handle, stream)

    for _ in range(args.warmup):
        prefill_phase()
        decode_phase()
    torch.cuda.synchronize()
    for m in (mp, md):
        if m is None:
            continue
        st = nc.nc_model_check(m.handle)
        if st != nc.NC_OK:
            raise RuntimeError(f"device status {st} after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    launches0 = nc.nc_launch_count()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            ev[k][0].record(stream)
            prefill_phase()
            ev[k][1].record(stream)
            decode_phase()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    launches = nc.nc_launch_count() - launches0
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    pre_ms, dec_ms, t_wall = reduce_max([pre_ms, dec_ms, t_wall], world, dev)
    clocks = clk.summary()

    if profiling_aid:
        # not a bench line: a plain summary for profiling runs
        if rank == 0:
            K = args.steps
            msg = f"profiling aid: prefill {pre_ms / K:.3f} ms/step (B{Bp}xT{Tp})"
            if args.phase != "prefill":
                msg += f", decode {dec_ms / K / steps * 1e3:.1f} us/token-step (B{Bd})"
            print(msg, flush=True)
            for m, name in ((mp, "prefill"), (md, "decode")):
                if m is None:
                    continue
                nc.nc_profile_begin(m.handle)
                (prefill_phase if name == "prefill" else decode_phase)()
                prof = nc.nc_profile_end(m.handle, stream)
                print("  " + name + ": " + ", ".join(f"{k} {v[0]:.3f} ms" for k, v in prof.items()
                                                     if v[1]), flush=True)
        return
    # per-kernel-class device time: one more step with the library's event pairs on
    nc.nc_profile_begin(mp.handle)
    prefill_phase()
    prof_p = nc.nc_profile_end(mp.handle, stream)
    nc.nc_profile_begin(md.handle)
    decode_phase()
    prof_d = nc.nc_profile_end(md.handle, stream)

    # end to end through the C ABI with host buffers
    e2e = (run_e2e(nc, synth, mp, cp, md, cd, sp, Bp, Tp, sd, Bd, Td, steps, args, dev, stream)
           if not args.no_e2e else {"prefill": None, "decode": None})
    report = (report_configs(nc, synth, peaks, peak_src, dev, stream)
              if not args.no_report else None)

    if rank != 0:
        return
    K = args.steps
    tok_pre = Bp * Tp * K * world
    tok_dec = Bd * steps * K * world
    value = tok_pre / (pre_ms / 1e3)
    dec_value = tok_dec / (dec_ms / 1e3)
    g_flops, a_flops = prefill_flops(sp, Bp, Tp)
    bf16_peak = peaks["bf16_tflops"]
    pre_tflops = (g_flops + a_flops) / (pre_ms / K / 1e3) / 1e12
    ctxs = [Td + j for j in range(steps)]
    dec_bytes = sum(decode_bytes(sd, Bd, c) for c in ctxs)
    dec_gbs = dec_bytes / (dec_ms / K / 1e3) / 1e9

    # dominant kernel class of the step (device time), its roofline
    merged = {}
    for name, prof in (("prefill", prof_p), ("decode", prof_d)):
        for kind, (ms, n) in prof.items():
            if n:
                merged[f"{name}.{kind}"] = (ms, n)
    dom, (dom_ms, dom_n) = max(merged.items(), key=lambda kv: kv[1][0])
    phase, kind = dom.split(".")
    if phase == "prefill" and kind in ("qkv", "oproj", "fc", "proj", "lm_head"):
        fl = gemm_flops_by_kind(sp, Bp * Tp)[kind]
        per_launch_flops = fl * (sp.n_layer if kind != "lm_head" else 1) / dom_n
        achieved = per_launch_flops / (dom_ms / dom_n / 1e3) / 1e12
        peak = peaks.get("bf16_tflops_sustained", bf16_peak)
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": None, "peak_source": f"{peak_src} bf16 sustained (fp16 operands, 1:1)",
                "per_launch_flops": per_launch_flops, "launch_ms": dom_ms / dom_n}
    elif phase == "prefill" and kind == "attn_prefill":
        per_launch = a_flops / dom_n
        achieved = per_launch / (dom_ms / dom_n / 1e3) / 1e12
        peak = peaks.get("bf16_tflops_sustained", bf16_peak)
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                "peak_source": f"{peak_src} bf16 sustained", "per_launch_flops": per_launch,
                "launch_ms": dom_ms / dom_n}
    else:
        # decode classes are HBM-bound: algorithmic bytes of the class per launch
        roof = decode_kind_roofline(sd, Bd, ctxs, kind, dom_ms, dom_n, peaks, peak_src)
        roof["kernel"] = dom

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tok/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round((pre_ms + dec_ms) / K, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1/sqrt(fan_in)) bf16 weights, uniform tokens)",
        "config": {"workload": f"d20 prefill B{Bp}xT{Tp} + d20-MQA decode B{Bd} ctx {Td}..{Td + steps - 1}, {steps} steps",
                   "global_batch": Bp * world, "seq_len": Tp, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush)"},
        "prefill": {"value": round(value, 1), "unit": "tok/s", "ms": round(pre_ms / K, 3),
                    "tflops": round(pre_tflops, 1), "algorithmic_tflop": round((g_flops + a_flops) / 1e12, 3),
                    "frac_of_peak": round(pre_tflops / bf16_peak, 4),
                    "peak": bf16_peak, "peak_source": f"{peak_src} bf16",
                    "frac_of_nominal_peak": round(pre_tflops / NOMINAL["bf16_tflops"], 4),
                    "operands": "fp16 GEMM operands, activations and KV cache on bf16 weights "
                                "(report.d20_prefill_bf16_mode times bf16 activations)"},
        "decode": {"value": round(dec_value, 1), "unit": "tok/s", "ms_per_token_step": round(dec_ms / K / steps, 4),
                   "gbs": round(dec_gbs, 1), "algorithmic_mb_per_step": round(dec_bytes / steps / 1e6, 1),
                   "frac_of_peak": round(dec_gbs / peaks["hbm_gbs"], 4),
                   "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                   "frac_of_nominal_peak": round(dec_gbs / NOMINAL["hbm_gbs"], 4),
                   "e2e": e2e["decode"]},
        "roofline": roof,
        "kernel_ms_per_step": {k: round(v[0], 3) for k, v in merged.items()},
        "report": report,
        "e2e": e2e["prefill"],
        "gpu_launches": int(launches),
        "clocks": clocks,
        "wall_s": round(t_wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def report_configs(nc, synth, peaks, peak_src, dev, stream, reps=5):
    """The other configurations of the workload table, each timed on its own after
    the headline step (CUDA events on the launching stream, warm-up first):
    d12 and d26 prefill (all logits) with their tensor-roofline fractions, d26
    KV-cache decode (B64, 64 steps at context 2048..2111) with its HBM fraction,
    the headline d20 prefill with literal bf16 activations and KV cache
    (act_dtype bf16) beside the default fp16 operands, and the d20 prefill with
    the training step's next-token loss in place of the logits. Inputs are larger
    than L2."""
    import numpy as np
    import torch
    out = {}

    def timed(fn, n):
        fn()
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def prefill_case(key, wl_name, act_dtype, note):
        wl = synth.WORKLOADS[wl_name]
        sh, B, T = wl.shape, wl.batch, wl.seq
        W = synth.make_weights(sh)
        m = nc.Model(W, max_seq=T, max_batch=B, act_dtype=act_dtype)
        del W
        c = m.cache(B, T)
        tok = torch.from_numpy(synth.make_tokens(sh, B, T)).to(dev)
        logits = torch.empty(B, T, sh.vocab, device=dev)
        ms = timed(lambda: nc.nc_prefill(m.handle, tok, B, T, logits, c.handle, stream), reps)
        g, a = prefill_flops(sh, B, T)
        tf = (g + a) / (ms / 1e3) / 1e12
        out[key] = {"workload": f"{sh.name} prefill B{B}xT{T}", "tok_s": round(B * T / (ms / 1e3), 1),
                    "ms": round(ms, 3), "tflops": round(tf, 1),
                    "frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
                    "peak": peaks["bf16_tflops"], "peak_source": f"{peak_src} bf16", "operands": note}
        del logits, tok
        c.close()
        m.close()
        torch.cuda.empty_cache()

    def loss_case():
        # the training step's forward pass and loss: the prefill with the LM head
        # reduced to per-position cross-entropy in its epilogue (no logits stored)
        wl = synth.WORKLOADS["d20_prefill"]
        sh, B, T = wl.shape, wl.batch, wl.seq
        W = synth.make_weights(sh)
        m = nc.Model(W, max_seq=T, max_batch=B)
        del W
        c = m.cache(B, T)
        toks = synth.make_tokens(sh, B, T)
        tgt = np.concatenate([toks[:, 1:], toks[:, :1]], axis=1)
        tok = torch.from_numpy(toks).to(dev)
        tgt_d = torch.from_numpy(np.ascontiguousarray(tgt)).to(dev)
        loss = torch.empty(B * T, device=dev)
        mean = torch.empty(1, device=dev)
        ms = timed(lambda: nc.nc_prefill_loss(m.handle, tok, tgt_d, B, T, loss, mean, c.handle, stream),
                   reps)
        g, a = prefill_flops(sh, B, T)
        tf = (g + a) / (ms / 1e3) / 1e12
        out["d20_prefill_loss"] = {"workload": f"{sh.name} prefill + next-token loss B{B}xT{T}",
                                   "tok_s": round(B * T / (ms / 1e3), 1), "ms": round(ms, 3),
                                   "tflops": round(tf, 1), "frac_of_peak": round(tf / peaks["bf16_tflops"], 4),
                                   "peak": peaks["bf16_tflops"], "peak_source": f"{peak_src} bf16",
                                   "mean_loss": round(float(mean.item()), 4),
                                   "logits_stored": False}
        if nc.nc_model_check(m.handle) != nc.NC_OK:
            raise RuntimeError("device status set during the loss configuration")
        c.close()
        m.close()
        torch.cuda.empty_cache()

    def decode_case():
        wl = synth.WORKLOADS["d26_decode"]
        sh, B, T0, steps = wl.shape, wl.batch, wl.seq, wl.decode_steps
        W = synth.make_weights(sh)
        m = nc.Model(W, max_seq=T0 + steps, max_batch=B)
        del W
        c = m.cache(B, T0 + steps)
        tok0 = torch.empty(B, dtype=torch.int32, device=dev)
        nc.nc_prefill_last(m.handle, torch.from_numpy(synth.make_tokens(sh, B, T0)).to(dev), B, T0, None,
                           tok0, c.handle, stream)
        buf = torch.empty(B, dtype=torch.int32, device=dev)

        def decode_window():
            nc.nc_kv_cache_set_length(c.handle, T0)
            buf.copy_(tok0)
            for j in range(steps):
                nc.nc_decode_step(m.handle, buf, B, T0 + j, None, buf, c.handle, stream)

        ms = timed(decode_window, 2)
        per_step = ms / steps
        byts = sum(decode_bytes(sh, B, T0 + j) for j in range(steps)) / steps
        gbs = byts / (per_step / 1e3) / 1e9
        out["d26_decode"] = {"workload": f"d26 decode B{B} ctx {T0}..{T0 + steps - 1}, {steps} steps",
                             "tok_s": round(B / (per_step / 1e3), 1), "ms_per_token_step": round(per_step, 4),
                             "gbs": round(gbs, 1), "algorithmic_mb_per_step": round(byts / 1e6, 1),
                             "frac_of_peak": round(gbs / peaks["hbm_gbs"], 4), "peak": peaks["hbm_gbs"],
                             "peak_source": f"{peak_src} HBM copy",
                             "launches_per_step": -(-B // 32)}
        if nc.nc_model_check(m.handle) != nc.NC_OK:
            raise RuntimeError("device status set during the report configurations")
        c.close()
        m.close()
        torch.cuda.empty_cache()

    def guarded(key, fn, *a):
        try:
            fn(*a)
        except Exception as e:   # a failing extra measurement is reported, not fatal
            out[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
            torch.cuda.empty_cache()

    guarded("d12_prefill", prefill_case, "d12_prefill", "d12_prefill", nc.NC_F16, "fp16 (bf16 weights)")
    guarded("d26_prefill", prefill_case, "d26_prefill", "d26_prefill", nc.NC_F16, "fp16 (bf16 weights)")
    guarded("d20_prefill_bf16_mode", prefill_case, "d20_prefill_bf16_mode", "d20_prefill", nc.NC_BF16,
            "bf16 activations and KV cache")
    guarded("d20_prefill_loss", loss_case)
    guarded("d26_decode", decode_case)
    return out


def recorded_traffic(kind):
    """Per-launch DRAM traffic (read + write) of a kernel class from its committed ncu
    summary under profiles/, or None if there is none or the kernel's source has
    changed since the counters were taken (the summary records a source hash)."""
    import hashlib
    files = {"decode_step": "decode_step_d20_mqa_B32_dram.md"}
    if kind not in files:
        return None
    path = os.path.join(ROOT, "profiles", files[kind])
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(("|", "#", " ")):
            k, _, v = line.partition(":")
            fields[k.strip()] = v.strip()
    try:
        src = os.path.join(ROOT, fields["kernel_source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if h != fields["kernel_source_sha256_16"]:
            return None
        return int(fields["traffic_bytes_per_launch_mean_ctx"])
    except (KeyError, OSError, ValueError):
        return None


def decode_kind_roofline(shape, B, ctxs, kind, ms, n, peaks, peak_src):
    d, H, Hkv, hd, F, L, V = (shape.d_model, shape.n_head, shape.n_kv_head, shape.head_dim,
                              shape.d_mlp, shape.n_layer, shape.vocab)
    steps = len(ctxs)
    per = {"qkv": 2 * L * d * (H + 2 * Hkv) * hd, "oproj": 2 * L * H * hd * d,
           "fc": 2 * L * d * F, "proj": 2 * L * F * d, "lm_head": 2 * V * d + 4 * B * V,
           "attn_decode": sum(2 * L * B * Hkv * hd * 2 * (c + 1) for c in ctxs) / steps,
           "decode_step": sum(decode_bytes(shape, B, c) for c in ctxs) / steps}
    total = per.get(kind, 0) * steps
    achieved = total / n / (ms / n / 1e3) / 1e9 if total else 0.0
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": recorded_traffic(kind), "algorithmic_bytes_per_launch": total / n if n else 0,
            "peak_source": f"{peak_src} HBM copy", "launch_ms": ms / n}


def run_e2e(nc, synth, mp, cp, md, cd, sp, Bp, Tp, sd, Bd, Td, steps, args, dev, stream):
    """Prefill through the C ABI with host buffers (pinned): tokens copied in,
    every position's logits copied out, inside the timed region. Decode through
    nc_generate_host (prompt in, generated tokens out; includes its prefill)."""
    import torch
    tok_h = torch.from_numpy(synth.make_tokens(sp, Bp, Tp)).pin_memory()
    tok_d = torch.empty(Bp, Tp, dtype=torch.int32, device=dev)
    logits_d = torch.empty(Bp, Tp, sp.vocab, device=dev)
    logits_h = torch.empty(Bp, Tp, sp.vocab).pin_memory()
    reps = max(1, min(3, args.steps))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(reps):
        tok_d.copy_(tok_h, non_blocking=True)
        nc.nc_prefill(mp.handle, tok_d, Bp, Tp, logits_d, cp.handle, stream)
        logits_h.copy_(logits_d, non_blocking=True)
        torch.cuda.synchronize()
    t_pre = (time.perf_counter() - t0) / reps
    prompt = torch.from_numpy(synth.make_tokens(sd, Bd, Td)).pin_memory()
    out = torch.empty(steps + 1, Bd, dtype=torch.int32).pin_memory()
    t0 = time.perf_counter()
    for _ in range(reps):
        nc.nc_generate_host(md.handle, prompt, Bd, Td, steps, out, cd.handle, stream)
    t_gen = (time.perf_counter() - t0) / reps
    return {"prefill": {"value": round(Bp * Tp / t_pre, 1), "unit": "tok/s",
                        "h2d_bytes_per_step": int(tok_h.numel() * 4),
                        "d2h_bytes_per_step": int(logits_h.numel() * 4)},
            "decode": {"value": round(Bd * steps / t_gen, 1), "unit": "tok/s",
                       "h2d_bytes_per_step": int(prompt.numel() * 4),
                       "d2h_bytes_per_step": int(out.numel() * 4),
                       "note": f"nc_generate_host: {Bd}x{Td} prompt prefill + {steps} greedy steps"}}


# ------------------------------------------------------- CPU oracle baseline
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else host_cores()
    except Exception:
        return host_cores()


def oracle_prefill_sample(T):
    """tok/s of the oracle on one sequence of the d20 prefill workload, T tokens."""
    from oracle import gpt_oracle as O
    from transformer_forward_gpt_b300 import synth
    shape = synth.D20
    W = synth.make_weights(shape)
    toks = synth.make_tokens(shape, 1, T)
    t0 = time.perf_counter()
    O.prefill(shape, W.wte, W.layers, W.lm_head, toks)
    dt = time.perf_counter() - t0
    return T / dt, dt


def oracle_decode_sample(n_steps, ctx=1024):
    """tok/s of the oracle decoding one sequence of the d20-MQA workload at ctx."""
    from oracle import gpt_oracle as O
    from transformer_forward_gpt_b300 import synth
    shape = synth.D20_MQA
    W = synth.make_weights(shape)
    toks = synth.make_tokens(shape, 1, ctx + n_steps)
    _, cache = O.prefill(shape, W.wte, W.layers, W.lm_head, toks[:, :ctx], t_cap=ctx + n_steps,
                         logit_positions=[ctx - 1])
    t0 = time.perf_counter()
    for j in range(n_steps):
        O.decode_step(shape, W.wte, W.layers, W.lm_head, toks[:, ctx + j], cache)
    dt = time.perf_counter() - t0
    return n_steps / dt, dt


def cpu_baseline(budget_s=30.0, T=2048):
    v, dt = oracle_prefill_sample(T)
    dv, ddt = oracle_decode_sample(8)
    return {"value": round(v, 2), "unit": "tok/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, 1 sequence x {T} tokens of the d20 prefill workload "
                      f"({dt:.1f} s)", "decode_value": round(dv, 3),
            "decode_sample": f"1 sequence of the d20-MQA workload, 8 steps at context 1024 ({ddt:.1f} s)"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    T = 512
    for _ in range(args.warmup):
        oracle_prefill_sample(T)
    times = []
    for _ in range(args.steps):
        _, dt = oracle_prefill_sample(T)
        times.append(dt)
    total = sum(times)
    value = T * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"d20 prefill, bounded sample: 1 sequence x {T} tokens per step",
                       "global_batch": 1, "seq_len": T, "parallelism": "none (host cores)"},
            "cpu_baseline": {"value": round(value, 2), "unit": "tok/s", "cores": blas_threads(),
                             "kind": "oracle", "sample": f"1 x {T} tokens of d20 prefill per step"},
            "e2e": {"value": round(value, 2), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_op_attention(args):
    """Profiling aid: the tcgen05 prefill attention alone, through the C ABI, at
    the d20 prefill shape (4 sequences, 10 query and 10 KV heads, 2048 positions,
    seeded N(0, 1) fp16 q, k, v). --warmup calls, then --steps calls timed with
    CUDA events; prints the time per call and the algorithmic rate (4 * head_dim
    FLOPs per visible (query, key) pair and head)."""
    import torch
    from transformer_forward_gpt_b300 import binding as nc
    B, H, Hkv, T, hd = 4, 10, 10, 2048, 128
    torch.manual_seed(0)
    q = torch.randn(B, H, T, hd, device="cuda").half()
    k = torch.randn(B, Hkv, T, hd, device="cuda").half()
    v = torch.randn(B, Hkv, T, hd, device="cuda").half()
    o = torch.empty(B, T, H * hd, device="cuda", dtype=torch.half)
    for _ in range(args.warmup):
        nc.nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, T, hd, nc.NC_F16)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        nc.nc_op_attention_prefill(q, k, v, o, B, H, Hkv, T, T, hd, nc.NC_F16)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    flop = 4.0 * hd * H * B * T * (T + 1) / 2
    print(f"profiling aid: attention B{B} H{H} Hkv{Hkv} T{T}: {ms * 1e3:.1f} us per call, "
          f"{flop / (ms / 1e3) / 1e12:.0f} TFLOP/s", flush=True)


def run_op_gemv_fp8(args):
    """Profiling aid: the fp8 (E4M3) projection variant alone, through the C ABI, at
    the d20 decode shapes with 32 tokens: FC (5120 x 1280), PROJ (1280 x 5120) and
    the LM head (65536 x 1280). Seeded N(0, 1/sqrt(K)) weights quantised once, N(0, 1)
    activations. Each call quantises the activations, runs the tcgen05 kind::f8f6f4
    product and adds the split-K partials. Prints the time per call and the rate of
    its bytes (1-byte weights, fp32 activations and output) against the measured HBM
    bandwidth."""
    import numpy as np
    import torch
    from transformer_forward_gpt_b300 import binding as nc
    peaks, src = load_peaks()
    B = 32
    rng = np.random.default_rng(0)
    for name, N, K in (("FC", 5120, 1280), ("PROJ", 1280, 5120), ("LM head", 65536, 1280)):
        w = torch.from_numpy((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)).cuda()
        wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
        ws = torch.empty(N, dtype=torch.float32, device="cuda")
        nc.nc_op_quantize_e4m3(w, nc.NC_F32, N, K, wq, ws)
        del w
        x = torch.randn(B, K, device="cuda")
        y = torch.empty(B, N, device="cuda")
        nbytes = nc.nc_op_gemv_e4m3_scratch_bytes(N, K, B)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        for _ in range(max(3, args.warmup)):
            nc.nc_op_gemv_e4m3(wq, ws, N, K, x, B, y, scratch, nbytes)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            nc.nc_op_gemv_e4m3(wq, ws, N, K, x, B, y, scratch, nbytes)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / args.steps * 1e3
        byts = N * K + 4 * N + 4 * B * K + 4 * B * N
        gbs = byts / (us / 1e6) / 1e9
        print(f"profiling aid: fp8 GEMV {name} {N}x{K}, {B} tokens: {us:.1f} us per call, "
              f"{gbs:.0f} GB/s = {gbs / peaks['hbm_gbs']:.2f} of {src} HBM "
              f"(16-bit weights would be {2 * N * K / 1e6:.1f} MB, fp8 {N * K / 1e6:.1f} MB)", flush=True)


def run_op_lm_loss(args):
    """Profiling aid: the d20 LM head of B4 x T2048 (8192 x 65536 x 1280, fp16
    operands, seeded N(0, 1) rows and N(0, 1/sqrt(K)) weights) through the C ABI,
    first with its fp32 logits stored (nc_op_gemm), then reduced to the next-token
    cross-entropy in the epilogue (nc_op_cross_entropy). Each is warmed up
    max(3, --warmup) times and timed over --steps calls; prints the time per call and
    the rate against the measured bf16 peak."""
    import torch
    from transformer_forward_gpt_b300 import binding as nc
    peaks, src = load_peaks()
    M, N, K = 8192, 65536, 1280
    g = torch.Generator().manual_seed(0)
    A = torch.randn(M, K, generator=g).to(torch.float16).cuda()
    W = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.float16).cuda()
    tgt = torch.randint(0, N, (M,), generator=g, dtype=torch.int32).cuda()
    C = torch.empty(M, N, device="cuda")
    loss = torch.empty(M, device="cuda")
    mean = torch.empty(1, device="cuda")
    nbytes = nc.nc_op_cross_entropy_scratch_bytes(M, N)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    calls = (("logits stored", lambda: nc.nc_op_gemm(A, W, C, M, N, K, nc.NC_F16)),
             ("cross-entropy", lambda: nc.nc_op_cross_entropy(A, W, tgt, M, N, K, nc.NC_F16, loss,
                                                              mean, scratch, nbytes)))
    for name, fn in calls:
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
        print(f"profiling aid: LM head {M}x{N}x{K}, {name}: {ms:.3f} ms per call, {tf:.0f} TFLOP/s "
              f"= {tf / peaks['bf16_tflops']:.3f} of {src} bf16", flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer runs")
    ap.add_argument("--no-report", action="store_true",
                    help="skip the other configurations (d12, d26, bf16 mode)")
    ap.add_argument("--phase", choices=("both", "prefill", "decode"), default="both",
                    help="profiling aid: run only one phase of the step (no JSON line)")
    ap.add_argument("--prefill-batch", type=int, default=None,
                    help="profiling aid: smaller prefill batch (no JSON line)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="profiling aid: fewer decode steps per step (no JSON line)")
    ap.add_argument("--op", choices=("attention", "gemv-fp8", "lm-loss"), default=None,
                    help="profiling aid: time one kernel on its own (no JSON line)")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "attention":
        run_op_attention(args)
    elif args.op == "gemv-fp8":
        run_op_gemv_fp8(args)
    elif args.op == "lm-loss":
        run_op_lm_loss(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
