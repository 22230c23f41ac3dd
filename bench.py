#!/usr/bin/env python
"""Batch-1 decode benchmark: tok/s and fraction of the weight+KV-bytes
HBM roofline, on one of the five synthetic workloads.

A step is one decode step of the whole model (every layer, attention over
the KV cache, LM head) for one token: one persistent kernel launch through
the C ABI.  Default workload: the Llama-3.1-8B-shaped bf16 model with the
KV cache prefilled to 2048 random tokens; the timed steps cycle over the
128 positions 2048..2175 with teacher-forced random tokens.

Legs:
  value         device time (CUDA events on the decode stream), inputs
                resident in HBM; the 15 GB of weights per step exceed L2,
                so no flush is needed between steps.
  e2e           the same steps through amk_decode_step_host: token and
                position go host->device as launch parameters, logits
                come back into pinned host memory, timed on the host.
  roofline      algorithmic bytes of each step (weights + KV read at
                context pos+1) over the measured launch duration, against
                the measured HBM copy bandwidth.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same step
                (one layer plus 1/L of the LM-head rows per sample).
  prefill       the prompt's prefill through amk_prefill (tensor-core
                GEMMs for bf16 weights), device-timed, against the
                measured bf16 tensor peak.
--impl reference times the oracle alone (the only other implementation).
Multi-GPU: independent replicas, one per rank (the path does not shard).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tok/s (Llama-8B-shape bf16); % of weight+KV bytes/HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e spec-sheet figure (context only)
DEFAULT_LEGS = "llama1b,llama8b-int8,llama8b-int4"
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["decode_kernel.cu", "device_model.hpp", "schedule.cpp", "schedule.hpp", "ptx.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b-bf16")
    ap.add_argument("--e2e-steps", type=int, default=0, help="default: --steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--num-ctas", type=int, default=0)
    ap.add_argument("--ring-slots", type=int, default=0)
    ap.add_argument("--attn-splits", type=int, default=0, help="context splits per KV head (0: library default)")
    ap.add_argument("--l2-prefetch-tiles", type=int, default=0, help="0: library default, -1: off")
    ap.add_argument("--prefill-chunk", type=int, default=0,
                    help="tokens per tensor-core prefill chunk (0: library default; -1: decode steps)")
    ap.add_argument("--prefill-parts", type=int, default=0,
                    help="bf16 parts of the prefill GEMM activations (0: library default, 2; or 3)")
    ap.add_argument("--kv", choices=["auto", "prefill", "synthetic"], default="auto",
                    help="KV history of the first P positions: the prompt's prefill, or a seeded "
                         "synthetic history (auto: prefill for bf16 weights up to 4096 tokens)")
    ap.add_argument("--legs", default=None,
                    help="comma-separated other workloads timed after the headline (one GPU); "
                         "default: the other three bench workloads when the headline is the default")
    ap.add_argument("--no-probe", action="store_true", help="skip the read-only HBM probe")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prompt's prefill (its last run bracketed by "
                         "cudaProfilerStart/Stop) and print its JSON block")
    args = ap.parse_args(argv)
    if args.legs is None:
        args.legs = DEFAULT_LEGS if args.workload == "llama8b-bf16" else ""
    return args


# ------------------------------------------------------------------ helpers

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_megakernel_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, alg_bytes: float):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources, else None: the summary's traffic_ratio
    (DRAM bytes / algorithmic bytes, measured on a case of the same layer
    shapes) times this launch's algorithmic bytes, or its
    traffic_bytes_per_launch where it gives no ratio."""
    path = os.path.join(PROFILE_DIR, f"decode_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                v = v.split()
                fields[k.strip()] = v[0].strip("`") if v else ""
    if fields.get("kernel_sources_sha256") != kernel_source_hash():
        return None
    try:
        if "traffic_ratio" in fields:
            return int(float(fields["traffic_ratio"]) * alg_bytes)
        return int(float(fields["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(dev) -> str:
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return str(dev.index or 0)


def reduce_over_ranks(local_ms: float, local_units: float, group=None):
    """(max time, summed units) over ranks; identity when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_ms, local_units
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------ cpu oracle leg

def oracle_sample(weights_cpu, kv_cpu, pos: int, token: int, n_samples: int | None,
                  seconds: float | None, warmup: int = 0, threads: int | None = None):
    """Time the oracle on samples of one decode step: sample i runs layer
    i mod L and LM-head rows of slice i mod L (1/L of the vocabulary).
    Returns (samples timed, seconds, cores)."""
    from oracle import binding as orc
    cfg = weights_cpu.cfg
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    if threads:
        cores = threads
    orc.set_threads(cores)
    om = orc.OracleModel(weights_cpu, kv_cpu.shape[3])
    L, V = cfg.n_layers, cfg.vocab
    x = om.embed(token)
    logits = None

    def one(i):
        nonlocal logits
        layer = i % L
        om.decode_layers(kv_cpu, x, pos, layer, layer + 1)
        r0, r1 = layer * V // L, (layer + 1) * V // L
        logits = om.logits_rows(x, r0, r1, logits)

    for i in range(warmup):
        one(i)
    t0 = time.perf_counter()
    n = 0
    while True:
        one(warmup + n)
        n += 1
        el = time.perf_counter() - t0
        if n_samples is not None and n >= n_samples:
            break
        if seconds is not None and el >= seconds and n >= 1:
            break
    return n, time.perf_counter() - t0, cores


def host_weights_and_kv(wl, dev):
    import torch
    from workload import synth
    cfg = wl.model
    gen_dev = dev if dev is not None else torch.device("cpu")
    w = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=gen_dev)
    w_cpu = w.to("cpu") if gen_dev.type != "cpu" else w
    del w
    kv = synth.synthetic_kv_cache(cfg, wl.prompt_len, wl.prompt_len + 1, device="cpu")
    return w_cpu, kv


def cpu_sample_desc(wl, n):
    return (f"{n} oracle samples of the {wl.name} decode step at position {wl.prompt_len} "
            f"(each: one transformer layer + 1/{wl.model.n_layers} of the LM-head rows, fp64, "
            f"synthetic KV history of {wl.prompt_len} positions) = {n / wl.model.n_layers:.3f} tokens")


# ----------------------------------------------------------------- arms

def config_block(wl, args, num_ctas):
    return {
        "workload": wl.name,
        "model": wl.description,
        "weights_dtype": wl.model.weight_format,
        "global_batch": 1,
        "seq_len": wl.prompt_len,
        "kv_positions_timed": f"{wl.prompt_len}..{wl.prompt_len + wl.decode_steps - 1} (cyclic)",
        "parallelism": "replicas" if args.gpus > 1 else "single",
        "persistent_ctas": num_ctas,
        "l2": "no flush: every step streams the weights (> L2 capacity)",
    }


def run_reference(args, wl, rank, world):
    import torch
    if rank != 0:
        return None
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    from workload import synth
    w_cpu, kv = host_weights_and_kv(wl, dev)
    tok = int(synth.decode_tokens(wl.model, 1)[0])
    n, secs, cores = oracle_sample(w_cpu, kv, wl.prompt_len, tok, n_samples=args.steps, seconds=None,
                                   warmup=args.warmup)
    tokens = n / wl.model.n_layers
    value = tokens / secs
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(wl, args, 0),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": cpu_sample_desc(wl, n)},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def measured_peak_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_block(wl, best_ms, runs_ms, dec_chunk, parts=3):
    """The prompt's prefill: tok/s and, for the tensor-core path, useful
    flops (workload.configs.prefill_flops) per second against the measured
    bf16 tensor peak (a burst figure: the prefill is timed alone)."""
    from workload import configs as wc
    cfg, P = wl.model, wl.prompt_len
    out = {"value": P / (best_ms / 1e3), "unit": "tok/s", "tokens": P, "ms": best_ms, "runs_ms": runs_ms,
           "path": "tensor-core GEMMs (tcgen05), chunk %d, %d activation parts" % (dec_chunk, parts)
           if dec_chunk else "decode kernel, one launch per token"}
    if dec_chunk:
        fl = wc.prefill_flops(cfg, P)
        peak, src = measured_peak_tflops()
        achieved = fl / (best_ms / 1e3) / 1e12
        out["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                           "frac": achieved / peak, "peak_source": f"{src} bf16_tflops (cuBLAS, burst)",
                           "algorithmic_flops": fl,
                           "note": "GEMM activations enter as %d bf16 parts: the tensor cores "
                                   "execute %dx the GEMM flops counted here" % (parts, parts)}
    return out


def load_decoder(amk, wl, dev, stream, sched, kv_mode):
    """The workload's model loaded through the C ABI, with the first P
    positions of its KV cache valid: prefilled by amk_prefill from the
    seeded prompt (kv_mode "prefill"), or a seeded synthetic history
    declared valid with amk_set_kv_length ("synthetic": the int8 / int4
    prefill is one decode launch per token, 16K launches for the int4
    workload)."""
    import torch
    from workload import synth
    cfg, P = wl.model, wl.prompt_len
    weights = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=dev)
    kv = None
    if kv_mode == "synthetic":
        kv = synth.synthetic_kv_cache(cfg, P, wl.max_seq, device=dev)
    dec = amk.Decoder(weights, wl.max_seq, stream=stream, sched=sched, kv_cache=kv)
    del weights
    torch.cuda.empty_cache()
    if kv_mode == "synthetic":
        dec.set_kv_length(P)
    else:
        dec.prefill(synth.prompt_tokens(cfg, P).tolist(), 0)
    dec.sync()
    return dec


def kv_mode_for(wl, args):
    if args.kv != "auto":
        return args.kv
    return "prefill" if wl.model.weight_format == "bf16" and wl.prompt_len <= 4096 else "synthetic"


def time_decode(dec, wl, args, dev, stream, K, W, profile=False):
    """W untimed then K timed decode steps (teacher-forced seeded tokens,
    positions P .. P + D - 1 cyclic) with CUDA events on the decode stream;
    returns (total ms, per-step ms, positions, clocks)."""
    import torch
    from workload import synth
    cfg, P, D = wl.model, wl.prompt_len, wl.decode_steps
    toks = synth.decode_tokens(cfg, D).tolist()
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    pos_of = lambda i: P + (i % D)  # noqa: E731
    sampler = ClockSampler(gpu_id_for(dev))
    for i in range(W):
        dec.decode_step(toks[i % D], pos_of(i), logits)
    dec.sync()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    barrier()
    torch.cuda.synchronize(dev)
    # cudaProfilerStart/Stop bracket the timed region so that a profiler run
    # with collection off at start (ncu --profile-from-start off) lists
    # exactly the launches timed here; without a profiler they do nothing.
    if profile:
        torch.cuda.profiler.start()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(K):
            j = W + i
            dec.decode_step(toks[j % D], pos_of(j), logits)
            evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    if profile:
        torch.cuda.profiler.stop()
    barrier()
    clocks = sampler.stop()
    dec.sync()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]
    total_ms = evs[0].elapsed_time(evs[K])
    positions = [pos_of(W + i) for i in range(K)]
    return total_ms, per, positions, clocks


def roofline_block(wl, per, positions):
    import numpy as np
    from workload import configs as wc
    K = len(per)
    mean_bytes = sum(wc.step_bytes(wl.model, p) for p in positions) / K
    mean_launch_s = (sum(per) / K) / 1e3
    achieved = mean_bytes / mean_launch_s / 1e9
    peak, peak_src = measured_peak_gbs()
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(wl.name, mean_bytes),
            "peak_source": f"{peak_src} hbm_gbs (copy)",
            "algorithmic_bytes_per_launch": mean_bytes,
            "mean_launch_ms": mean_launch_s * 1e3,
            "launch_ms_p10_p50_p90": [float(np.percentile(per, q)) for q in (10, 50, 90)]}


def time_e2e(dec, wl, n):
    """n steps through amk_decode_step_host (launch parameters in, logits
    back into pinned host memory), timed on the host."""
    import numpy as np
    import torch
    from workload import synth
    cfg, P, D = wl.model, wl.prompt_len, wl.decode_steps
    toks = synth.decode_tokens(cfg, D).tolist()
    host_logits = torch.empty(cfg.vocab, dtype=torch.float32, pin_memory=True)
    for i in range(min(3, n)):
        dec.decode_step_host(toks[i % D], P + (i % D), host_logits)
    barrier()
    t0 = time.perf_counter()
    for i in range(n):
        dec.decode_step_host(toks[i % D], P + (i % D), host_logits)
    secs = time.perf_counter() - t0
    assert np.isfinite(host_logits.numpy()).all()
    return secs


def hbm_read_probe(amk, dev, gib=4.0, reps=10):
    """Read-only stream rate of this GPU (amk_debug_hbm_read_probe): best of
    `reps` passes over a buffer of `gib` GiB (> 30x L2), per mode."""
    import torch
    nbytes = int(gib * (1 << 30)) // 16384 * 16384
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.zeros(8 * sms, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {"bytes": nbytes}
    for mode, name in ((0, "bulk_ring_gbs"), (1, "ld128_gbs")):
        best = None
        for r in range(reps + 2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            amk.check(amk.amk_debug_hbm_read_probe(mode, buf.data_ptr(), nbytes, out.data_ptr(), out.numel(),
                                                   stream.cuda_stream))
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if mode == 0 and int(out[1::2][:sms].abs().sum()) != 0:
                raise RuntimeError("hbm read probe: a bulk copy did not land")
            ms = e0.elapsed_time(e1)
            if r >= 2:
                best = ms if best is None else min(best, ms)
        res[name] = nbytes / (best / 1e3) / 1e9
    del buf
    torch.cuda.empty_cache()
    return res


def run_leg(amk, wl, args, dev, stream, sched, K, W, n_e2e, profile=False, greedy=True, dec=None):
    """One workload: load (unless given a loaded decoder), time K decode
    steps, e2e and device greedy."""
    import torch
    from workload import synth
    kv_mode = kv_mode_for(wl, args)
    if dec is None:
        dec = load_decoder(amk, wl, dev, stream, sched, kv_mode)
    total_ms, per, positions, clocks = time_decode(dec, wl, args, dev, stream, K, W, profile)
    leg = {"workload": wl.name, "model": wl.description, "kv_history": kv_mode,
           "steps": K, "warmup": W, "total_ms": total_ms, "per_ms": per,
           "roofline": roofline_block(wl, per, positions), "clocks": clocks}
    if n_e2e > 0:
        leg["e2e_s"] = time_e2e(dec, wl, n_e2e)
        leg["e2e_steps"] = n_e2e
    if greedy:
        # greedy decoding on the device (amk_generate: the argmax feeds the
        # next step with no host round trip), device-timed on the decode stream
        D = wl.decode_steps
        n_gen = min(K, D)
        tok0 = int(synth.decode_tokens(wl.model, 1)[0])
        gen_tokens = torch.empty(n_gen, dtype=torch.int32, device=dev)
        dec.generate(tok0, wl.prompt_len, min(4, n_gen), gen_tokens)
        dec.sync()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        dec.generate(tok0, wl.prompt_len, n_gen, gen_tokens)
        g1.record(stream)
        dec.sync()
        leg["greedy_ms"] = g0.elapsed_time(g1)
        leg["greedy_steps"] = n_gen
    leg["_dec"] = dec
    return leg


def leg_summary(leg, cfg):
    """The per-workload object of the bench line (one GPU)."""
    K = leg["steps"]
    value = K / (leg["total_ms"] / 1e3)
    out = {"workload": leg["workload"], "model": leg["model"], "kv_history": leg["kv_history"],
           "metric": "batch-1 decode tok/s", "value": value, "unit": "tok/s",
           "ms_per_step": leg["total_ms"] / K, "steps": K, "warmup": leg["warmup"],
           "roofline": {k: v for k, v in leg["roofline"].items()
                        if k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                 "algorithmic_bytes_per_launch", "mean_launch_ms")},
           "clocks": leg["clocks"]}
    if "e2e_s" in leg:
        out["e2e"] = {"value": leg["e2e_steps"] / leg["e2e_s"], "unit": "tok/s", "h2d_bytes_per_step": 8,
                      "d2h_bytes_per_step": cfg.vocab * 4}
    if "greedy_ms" in leg:
        out["device_greedy_tok_s"] = leg["greedy_steps"] / (leg["greedy_ms"] / 1e3)
    return out


def run_ours(args, wl, rank, world, local_rank):
    import torch

    import __graft_entry__
    from workload import configs as wc
    from workload import synth

    __graft_entry__.build()
    from decode_megakernel_gb300 import amk

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = wl.model
    P = wl.prompt_len
    stream = torch.cuda.Stream(device=dev)
    sched = amk.make_schedule_config(num_ctas=args.num_ctas, ring_slots=args.ring_slots,
                                     attn_splits=args.attn_splits,
                                     l2_prefetch_tiles=args.l2_prefetch_tiles,
                                     prefill_chunk=args.prefill_chunk, prefill_parts=args.prefill_parts)
    num_ctas = args.num_ctas or torch.cuda.get_device_properties(dev).multi_processor_count
    kv_mode = kv_mode_for(wl, args)

    # the prompt's prefill (tensor-core GEMMs with bf16 weights), timed on
    # the decode stream; rerunning it rewrites the same K,V
    pf = None
    if kv_mode == "prefill" or args.prefill_only:
        dec = load_decoder(amk, wl, dev, stream, sched, "prefill")
        prompt = synth.prompt_tokens(cfg, P).tolist()
        pf_ms = []
        for r in range(3):
            last = args.prefill_only and r == 2
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if last:
                torch.cuda.synchronize(dev)
                torch.cuda.profiler.start()
            p0.record(stream)
            dec.prefill(prompt, 0)
            p1.record(stream)
            dec.sync()
            if last:
                torch.cuda.profiler.stop()
            pf_ms.append(p0.elapsed_time(p1))
        pf = prefill_block(wl, min(pf_ms), pf_ms, dec.prefill_chunk, args.prefill_parts or 2)
        if args.prefill_only:
            dec.close()
            return {"impl": "ours", "workload": wl.name, "prefill": pf}
    else:
        dec = None

    K = args.steps
    leg = run_leg(amk, wl, args, dev, stream, sched, K, args.warmup, args.e2e_steps or K, profile=True,
                  dec=dec)
    dec = leg.pop("_dec")
    dec.close()
    del dec
    torch.cuda.empty_cache()
    max_ms, units = reduce_over_ranks(leg["total_ms"], float(K))
    value = units / (max_ms / 1e3)
    e2e_max_ms, e2e_units = reduce_over_ranks(leg["e2e_s"] * 1e3, float(leg["e2e_steps"]))
    gen_max_ms, gen_units = reduce_over_ranks(leg["greedy_ms"], float(leg["greedy_steps"]))

    roof = leg["roofline"]
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(wl, args, num_ctas),
        "gpu_launches": K,
        "roofline": roof,
        "e2e": {"value": e2e_units / (e2e_max_ms / 1e3), "unit": "tok/s", "h2d_bytes_per_step": 8,
                "d2h_bytes_per_step": cfg.vocab * 4},
        "device_greedy": {"value": gen_units / (gen_max_ms / 1e3), "unit": "tok/s",
                          "steps": leg["greedy_steps"],
                          "what": "amk_generate: argmax fused into the LM head, launches back "
                                  "to back with no host round trip (+1 final reduction)"},
        "clocks": leg["clocks"],
        "prefill": pf,
    }
    if world == 1 and not args.no_probe:
        probe = hbm_read_probe(amk, dev)
        best = max(probe["bulk_ring_gbs"], probe["ld128_gbs"])
        probe["nominal_gbs"] = NOMINAL_HBM_GBS
        probe["read_probe_frac_of_nominal"] = best / NOMINAL_HBM_GBS
        line["hbm_read_probe"] = probe
        roof["frac_of_read_probe"] = roof["achieved"] / best
        roof["frac_of_nominal"] = roof["achieved"] / NOMINAL_HBM_GBS
    # the other workloads, one GPU only (replicas report the headline alone)
    if world == 1 and args.legs:
        legs = {}
        for name in [n.strip() for n in args.legs.split(",") if n.strip()]:
            if name == wl.name or name == args.workload:
                continue
            lw = wc.workload(name)
            lsched = amk.make_schedule_config(num_ctas=args.num_ctas)
            lk = min(K, lw.decode_steps)
            lg = run_leg(amk, lw, args, dev, stream, lsched, lk, args.warmup, lk, greedy=True)
            d = lg.pop("_dec")
            d.close()
            del d
            torch.cuda.empty_cache()
            legs[name] = leg_summary(lg, lw.model)
        line["workloads"] = legs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w_cpu, kv = host_weights_and_kv(wl, dev)
        tok = int(synth.decode_tokens(cfg, 1)[0])
        n, secs, cores = oracle_sample(w_cpu, kv, P, tok, n_samples=None, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": (n / cfg.n_layers) / secs, "unit": "tok/s", "cores": cores,
                                "kind": "oracle", "sample": cpu_sample_desc(wl, n)}
        n1, secs1, _ = oracle_sample(w_cpu, kv, P, tok, n_samples=None, seconds=args.cpu_seconds / 2,
                                     threads=1)
        line["cpu_baseline_1core"] = {"value": (n1 / cfg.n_layers) / secs1, "unit": "tok/s", "cores": 1,
                                      "kind": "oracle", "sample": cpu_sample_desc(wl, n1)}
    return line if rank == 0 else None


def main(argv=None):
    args = parse_args(argv)
    from workload import configs as wc
    wl = wc.workload(args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
            world_eff = 1
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
            world_eff = world
    else:
        world_eff = 1
    if args.impl == "reference":
        line = run_reference(args, wl, rank, world_eff)
    else:
        line = run_ours(args, wl, rank, world_eff, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
