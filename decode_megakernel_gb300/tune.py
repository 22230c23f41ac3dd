"""Schedule search: measured tuning of the schedule knobs, gated by the
safety gate and by parity.

    python -m decode_megakernel_gb300.tune --workload llama8b-bf16 --trials 12

The AutoMegaKernel pages tune a ScheduleConfig (tiling, SM assignment,
prefetch depth) in an outer loop that keeps a change only when it is both
accepted by the static validator and measured faster ("autoresearch";
AMK "Layer 3").  This is that loop without the agent: candidates come from
a fixed neighbourhood of the defaults (CTA count, attention splits, rows
per GEMV task, weight-ring depth, L2 prefetch budget), and each one is

  1. lowered and run through the safety gate (amk_build_schedule +
     amk_validate_serialized) — a rejected schedule is never launched;
  2. loaded and run; its logits after a fixed sequence of steps must match
     the default schedule's within 1e-3 relative (the knobs change only
     the order of fp32 sums, never the arithmetic), else it is discarded;
  3. timed with CUDA events over --steps steps; kept if faster than the
     best so far.

It prints one line per candidate and, last, the best knobs as JSON (a
schedule config to pass to amk_load_weights).
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import random
import sys


def candidates(sms: int, n_kv: int, rng: random.Random, trials: int):
    grid = {
        "num_ctas": sorted({sms, sms - 2, sms - 8, (sms // 2) * 2}),
        "attn_splits": sorted({0, max(1, sms // n_kv // 2), max(1, sms // n_kv)}),
        "max_rows_per_task": [0, 128, 64],
        "ring_slots": [0, 6, 4],
        "l2_prefetch_tiles": [0, 16],
    }
    keys = list(grid)
    combos = list(itertools.product(*(grid[k] for k in keys)))
    rng.shuffle(combos)
    out = [dict(zip(keys, c)) for c in combos[:max(0, trials)]]
    return out


def main(argv=None):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import numpy as np
    import torch

    from workload import configs as wc
    from workload import synth

    from . import amk

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b-bf16")
    ap.add_argument("--trials", type=int, default=12)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)

    wl = wc.workload(args.workload)
    cfg = wl.model
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=dev)
    kv_init = synth.synthetic_kv_cache(cfg, wl.prompt_len, wl.max_seq, device=dev)
    toks = synth.decode_tokens(cfg, args.steps).tolist()
    P = wl.prompt_len

    def trial(knobs):
        sched = amk.make_schedule_config(**knobs)
        c = amk.make_config(cfg, wl.max_seq)
        blob = amk.amk_build_schedule(c, sched)
        st, rep = amk.amk_validate_serialized(blob)
        if st != amk.AMK_OK:
            return None, f"rejected by the safety gate: {rep}"
        dec = amk.Decoder(w, wl.max_seq, kv_cache=kv_init.clone(), sched=sched)
        dec.set_kv_length(P)
        logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
        for i, t in enumerate(toks[:4]):        # warm-up, also the parity sequence
            dec.decode_step(t, P + i, logits)
        dec.sync()
        ref = logits.clone()
        stream = dec.stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dec.set_kv_length(P)
        e0.record(stream)
        for i, t in enumerate(toks):
            dec.decode_step(t, P + i, logits)
        e1.record(stream)
        dec.sync()
        us = e0.elapsed_time(e1) * 1e3 / len(toks)
        dec.close()
        return (us, ref), "ok"

    base, why = trial({})
    if base is None:
        raise SystemExit(f"default schedule failed: {why}")
    base_us, base_ref = base
    print(f"default: {base_us:.1f} us/step")
    best = ({}, base_us)
    rng = random.Random(args.seed)
    for knobs in candidates(sms, cfg.n_kv_heads, rng, args.trials):
        res, why = trial(knobs)
        if res is None:
            print(f"{json.dumps(knobs)}: {why}")
            continue
        us, ref = res
        rel = float((ref - base_ref).abs().max() / base_ref.abs().max())
        if not np.isfinite(rel) or rel > 1e-3:
            print(f"{json.dumps(knobs)}: logits differ from the default schedule's (rel {rel:.2e}); discarded")
            continue
        kept = us < best[1]
        if kept:
            best = (knobs, us)
        print(f"{json.dumps(knobs)}: {us:.1f} us/step, rel diff {rel:.1e}{'  (best)' if kept else ''}")
    print(json.dumps({"workload": args.workload, "best_knobs": best[0], "us_per_step": best[1],
                      "default_us_per_step": base_us}))


if __name__ == "__main__":
    main()
