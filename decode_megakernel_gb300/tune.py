"""Schedule search: measured tuning of the schedule, gated by the safety
gate and by parity with a reference.

    python -m oracle.reference_logits --workload llama8b-bf16 --out ref.npy
    python -m decode_megakernel_gb300.tune --workload llama8b-bf16 --reference ref.npy --trials 12

The AutoMegaKernel pages tune a ScheduleConfig (tiling, SM assignment,
pipelining depth) in an outer loop that proposes a change, checks it
against a CPU reference, measures its latency and keeps or reverts it
(AMK "Layer 2" and the autoresearch loop).  This is that loop without the
agent.  Candidates are

  * knob settings from a fixed neighbourhood of the defaults (CTA count,
    attention splits, rows per GEMV task, weight-ring depth, L2 prefetch);
  * structural edits of the lowering: which CTA runs which task, and in
    which order (schedule_ir: queue rotations, merge tasks moved to other
    CTAs), loaded with amk_load_weights_requeued.

Each candidate is

  1. lowered and run through the safety gate (amk_validate_serialized, or
     amk_validate_requeued for a structural edit): a rejected schedule is
     never launched;
  2. loaded and run on the parity sequence (a seeded synthetic KV history
     of P positions, then PARITY_STEPS teacher-forced steps); every step's
     logits must match the reference's within 5e-2 with the same top-1,
     else the candidate is discarded.  The reference is the CPU oracle's
     logits for the same sequence (the oracle belongs to the tests, so it
     is computed outside this module and handed in: oracle/reference_logits.py
     writes it for a workload); the default schedule's logits are a second
     check;
  3. timed with CUDA events over --steps steps and kept if faster than the
     best so far.

It prints one line per candidate and, last, the best candidate as JSON.
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import random
import sys

PARITY_STEPS = 4
TOL = 5e-2


def knob_candidates(sms: int, n_kv: int, rng: random.Random, trials: int):
    grid = {
        "num_ctas": sorted({sms, sms - 2, sms - 8, (sms // 2) * 2}),
        "attn_splits": sorted({0, max(1, sms // n_kv // 2), max(1, sms // n_kv)}),
        "max_rows_per_task": [0, 128, 64],
        "ring_slots": [0, 4, 8],   # copies in flight (0: the default, 6)
        "l2_prefetch_tiles": [0, 16],
    }
    keys = list(grid)
    combos = list(itertools.product(*(grid[k] for k in keys)))
    rng.shuffle(combos)
    return [{"knobs": dict(zip(keys, c))} for c in combos[:max(0, trials)]]


def structural_candidates(num_ctas: int):
    """Edits of the default lowering's placement (schedule_ir)."""
    out = [{"knobs": {}, "edit": f"rotate_queues:{k}"} for k in (1, num_ctas // 2)]
    out.append({"knobs": {}, "edit": "spread_combines:1"})
    return out


def apply_edit(blob: bytes, edit: str) -> bytes:
    from . import schedule_ir as ir
    name, _, arg = edit.partition(":")
    s = ir.parse(blob)
    if name == "rotate_queues":
        s = ir.rotate_queues(s, int(arg))
    elif name == "spread_combines":
        s = ir.spread_combines(s, int(arg))
    elif name == "hoist_next_layer":
        s = ir.hoist_next_layer(s)
    else:
        raise ValueError(f"unknown edit {edit}")
    return ir.serialize(s)


def parity_inputs(wl, device):
    """The parity sequence: seeded weights, the synthetic KV history of P
    positions, PARITY_STEPS teacher-forced tokens at positions P.."""
    from workload import synth
    cfg = wl.model
    w = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=device)
    kv = synth.synthetic_kv_cache(cfg, wl.prompt_len, wl.max_seq, device=device)
    toks = synth.decode_tokens(cfg, max(PARITY_STEPS, 1)).tolist()
    return w, kv, toks


class Search:
    """One search over a workload: gate, parity against `reference`
    (float64 [PARITY_STEPS, vocab]), timing.  `launched` counts the
    candidates that reached the GPU."""

    def __init__(self, wl, reference, steps: int = 16, device=None):
        import torch

        from . import amk
        self.amk = amk
        self.wl = wl
        self.cfg = wl.model
        self.dev = device or torch.device("cuda:0")
        self.reference = reference
        self.steps = steps
        self.w, self.kv_init, self.parity_toks = parity_inputs(wl, self.dev)
        from workload import synth
        self.timed_toks = synth.decode_tokens(self.cfg, max(steps, PARITY_STEPS)).tolist()
        self.launched = 0
        self.default_logits = None

    def gate(self, cand):
        """(lowering bytes or None, requeued?, report): the safety gate's verdict."""
        amk = self.amk
        sched = amk.make_schedule_config(**cand.get("knobs", {}))
        c = amk.make_config(self.cfg, self.wl.max_seq)
        blob = amk.amk_build_schedule(c, sched)
        if "edit" in cand:
            blob = apply_edit(blob, cand["edit"])
            st, rep = amk.amk_validate_requeued(c, sched, blob)
            return (blob if st == amk.AMK_OK else None), True, rep
        st, rep = amk.amk_validate_serialized(blob)
        return (blob if st == amk.AMK_OK else None), False, rep

    def trial(self, cand):
        """Returns (status, microseconds per step or None, parity report)."""
        import numpy as np
        import torch
        amk = self.amk
        blob, requeued, rep = self.gate(cand)
        if blob is None:
            return "rejected by the safety gate: " + rep, None, None
        sched = amk.make_schedule_config(**cand.get("knobs", {}))
        self.launched += 1
        dec = amk.Decoder(self.w, self.wl.max_seq, kv_cache=self.kv_init.clone(), sched=sched,
                          schedule=blob if requeued else None)
        P = self.wl.prompt_len
        dec.set_kv_length(P)
        logits = torch.empty(self.cfg.vocab, dtype=torch.float32, device=self.dev)
        got = []
        for i, t in enumerate(self.parity_toks[:PARITY_STEPS]):
            dec.decode_step(t, P + i, logits)
            got.append(logits.double().cpu().numpy())
        dec.sync()
        got = np.stack(got)
        err = float(np.abs(got - self.reference).max())
        top1 = bool((got.argmax(1) == self.reference.argmax(1)).all())
        dflt = None if self.default_logits is None else float(np.abs(got - self.default_logits).max())
        report = {"max_dlogit_vs_reference": err, "top1_equal": top1, "max_dlogit_vs_default": dflt}
        if not (np.isfinite(err) and err <= TOL and top1):
            dec.close()
            return "discarded: logits differ from the reference", None, report
        if self.default_logits is None:
            self.default_logits = got
        stream = dec.stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dec.set_kv_length(P)
        e0.record(stream)
        for i in range(self.steps):
            dec.decode_step(self.timed_toks[i], P + i % self.wl.decode_steps, logits)
        e1.record(stream)
        dec.sync()
        us = e0.elapsed_time(e1) * 1e3 / self.steps
        dec.close()
        return "ok", us, report

    def run(self, candidates, log=print):
        """The default schedule first, then each candidate; keeps the fastest."""
        status, base_us, rep = self.trial({"knobs": {}})
        if base_us is None:
            raise RuntimeError(f"default schedule failed: {status} {rep}")
        log(f"default: {base_us:.1f} us/step, {json.dumps(rep)}")
        best = ({"knobs": {}}, base_us)
        results = [({"knobs": {}}, status, base_us, rep)]
        for cand in candidates:
            status, us, rep = self.trial(cand)
            results.append((cand, status, us, rep))
            if us is None:
                log(f"{json.dumps(cand)}: {status}")
                continue
            kept = us < best[1]
            if kept:
                best = (cand, us)
            log(f"{json.dumps(cand)}: {us:.1f} us/step, {json.dumps(rep)}{'  (best)' if kept else ''}")
        return best, base_us, results


def main(argv=None):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import numpy as np
    import torch

    from workload import configs as wc

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b-bf16")
    ap.add_argument("--reference", required=True,
                    help="float64 [4, vocab] .npy of reference logits for the parity sequence "
                         "(oracle/reference_logits.py writes the oracle's)")
    ap.add_argument("--trials", type=int, default=12)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-structural", action="store_true")
    args = ap.parse_args(argv)

    wl = wc.workload(args.workload)
    ref = np.load(args.reference)
    if ref.shape != (PARITY_STEPS, wl.model.vocab):
        raise SystemExit(f"reference logits have shape {ref.shape}, want {(PARITY_STEPS, wl.model.vocab)}")
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rng = random.Random(args.seed)
    cands = knob_candidates(sms, wl.model.n_kv_heads, rng, args.trials)
    if not args.no_structural:
        cands += structural_candidates(sms)
    search = Search(wl, ref, steps=args.steps, device=dev)
    best, base_us, _ = search.run(cands)
    print(json.dumps({"workload": args.workload, "best": best[0], "us_per_step": best[1],
                      "default_us_per_step": base_us, "launched": search.launched}))


if __name__ == "__main__":
    main()
