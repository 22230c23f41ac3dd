"""Per-task timing of one decode step (amk_debug_trace_step) and a summary.

    python -m decode_megakernel_gb300.trace --workload llama8b-bf16

loads the workload's model (seeded weights, a KV cache whose first P
positions are declared valid), runs a few untraced warm-up steps, records
one step and prints, per task type averaged over layers: the time
consumers spend polling for their tagged inputs, the time their work takes
after the inputs arrived, the hand-off lag (from the last task of the
previous phase finishing to the median CTA of this phase having its
inputs), the span each phase adds to the step's critical path, and how
long the producer warps sat on a full ring.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

TYPE_NAMES = {0: "qkv", 1: "attn", 6: "combine", 2: "o_proj", 3: "gate_up", 4: "down",
              5: "lm_head"}
WORDS = 16  # int64 words per trace row


def trace_step(dec, token: int, pos: int, logits):
    """Run one traced decode step; returns int64 [num_ctas, 1 + S, 16]."""
    import torch

    from . import amk
    nbytes, stride = amk.amk_debug_trace_bytes(dec.ctx)
    buf = torch.zeros(nbytes // 8, dtype=torch.int64, device=logits.device)
    amk.check(amk.amk_debug_trace_step(dec.ctx, token, pos, logits.data_ptr(), buf.data_ptr(),
                                       nbytes), dec.ctx)
    return buf.cpu().numpy().reshape(-1, 1 + stride, WORDS)


def summarize(tr: np.ndarray, n_layers: int) -> str:
    hdr = tr[:, 0, :]
    t0 = hdr[:, 0].min()
    step_us = (hdr[:, 2].max() - t0) / 1e3
    clk_ghz = np.median((hdr[:, 3] - hdr[:, 1]) / np.maximum(hdr[:, 2] - hdr[:, 0], 1))
    rows = []
    for c in range(tr.shape[0]):
        for i in range(int(hdr[c, 4])):
            r = tr[c, 1 + i]
            rows.append((c, int(r[7]) & 0xFF, int(r[7]) >> 8, r))
    out = [f"step {step_us:.1f} us on {tr.shape[0]} CTAs; SM clock ~{clk_ghz:.2f} GHz"]
    out.append(f"{'task':8s} {'wait':>8s} {'work':>8s} {'work max':>9s} {'store':>7s} "
               f"{'lag':>7s} {'span':>8s} {'blocked':>8s} {'starved':>8s}   (us, mean over layers; "
               f"wait/work/store/blocked/starved mean over CTAs)")
    # phase order along the critical path
    order = [0, 1, 6, 2, 3, 4]
    last_end = None
    att = []
    spans = {k: [] for k in order + [5]}
    lags = {k: [] for k in order + [5]}
    stats = {k: [] for k in order + [5]}
    for layer in range(n_layers):
        for ty in order + ([5] if layer == n_layers - 1 else []):
            sel = [r for (c, t, lyr, r) in rows if t == ty and lyr == layer]
            if not sel:
                continue
            a = np.array(sel, dtype=np.float64)
            wait = (a[:, 1] - a[:, 0]) / 1e3
            work = (a[:, 2] - a[:, 1]) / 1e3
            store = (a[:, 3] - a[:, 2]) / 1e3
            blocked = a[:, 6] / 1e3
            starved = a[:, 8] / clk_ghz / 1e3
            if ty == 1:
                att.append(((a[:, 11] - a[:, 0]).mean() / 1e3, (a[:, 9] - a[:, 11]).mean() / 1e3,
                            (a[:, 10] - a[:, 9]).mean() / 1e3))
            end = a[:, 3].max()
            start_ref = last_end if last_end is not None else a[:, 0].min()
            spans[ty].append((end - start_ref) / 1e3)
            lags[ty].append((np.median(a[:, 1]) - start_ref) / 1e3)
            last_end = end
            stats[ty].append((wait.mean(), work.mean(), work.max(), store.mean(), blocked.mean(),
                              starved.mean()))
    total_span = 0.0
    for ty in order + [5]:
        if not stats[ty]:
            continue
        s = np.array(stats[ty]).mean(0)
        sp = float(np.mean(spans[ty]))
        total_span += sp * len(spans[ty])
        out.append(f"{TYPE_NAMES[ty]:8s} {s[0]:8.2f} {s[1]:8.2f} {s[2]:9.2f} {s[3]:7.2f} "
                   f"{float(np.mean(lags[ty])):7.2f} {sp:8.2f} {s[4]:8.2f} {s[5]:8.2f}")
    out.append(f"sum of spans {total_span:.1f} us")
    if att:
        a = np.array(att).mean(0)
        out.append(f"attention: all inputs arrived {a[0]:.2f} after begin, chunk loop {a[1]:.2f}, "
                   f"warp merge + partial store {a[2]:.2f} us")
    return "\n".join(out)


def main(argv=None):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch

    from workload import configs as wc
    from workload import synth

    from . import amk

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b-bf16")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--num-ctas", type=int, default=0)
    ap.add_argument("--ring-slots", type=int, default=0)
    ap.add_argument("--l2-prefetch-tiles", type=int, default=0)
    ap.add_argument("--save", default="")
    args = ap.parse_args(argv)
    wl = wc.workload(args.workload)
    cfg = wl.model
    dev = torch.device("cuda:0")
    w = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=dev)
    kv = synth.synthetic_kv_cache(cfg, wl.prompt_len, wl.max_seq, device=dev)
    dec = amk.Decoder(w, wl.max_seq, kv_cache=kv,
                      sched=amk.make_schedule_config(num_ctas=args.num_ctas,
                                                     ring_slots=args.ring_slots,
                                                     l2_prefetch_tiles=args.l2_prefetch_tiles))
    del w
    torch.cuda.empty_cache()
    dec.set_kv_length(wl.prompt_len)
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    tok = int(synth.decode_tokens(cfg, 1)[0])
    for _ in range(args.warmup):
        dec.decode_step(tok, wl.prompt_len, logits)
    dec.sync()
    tr = trace_step(dec, tok, wl.prompt_len, logits)
    if args.save:
        np.save(args.save, tr)
    print(summarize(tr, cfg.n_layers))
    dec.close()


if __name__ == "__main__":
    main()
