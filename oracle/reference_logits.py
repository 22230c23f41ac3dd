"""Oracle logits of the schedule search's parity sequence (TEST
INFRASTRUCTURE: it runs the CPU oracle only).

    python -m oracle.reference_logits --workload llama8b-bf16 --out ref.npy

The sequence: the workload's seeded weights, its seeded synthetic KV history
of P positions, then the first 4 seeded decode tokens teacher-forced at
positions P .. P + 3.  Writes float64 [4, vocab]: the reference the schedule
search (decode_megakernel_gb300/tune.py) holds every candidate to.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

PARITY_STEPS = 4


def reference_logits(wl, device="cuda") -> np.ndarray:
    """Oracle logits [PARITY_STEPS, vocab] of the parity sequence.  The
    seeded inputs are generated on `device`, as the schedule search
    generates them (a seeded generator draws different numbers on a GPU and
    on the CPU), then copied to the host; the oracle runs on the CPU."""
    from workload import synth

    from . import binding
    cfg = wl.model
    w = synth.model_weights(cfg, seed=synth.WEIGHT_SEED, device=device).to("cpu")
    kv = synth.synthetic_kv_cache(cfg, wl.prompt_len, wl.max_seq, device=device).cpu()
    om = binding.OracleModel(w, wl.max_seq)
    toks = synth.decode_tokens(cfg, PARITY_STEPS).tolist()
    out = [om.decode_step(kv, t, wl.prompt_len + i) for i, t in enumerate(toks)]
    return np.stack(out)


def main(argv=None):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    from workload import configs as wc
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b-bf16")
    ap.add_argument("--out", required=True)
    ap.add_argument("--device", default="cuda",
                    help="where the seeded inputs are generated (the schedule search generates them on cuda)")
    args = ap.parse_args(argv)
    ref = reference_logits(wc.workload(args.workload), args.device)
    np.save(args.out, ref)
    print(f"wrote {args.out}: {ref.shape}")


if __name__ == "__main__":
    main()
