"""The schedule search, end to end on the tiny model: candidates pass the
safety gate before anything is launched, run the parity sequence and are
held to the CPU oracle's logits (AMK's autoresearch loop: propose, check
against a CPU reference, measure, keep or revert)."""
import numpy as np
import pytest
import torch

from workload import configs as wc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_search_gates_on_the_oracle_and_rejects_an_unsafe_lowering(dev):
    from decode_megakernel_gb300 import tune
    from oracle import reference_logits
    wl = wc.workload("tiny")
    ref = reference_logits.reference_logits(wl, device=dev)
    assert ref.shape == (tune.PARITY_STEPS, wl.model.vocab)
    search = tune.Search(wl, ref, steps=8, device=dev)
    cands = [
        {"knobs": {"num_ctas": 8, "attn_splits": 3}},               # another lowering, same model
        {"knobs": {}, "edit": "rotate_queues:5"},                   # another SM assignment
        {"knobs": {"num_ctas": 8}, "edit": "spread_combines:3"},    # merges run by other CTAs
        {"knobs": {"num_ctas": 8}, "edit": "hoist_next_layer"},     # a queue order that deadlocks
    ]
    lines = []
    best, base_us, results = search.run(cands, log=lines.append)
    print("\n".join(lines))
    by = {json_key(c): (st, us, rep) for c, st, us, rep in results}
    # the unsafe lowering never reached the GPU: the gate rejected it first
    st, us, rep = by[json_key(cands[3])]
    assert st.startswith("rejected by the safety gate") and us is None and rep is None
    assert "cycle" in st or "deadlock" in st or "never" in st, st
    assert search.launched == 4   # the default and the three safe candidates
    for c in [{"knobs": {}}] + cands[:3]:
        st, us, rep = by[json_key(c)]
        assert st == "ok" and us > 0, (c, st, rep)
        assert rep["max_dlogit_vs_reference"] <= tune.TOL and rep["top1_equal"]
    # a candidate whose logits are wrong is discarded, not timed
    bad = tune.Search(wl, ref + np.eye(1, wl.model.vocab, 0) * 1.0, steps=4, device=dev)
    st, us, rep = bad.trial({"knobs": {}})
    assert st.startswith("discarded") and us is None
    assert rep["max_dlogit_vs_reference"] > tune.TOL


def json_key(c):
    import json
    return json.dumps(c, sort_keys=True)
