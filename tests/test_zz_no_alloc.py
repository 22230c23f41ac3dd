"""The decode step that allocates nothing: amk_decode_step_static_scratch.

Some callers cannot call cudaMalloc, for instance code running under a host
application whose allocator owns all device memory and only lends out the
weight and cache buffers.  For them the library offers a decode step whose
scratch (activations, attention partials, counters, status) comes from a
fixed 1 MiB array inside libamk.so instead of the context's workspace.

Checked here through the C ABI: two calls in a row give the logits of the
regular decode step (same tolerance as the other parity tests) and write
the same K,V; the second call leaves the device's free memory and torch's
allocator untouched (the first may load the library's device code, which
holds the array); a model whose per-step scratch exceeds the array is
refused with AMK_ERR_OOM without harming the context.  Kept in a file of
its own, collected last.
"""
import numpy as np
import pytest
import torch

from workload import configs as wc
from workload import synth

pytestmark = pytest.mark.gpu

TOL = 5e-2


@pytest.fixture(scope="module")
def amk():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    from decode_megakernel_gb300 import amk as m
    return m


@pytest.mark.parametrize("model", [wc.TINY, wc.LLAMA_1B], ids=["tiny", "llama1b"])
def test_two_calls_match_the_regular_step(amk, model):
    dev = torch.device("cuda:0")
    prompt_len, max_seq = 12, 16
    w = synth.model_weights(model, seed=7, device=dev)
    regular = amk.Decoder(w, max_seq)
    no_alloc = amk.Decoder(w, max_seq)
    del w
    prompt = synth.prompt_tokens(model, prompt_len).tolist()
    regular.prefill(prompt, 0)
    no_alloc.prefill(prompt, 0)
    regular.sync()
    no_alloc.sync()
    ref = torch.empty(model.vocab, dtype=torch.float32, device=dev)
    got = torch.empty(model.vocab, dtype=torch.float32, device=dev)
    for i, tok in enumerate(synth.decode_tokens(model, 2).tolist()):
        pos = prompt_len + i
        regular.decode_step(tok, pos, ref)
        regular.sync()
        got.fill_(float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info(dev)[0]
        stats0 = torch.cuda.memory_stats(dev)
        st = amk.amk_decode_step_static_scratch(no_alloc.ctx, tok, pos, got.data_ptr())
        assert st == amk.AMK_OK, amk.last_error(no_alloc.ctx)
        free1 = torch.cuda.mem_get_info(dev)[0]
        stats1 = torch.cuda.memory_stats(dev)
        for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
            assert stats1.get(key, 0) == stats0.get(key, 0), key
        if i > 0:   # the first call may load the library's device code (and the array with it)
            assert free1 == free0, (free0, free1)
        diff = float((got - ref).abs().max())
        print(f"{model.name} call {i}: max |dlogit| vs regular step {diff:.3e}")
        assert np.isfinite(diff) and diff <= TOL
        assert int(torch.argmax(got)) == int(torch.argmax(ref))
        assert amk.amk_kv_length(no_alloc.ctx) == pos + 1
    assert torch.equal(regular.kv[:, :, :, :prompt_len + 2], no_alloc.kv[:, :, :, :prompt_len + 2])
    regular.close()
    no_alloc.close()


def test_scratch_beyond_the_maximum_is_refused(amk):
    dev = torch.device("cuda:0")
    model = wc.TINY
    # 1024 context splits per KV head: the attention partials alone exceed 1 MiB
    sched = amk.make_schedule_config(attn_splits=1024)
    w = synth.model_weights(model, seed=7, device=dev)
    dec = amk.Decoder(w, 8, sched=sched)
    dec.prefill([1, 2, 3], 0)
    out = torch.empty(model.vocab, dtype=torch.float32, device=dev)
    st = amk.amk_decode_step_static_scratch(dec.ctx, 4, 3, out.data_ptr())
    assert st == amk.AMK_ERR_OOM
    assert "at most" in amk.last_error(dec.ctx)
    # the refusal launched nothing and left the context usable
    dec.decode_step(4, 3, out)
    dec.sync()
    assert torch.isfinite(out).all()
    dec.close()
