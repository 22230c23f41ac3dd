"""Parity of the CUDA decode path (through the C ABI) with the CPU oracle.

Bar (the decode step's contract): max |logit_gpu - logit_oracle| <= 5e-2
and >= 99% top-1 agreement under teacher forcing; int8 / int4 weight
decoding bit exact.  The CUDA path computes in fp32 (fp64 in the oracle);
its expected error is ~1e-5 on logits of spread ~1, so the bar leaves
room for fp32 summation order only, not for a wrong term.
"""
import gc

import numpy as np
import pytest
import torch

from workload import configs as wc
from workload import synth

pytestmark = pytest.mark.gpu

TOL = 5e-2


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="module")
def amk(dev):
    from decode_megakernel_gb300 import amk as m
    return m


@pytest.fixture(scope="module")
def orc():
    from oracle import binding
    return binding


def bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().astype(np.int32) & 0xFFFF


def kv_close(a, b):
    """bf16 K,V written by the GPU (rounded from fp32) against the oracle's
    (rounded from fp64): within two bf16 steps of the value, or, for
    entries near zero, within 1e-4 of the largest magnitude (fp32 vs fp64
    drift of the residual stream moves small entries by an absolute, not
    relative, amount).  Returns (all close, fraction bit-identical,
    worst |difference| / allowance)."""
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    allow = 2.0 ** -7 * np.abs(y) + 1e-4 * np.abs(y).max()
    ratio = float((np.abs(x - y) / allow).max())
    return ratio <= 1.0, float((bits(a) == bits(b)).mean()), ratio


def run_teacher_forced(amk, orc, dev, cfg, prompt_len, steps, sched=None, max_seq=None):
    max_seq = max_seq or prompt_len + steps
    w = synth.model_weights(cfg, seed=0, device=dev)
    dec = amk.Decoder(w, max_seq, sched=sched)
    om = orc.OracleModel(w.to("cpu"), max_seq)
    kv_o = synth.empty_kv_cache(cfg, max_seq)
    prompt = synth.prompt_tokens(cfg, prompt_len).tolist()
    toks = synth.decode_tokens(cfg, steps).tolist()
    dec.prefill(prompt, 0)
    om.prefill(kv_o, prompt, 0)
    dec.sync()
    ul = kv_close(dec.kv[:, :, :, :prompt_len], kv_o[:, :, :, :prompt_len])
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    errs, agree = [], 0
    for i, tok in enumerate(toks):
        pos = prompt_len + i
        dec.decode_step(tok, pos, logits)
        ref = om.decode_step(kv_o, tok, pos)
        got = logits.double().cpu().numpy()
        errs.append(float(np.abs(got - ref).max()))
        agree += int(np.argmax(got) == np.argmax(ref))
    dec.sync()
    dec.close()
    return max(errs), agree / steps, ul


def test_tiny_teacher_forced(amk, orc, dev):
    err, agree, ul = run_teacher_forced(amk, orc, dev, wc.TINY, 16, 32)
    print(f"tiny: max|dlogit| {err:.3e}, top-1 {agree:.3f}, kv bit-identical {ul[1]:.4f}, "
          f"worst kv diff / allowance {ul[2]:.3f}")
    assert err <= TOL
    assert agree >= 0.99
    assert ul[0] and ul[1] > 0.99


@pytest.mark.parametrize("variant", ["tied", "mha", "hd128", "int8", "int8-lmbf16", "int4", "int4-lmbf16",
                                     "int8-longrow", "int4-longrow"])
def test_tiny_variants(amk, orc, dev, variant):
    base = dict(wc.TINY.__dict__)
    if variant == "tied":
        base.update(tied_embeddings=True)
    elif variant == "mha":
        base.update(n_kv_heads=4)
    elif variant == "hd128":
        base.update(n_heads=4, n_kv_heads=1, head_dim=128, hidden=512)
    elif variant.startswith("int8"):
        base.update(weight_format="int8", lm_head_bf16=variant.endswith("lmbf16"))
    else:
        base.update(weight_format="int4", ffn=768, lm_head_bf16=variant.endswith("lmbf16"))
    if variant.endswith("longrow"):
        # a down projection of 4 K tiles (in_features 8192): the int4 consumer
        # runs its rolled tile loop over rotated fragments there
        base.update(ffn=8192)
    cfg = wc.ModelConfig(**base)
    err, agree, ul = run_teacher_forced(amk, orc, dev, cfg, 9, 6)
    print(f"{variant}: max|dlogit| {err:.3e}, top-1 {agree:.3f}, kv same {ul[1]:.4f}, "
          f"kv worst/allow {ul[2]:.3f}")
    assert err <= TOL and agree >= 0.99
    # the prompt's K,V: bf16 variants run the tensor-core prefill, whose
    # activations enter its GEMMs as two bf16 parts (2^-18 relative): every
    # entry within two bf16 steps, and rounding flips inherited through the
    # layers leave >= 98% bit-identical; the others prefill by decode steps
    assert ul[0] and ul[1] > (0.98 if cfg.weight_format == "bf16" else 0.99)


@pytest.mark.parametrize("knobs", [dict(num_ctas=37, attn_splits=5, max_rows_per_task=32),
                                   dict(num_ctas=8, attn_splits=1),
                                   dict(num_ctas=152, attn_splits=64)])
def test_schedule_knobs(amk, orc, dev, knobs):
    sched = amk.make_schedule_config(**knobs)
    err, agree, _ = run_teacher_forced(amk, orc, dev, wc.TINY, 20, 4, sched=sched)
    assert err <= TOL and agree >= 0.99


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
@pytest.mark.parametrize("ring_slots", [0, 1, 4, 8])
def test_ring_split_long_context(amk, orc, dev, fmt, ring_slots):
    # one context split per KV head holding 600 positions: three attention
    # chunks of 256 (head_dim 64) between the weight tiles in the CTA's
    # ring, with 1, 4 or 8 copies in flight (0: the default, 6); the chunk
    # loop wraps around the ring's 12 slots
    base = dict(wc.TINY.__dict__)
    if fmt == "int4":
        base.update(weight_format="int4", ffn=768)
    cfg = wc.ModelConfig(**base)
    sched = amk.make_schedule_config(num_ctas=8, attn_splits=1, ring_slots=ring_slots, prefill_chunk=-1)
    err, agree, ul = run_teacher_forced(amk, orc, dev, cfg, 600, 4, sched=sched)
    print(f"{fmt} ring_slots {ring_slots}: max|dlogit| {err:.3e}, top-1 {agree:.3f}, kv same {ul[1]:.4f}")
    assert err <= TOL and agree >= 0.99
    assert ul[0] and ul[1] > 0.99


def test_tiny_greedy_loop(amk, orc, dev):
    cfg = wc.TINY
    steps, max_seq = 32, 48
    w = synth.model_weights(cfg, seed=3, device=dev)
    dec = amk.Decoder(w, max_seq)
    om = orc.OracleModel(w.to("cpu"), max_seq)
    kv_o = synth.empty_kv_cache(cfg, max_seq)
    prompt = synth.prompt_tokens(cfg, 16).tolist()
    dec.prefill(prompt, 0)
    om.prefill(kv_o, prompt, 0)
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    tg = to = prompt[-1]
    gpu_seq, orc_seq, near_tie = [], [], 0
    # both sides start from the last prompt token re-fed at the last position
    pos = len(prompt) - 1
    for i in range(steps):
        dec.decode_step(tg, pos + i, logits)
        ref = om.decode_step(kv_o, to, pos + i)
        tg = int(torch.argmax(logits).item())
        srt = np.sort(ref)
        near_tie += int(srt[-1] - srt[-2] < 1e-3)
        to = int(np.argmax(ref))
        gpu_seq.append(tg)
        orc_seq.append(to)
        if tg != to:
            break
    dec.close()
    assert gpu_seq == orc_seq or near_tie > 0, (gpu_seq, orc_seq)


@pytest.mark.parametrize("knobs,steps", [(dict(), 24), (dict(num_ctas=8), 12), (dict(), 1)])
def test_device_greedy_matches_host_loop(amk, dev, knobs, steps):
    """amk_generate (argmax fused into the LM head, the token never leaves
    the GPU) produces exactly the tokens and final logits of a host loop of
    amk_decode_step + torch.argmax (first index on ties, as the device)."""
    cfg = wc.TINY
    max_seq = 16 + steps
    w = synth.model_weights(cfg, seed=5, device=dev)
    sched = amk.make_schedule_config(**knobs)
    prompt = synth.prompt_tokens(cfg, 16).tolist()
    a = amk.Decoder(w, max_seq, sched=sched)
    b = amk.Decoder(w, max_seq, sched=sched)
    for d in (a, b):
        d.prefill(prompt[:-1], 0)
    pos = len(prompt) - 1
    toks = torch.full((steps,), -7, dtype=torch.int32, device=dev)
    la = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    a.generate(prompt[-1], pos, steps, toks, la)
    a.sync()
    assert amk.amk_kv_length(a.ctx) == pos + steps
    lb = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    t, host = prompt[-1], []
    for i in range(steps):
        b.decode_step(t, pos + i, lb)
        t = int(torch.argmax(lb).item())
        host.append(t)
    b.sync()
    assert toks.cpu().tolist() == host
    assert torch.equal(la, lb)
    assert torch.equal(a.kv, b.kv)
    a.close()
    b.close()


def test_prefill_equals_decode_steps_and_rollback(amk, dev):
    """The decode-kernel prefill (prefill_chunk = -1) is the decode step
    with the LM head skipped: bit-identical K,V."""
    cfg = wc.TINY
    w = synth.model_weights(cfg, seed=4, device=dev)
    toks = synth.prompt_tokens(cfg, 12).tolist()
    a = amk.Decoder(w, 16, sched=amk.make_schedule_config(prefill_chunk=-1))
    assert a.prefill_chunk == 0
    a.prefill(toks, 0)
    a.sync()
    b = amk.Decoder(w, 16)
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    for p, t in enumerate(toks):
        b.decode_step(t, p, logits)
    b.sync()
    assert torch.equal(a.kv, b.kv)
    # rolling back to position 5 and re-running reproduces the same logits
    b.decode_step(toks[5], 5, logits)
    first = logits.clone()
    b.decode_step(toks[5], 5, logits)
    assert torch.equal(first, logits)
    with pytest.raises(amk.AmkError) as e:
        b.decode_step(toks[7], 9, logits)   # valid length is now 6
    assert e.value.status == amk.AMK_ERR_INVALID_ARG
    with pytest.raises(amk.AmkError):
        b.decode_step(cfg.vocab, 6, logits)
    a.close()
    b.close()


def kv_layers(a, b):
    """Per-layer view of two K,V caches [L, 2, n_kv, P, hd]: layer 0 strict
    (kv_close), every layer's bit-identical share, and the mean |difference|
    relative to the mean |value| over all layers."""
    first = kv_close(a[:1], b[:1])
    same = [float((bits(a[l]) == bits(b[l])).mean()) for l in range(a.shape[0])]
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    rel_mean = float(np.abs(x - y).sum() / np.abs(y).sum())
    return first, same, rel_mean


@pytest.mark.parametrize("variant,chunk,prompt,split,parts,rows", [
    ("tiny", 0, 12, None, 0, 0),       # one chunk, one partial 128-token tile (default: two parts)
    ("tiny", 128, 300, 100, 0, 0),     # two calls (history from the first), three chunks, ragged tail
    ("hd128", 128, 200, None, 0, 0),   # head_dim 128, group 4
    ("mha", 0, 40, 17, 0, 0),          # group 1
    ("tied", 256, 260, None, 0, 0),
    ("tiny", 128, 300, 100, 3, 0),     # three activation parts
    ("hd128", 0, 200, None, 3, 0),
    ("tiny", 128, 300, 100, 0, 256),   # 256-row GEMM tiles for every matrix
    ("hd128", 0, 200, None, 3, 256),
    ("tiny", 0, 140, None, 0, 224),    # 224-row tiles: partial last tile of 256-row matrices
    ("mha", 0, 200, 70, 0, 0),         # group 1 on the tensor-core attention (128 tokens per CTA)
])
def test_tensor_core_prefill_matches_oracle(amk, orc, dev, variant, chunk, prompt, split, parts, rows):
    """The tensor-core prefill (tcgen05 GEMMs; tcgen05 attention once the
    cache holds 64 positions, mma.sync attention before) against
    the oracle's batched causal prefill (orc_prefill_batched, itself pinned
    equal to sequential decode steps), then decode steps on top of it.

    Layer 0's K,V come straight from the embedding, RMSNorm, the QKV GEMM
    and RoPE: within two bf16 steps of the oracle and >= 99.5% bit-identical
    with the default two activation parts (2^-18), >= 99.9% with three
    (2^-27).
    Deeper layers inherit every bf16 rounding of the layers below: a V entry
    that rounds the other way moves the next layer's input by a bf16 step
    of that value (divided by the tokens attending to it), so the shares of
    identical entries drop by a few percent per layer for any fp32
    implementation (the decode kernel run with two CTA counts differs the
    same way); those layers are held to >= 90% identical and a mean
    |difference| <= 1e-3 of the mean |value|.  The contract itself: the
    logits of the decode steps that follow within 5e-2, same top-1."""
    base = dict(wc.TINY.__dict__)
    if variant == "hd128":
        base.update(n_heads=4, n_kv_heads=1, head_dim=128, hidden=512)
    elif variant == "mha":
        base.update(n_kv_heads=4)
    elif variant == "tied":
        base.update(tied_embeddings=True)
    cfg = wc.ModelConfig(**base)
    steps = 4
    max_seq = prompt + steps
    w = synth.model_weights(cfg, seed=6, device=dev)
    dec = amk.Decoder(w, max_seq, sched=amk.make_schedule_config(prefill_chunk=chunk, prefill_parts=parts,
                                                                  prefill_tile_rows=rows))
    om = orc.OracleModel(w.to("cpu"), max_seq)
    kv_o = synth.empty_kv_cache(cfg, max_seq)
    toks = synth.prompt_tokens(cfg, prompt).tolist()
    want = min(((chunk or 2048) + 127) // 128 * 128, (max_seq + 127) // 128 * 128)
    assert dec.prefill_chunk == want   # the tensor-core path is the one that runs
    if split:
        dec.prefill(toks[:split], 0)
        dec.prefill(toks[split:], split)
    else:
        dec.prefill(toks, 0)
    assert amk.amk_kv_length(dec.ctx) == prompt
    om.prefill_batched(kv_o, toks, 0)
    dec.sync()
    (ok0, same0, worst0), same, rel_mean = kv_layers(dec.kv[:, :, :, :prompt], kv_o[:, :, :, :prompt])
    print(f"{variant} chunk {chunk} P {prompt} parts {parts or 2} tile rows {rows or 'auto'}: "
          f"layer 0 identical {same0:.4f} "
          f"worst/allow {worst0:.3f}; per layer {' '.join(f'{x:.4f}' for x in same)}; "
          f"mean |diff| / mean |kv| {rel_mean:.2e}")
    assert ok0 and same0 >= (0.999 if parts == 3 else 0.995)
    assert min(same) >= 0.90 and rel_mean <= 1e-3
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    for i, tok in enumerate(synth.decode_tokens(cfg, steps).tolist()):
        dec.decode_step(tok, prompt + i, logits)
        ref = om.decode_step(kv_o, tok, prompt + i)
        got = logits.double().cpu().numpy()
        assert float(np.abs(got - ref).max()) <= TOL
        assert int(np.argmax(got)) == int(np.argmax(ref))
    dec.close()


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_dequant_bit_exact(amk, orc, dev, fmt):
    out_f, in_f = 67, 512
    wb = synth.gaussian_bf16((out_f, in_f), 0.02, 17, "dq", "cpu")
    lin = synth.make_linear(fmt, wb)
    # make every code value appear
    if fmt == "int8":
        lin.w[0, :255] = torch.arange(-127, 128, dtype=torch.int16).to(torch.int8)
    else:
        lin.w[0, :8] = torch.tensor([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], dtype=torch.uint8)
        lin.zeros[1, :] = 0xF0
    ref = orc.dequant(lin)
    g = lin.to(dev)
    out = torch.empty((out_f, in_f), dtype=torch.float32, device=dev)
    st = amk.amk_debug_dequant(amk.FORMAT_CODE[fmt], g.w.data_ptr(), g.scales.data_ptr(),
                               g.zeros.data_ptr() if g.zeros is not None else 0, out_f, in_f,
                               out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == amk.AMK_OK
    assert np.array_equal(out.double().cpu().numpy(), ref)


def test_watchdog_reports_timeout_without_hanging(amk, dev):
    scratch = torch.zeros(64, dtype=torch.int32, device=dev)
    st, dstat = amk.amk_debug_watchdog_probe(scratch.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream, 2000)
    assert st == amk.AMK_OK
    assert dstat == amk.AMK_ERR_TIMEOUT
    # the context is still usable afterwards
    torch.cuda.synchronize()
    x = torch.ones(8, device=dev)
    assert float(x.sum()) == 8.0


# ---------------------------------------------------------------- full size

# (workload, KV history length, teacher-forced decode steps)
FULL = [("llama1b", 512, 128), ("llama8b-bf16", 2048, 32), ("llama8b-int8", 2048, 16),
        ("llama8b-int4", 16384, 8)]


@pytest.mark.slow
@pytest.mark.parametrize("name,prompt_len,steps", FULL)
def test_full_size_teacher_forced(amk, orc, dev, name, prompt_len, steps):
    """Full-size model in the launch configuration the benchmark times (one
    CTA per SM), teacher-forced: the KV history [0, P) is a seeded synthetic
    input given to both sides, then `steps` decode steps at P, P+1, ... on
    the seeded token stream are compared on every logit (max |dlogit| <=
    5e-2 at every step, top-1 agreement >= 99%), and the K,V rows the steps
    append are compared layer by layer with the oracle's."""
    wl = wc.workload(name)
    cfg = wl.model
    max_seq = prompt_len + steps
    w = synth.model_weights(cfg, seed=0, device=dev)
    kv = synth.synthetic_kv_cache(cfg, prompt_len, max_seq, device=dev)
    kv_o = kv.cpu()
    om = orc.OracleModel(w.to("cpu"), max_seq)
    dec = amk.Decoder(w, max_seq, kv_cache=kv)
    del w
    gc.collect()
    dec.set_kv_length(prompt_len)
    logits = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    toks = synth.decode_tokens(cfg, steps).tolist()
    errs, agree = [], 0
    for i, tok in enumerate(toks):
        pos = prompt_len + i
        dec.decode_step(tok, pos, logits)
        ref = om.decode_step(kv_o, tok, pos)
        got = logits.double().cpu().numpy()
        errs.append(float(np.abs(got - ref).max()))
        agree += int(np.argmax(got) == np.argmax(ref))
    dec.sync()
    new = kv[:, :, :, prompt_len:max_seq]
    new_o = kv_o[:, :, :, prompt_len:max_seq]
    per_layer = [float((bits(new[l]) == bits(new_o[l])).mean()) for l in range(cfg.n_layers)]
    print(f"{name}: {steps} steps, max|dlogit| {max(errs):.3e} (mean {np.mean(errs):.3e}), "
          f"top-1 {agree / steps:.3f}; K,V bit-identical per layer "
          + " ".join(f"{x:.3f}" for x in per_layer))
    assert max(errs) <= TOL
    assert agree / steps >= 0.99
    # K,V the steps append agree with the oracle's within two bf16 steps
    # everywhere; at full depth the residual stream has drifted by ~1e-5
    # relative (fp32 and 28-bit hand-offs, attention sums on the tensor
    # cores), which flips the bf16 rounding of a few percent of the entries
    # of the deepest layers.
    ok, same, worst = kv_close(new, new_o)
    print(f"{name}: kv bit-identical {same:.4f}, worst diff / allowance {worst:.3f}")
    assert ok and same > 0.98
    dec.close()
    del dec, kv, kv_o, om
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("parts", [3, 2])
def test_full_size_tensor_core_prefill_matches_decode_steps(amk, dev, parts):
    """8B bf16 shape: the tensor-core prefill of 256 prompt tokens (chunks
    of 128: the second chunk attends to the first through the cache)
    against the decode-kernel prefill (one decode step per token, itself
    held to the oracle by the tests above).  Layer 0 within two bf16 steps
    and >= 99.9% identical; through 32 layers the bf16 K,V round trips
    amplify every rounding difference (the decode kernel against itself
    with 76 instead of 152 CTAs: 74% identical at the last layer), so the
    deep layers are held to a mean |difference| <= 3% of the mean |value|;
    the next decode step's logits within 5e-2, same top-1."""
    wl = wc.workload("llama8b-bf16")
    cfg = wl.model
    P, max_seq = 256, 264
    w = synth.model_weights(cfg, seed=0, device=dev)
    a = amk.Decoder(w, max_seq, sched=amk.make_schedule_config(prefill_chunk=128, prefill_parts=parts))
    b = amk.Decoder(w, max_seq, sched=amk.make_schedule_config(prefill_chunk=-1))
    del w
    gc.collect()
    toks = synth.prompt_tokens(cfg, P).tolist()
    a.prefill(toks, 0)
    b.prefill(toks, 0)
    a.sync()
    b.sync()
    (ok0, same0, worst0), same, rel_mean = kv_layers(a.kv[:, :, :, :P], b.kv[:, :, :, :P])
    print(f"8B prefill, {parts} parts: layer 0 identical {same0:.4f} worst/allow {worst0:.3f}; last layer "
          f"identical {same[-1]:.4f}; mean |diff| / mean |kv| {rel_mean:.2e}")
    assert ok0 and same0 >= (0.995 if parts == 2 else 0.999)
    assert rel_mean <= 0.03
    la = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    lb = torch.empty(cfg.vocab, dtype=torch.float32, device=dev)
    tok = int(synth.decode_tokens(cfg, 1)[0])
    a.decode_step(tok, P, la)
    b.decode_step(tok, P, lb)
    a.sync()
    b.sync()
    err = float((la - lb).abs().max())
    print(f"8B prefill: next-step max|dlogit| {err:.3e}")
    assert err <= TOL
    assert int(la.argmax()) == int(lb.argmax())
    a.close()
    b.close()
    del a, b
    gc.collect()
    torch.cuda.empty_cache()
