"""Pins of the CPU oracle to things other than itself.

Every oracle function is checked against closed forms, invariants, special
cases that reduce to a library routine (numpy / scipy / torch float64), or
brute force on tiny inputs, so that a dropped term, a wrong sign or index or
a transposed operand fails at least one test.  The decode step definition
these follow is the HF Llama-family decoder named by the AutoMegaKernel
summaries ("Methodology") with the Layer-1 instruction set (GEMV,
attention, RMSNorm) and Argus' megakernel contents (KV-cache update, logits).
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from workload import configs as wc
from workload import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().astype(np.uint16)


# --------------------------------------------------------------- numbers

def test_bf16_to_double_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_fp16_to_double_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_rounding_golden(oracle):
    n = 0
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            x, want = line.split()
            v = float("inf") if x == "inf" else float("-inf") if x == "-inf" else float.fromhex(x)
            got = oracle.bf16_from_double(v)
            assert got == int(want, 16), (x, hex(got), want)
            n += 1
    assert n >= 20


def test_bf16_rounding_matches_library_on_binary32_inputs(oracle):
    # for inputs exactly representable in binary32 direct rounding equals
    # torch's binary32 -> bf16 conversion (round to nearest even)
    g = torch.Generator().manual_seed(7)
    f = torch.randn(4000, generator=g) * torch.exp(torch.randn(4000, generator=g) * 20)
    ref = bf16_bits(f.to(torch.bfloat16))
    got = np.array([oracle.bf16_from_double(float(v)) for v in f.double()], dtype=np.uint16)
    assert (got == ref).all()
    assert oracle.bf16_from_double(float("nan")) & 0x7F80 == 0x7F80


# --------------------------------------------------------------- weights

def _linear_from(fmt, codes, scales=None, zeros=None, out_f=None, in_f=None):
    return synth.Linear(fmt, out_f, in_f, codes, scales, zeros)


def test_dequant_int8_exhaustive_codes(oracle):
    codes = torch.arange(-128, 128, dtype=torch.int16).to(torch.int8)
    scale_bits = [0x3C00, 0x1400, 0x0001, 0x03FF, 0x7BFF, 0xBC00]  # 1, 2^-10ish, subnormals, max, -1
    q = codes.repeat(len(scale_bits), 1).contiguous()
    s = torch.tensor(scale_bits, dtype=torch.int32).to(torch.int16).view(torch.float16)
    lin = _linear_from("int8", q, s.contiguous(), None, len(scale_bits), 256)
    got = oracle.dequant(lin)
    ref = q.numpy().astype(np.float64) * s.numpy().astype(np.float64)[:, None]
    assert np.array_equal(got, ref)


def test_dequant_int4_exhaustive_codes_and_nibble_order(oracle):
    # in_features 256 = 2 groups; every (code, zero) pair appears
    rows = 16
    qv = np.zeros((rows, 256), dtype=np.uint8)
    for r in range(rows):
        qv[r, :] = np.arange(256) % 16
    zv = np.zeros((rows, 2), dtype=np.uint8)
    zv[:, 0] = np.arange(rows) % 16
    zv[:, 1] = (15 - np.arange(rows)) % 16
    packed = (qv[:, 0::2] | (qv[:, 1::2] << 4)).astype(np.uint8)
    zpacked = (zv[:, 0] | (zv[:, 1] << 4)).astype(np.uint8)[:, None]
    s = np.array([[0.5, -0.25]] * rows, dtype=np.float16)
    lin = _linear_from("int4", torch.from_numpy(packed), torch.from_numpy(s),
                       torch.from_numpy(zpacked.copy()), rows, 256)
    got = oracle.dequant(lin)
    z_full = np.repeat(zv, 128, axis=1).astype(np.float64)
    s_full = np.repeat(s.astype(np.float64), 128, axis=1)
    ref = (qv.astype(np.float64) - z_full) * s_full
    assert np.array_equal(got, ref)
    # a hand-built byte: 0x21 holds k=0 -> 1 (low nibble), k=1 -> 2 (high nibble)
    one = np.zeros((1, 128), dtype=np.uint8)
    one[0, 0] = 0x21
    lin1 = _linear_from("int4", torch.from_numpy(one), torch.ones(1, 2, dtype=torch.float16),
                        torch.tensor([[0x53]], dtype=torch.uint8), 1, 256)
    d = oracle.dequant(lin1)[0]
    assert d[0] == 1 - 3 and d[1] == 2 - 3 and d[2] == -3 and d[128] == -5


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_quantiser_roundtrip_through_oracle_dequant(oracle, fmt):
    w = synth.gaussian_bf16((24, 512), 0.02, 11, "rt", "cpu")
    lin = synth.make_linear(fmt, w)
    deq = oracle.dequant(lin)
    wf = w.double().numpy()
    if fmt == "int8":
        s = lin.scales.double().numpy()[:, None]
    else:
        s = np.repeat(lin.scales.double().numpy(), 128, axis=1)
    # unclipped codes reconstruct within half a quantisation step
    err = np.abs(deq - wf)
    assert (err <= s / 2 * (1 + 1e-3) + 1e-12).mean() > 0.999
    # dequantised values are exact in binary32 (<= 18 significant bits)
    assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)


@pytest.mark.parametrize("fmt", ["int8", "int4"])
def test_quantise_of_dequantised_codes_is_identity(oracle, fmt):
    """With power-of-two scales and codes that reach both ends of their range
    the dequantised matrix is exact in bf16; quantising it again must give the
    same codes, scales and zeros back, and the oracle must dequantise both
    to the same values."""
    rng = np.random.default_rng(9)
    rows, cols = 8, 256
    if fmt == "int8":
        q = rng.integers(-127, 128, size=(rows, cols))
        q[:, 0] = 127
        s = 2.0 ** rng.integers(-12, -4, size=rows)
        w = q * s[:, None]
    else:
        q = rng.integers(0, 16, size=(rows, cols))
        q[:, 0::128] = 0
        q[:, 1::128] = 15
        z = rng.integers(0, 16, size=(rows, cols // 128))
        s = 2.0 ** rng.integers(-12, -4, size=(rows, cols // 128))
        w = (q - np.repeat(z, 128, 1)) * np.repeat(s, 128, 1)
    wb = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(wb.double().numpy(), w)
    lin = synth.make_linear(fmt, wb)
    if fmt == "int8":
        assert np.array_equal(lin.w.numpy(), q)
        assert np.array_equal(lin.scales.double().numpy(), s)
    else:
        assert np.array_equal(lin.w.numpy(), (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))
        assert np.array_equal(lin.scales.double().numpy(), s)
        zz = z.astype(np.uint8)
        assert np.array_equal(lin.zeros.numpy()[:, 0], zz[:, 0] | (zz[:, 1] << 4))
    np.testing.assert_array_equal(oracle.dequant(lin), w)


@pytest.mark.parametrize("fmt", ["bf16", "int8", "int4"])
def test_linear_matches_library_matmul(oracle, fmt):
    out_f, in_f = 37, 384
    w = synth.gaussian_bf16((out_f, in_f), 0.02, 5, "lin", "cpu")
    lin = synth.make_linear(fmt, w)
    x = np.random.default_rng(3).standard_normal(in_f)
    ref = oracle.dequant(lin) @ x
    got = oracle.linear(lin, x)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_linear_integer_brute_force(oracle):
    # small integers are exact in bf16 and their dot products exact in double
    rng = np.random.default_rng(1)
    W = rng.integers(-8, 9, size=(5, 16))
    x = rng.integers(-5, 6, size=16)
    w = torch.from_numpy(W.astype(np.float32)).to(torch.bfloat16)
    lin = synth.make_linear("bf16", w)
    got = oracle.linear(lin, x.astype(np.float64))
    want = [sum(int(W[o, k]) * int(x[k]) for k in range(16)) for o in range(5)]
    assert got.tolist() == [float(v) for v in want]


# --------------------------------------------------------------- rmsnorm

def test_rmsnorm_unit_rms_and_weight(oracle):
    rng = np.random.default_rng(0)
    x = rng.standard_normal(4096) * 3.0
    eps = 1e-5
    out = oracle.rmsnorm(x, None, eps)
    ms = np.mean(x * x)
    assert math.isclose(np.sqrt(np.mean(out * out)), math.sqrt(ms / (ms + eps)), rel_tol=1e-12)
    # scale invariance (eps = 0) and elementwise weight
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, None, 0.0), oracle.rmsnorm(x, None, 0.0),
                               rtol=1e-13)
    w = synth.gaussian_bf16((4096,), 1.0, 2, "normw", "cpu")
    np.testing.assert_allclose(oracle.rmsnorm(x, w, eps), out * w.double().numpy(), rtol=1e-14)
    ref = F.rms_norm(torch.from_numpy(x), (4096,), w.double(), eps).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, w, eps), ref, rtol=1e-12)


# ------------------------------------------------------------------ rope

@pytest.mark.parametrize("head_dim,theta", [(64, 10000.0), (128, 500000.0)])
def test_rope_closed_form_on_basis_vectors(oracle, head_dim, theta):
    half = head_dim // 2
    pos = 37
    for i in (0, 1, half // 2, half - 1):
        ang = pos * theta ** (-2.0 * i / head_dim)
        e = np.zeros(head_dim)
        e[i] = 1.0
        r = oracle.rope(e, 1, head_dim, pos, theta)
        assert math.isclose(r[i], math.cos(ang), abs_tol=1e-12)
        assert math.isclose(r[i + half], math.sin(ang), abs_tol=1e-12)
        assert np.count_nonzero(np.abs(r) > 1e-15) <= 2
        e2 = np.zeros(head_dim)
        e2[i + half] = 1.0
        r2 = oracle.rope(e2, 1, head_dim, pos, theta)
        assert math.isclose(r2[i], -math.sin(ang), abs_tol=1e-12)
        assert math.isclose(r2[i + half], math.cos(ang), abs_tol=1e-12)


def test_rope_invariants(oracle):
    rng = np.random.default_rng(4)
    hd, nh, theta = 128, 3, 500000.0
    v = rng.standard_normal(nh * hd)
    # position 0 is the identity
    np.testing.assert_array_equal(oracle.rope(v, nh, hd, 0, theta), v)
    # each rotation pair keeps its norm
    r = oracle.rope(v, nh, hd, 12345, theta).reshape(nh, hd)
    vv = v.reshape(nh, hd)
    pn = lambda a: a[:, :hd // 2] ** 2 + a[:, hd // 2:] ** 2  # noqa: E731
    np.testing.assert_allclose(pn(r), pn(vv), rtol=1e-11)
    # heads are rotated independently and identically
    single = oracle.rope(v[:hd], 1, hd, 12345, theta)
    np.testing.assert_array_equal(single, r[0])
    # q(m).k(n) depends only on m - n
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    d1 = np.dot(oracle.rope(q, 1, hd, 100, theta), oracle.rope(k, 1, hd, 60, theta))
    d2 = np.dot(oracle.rope(q, 1, hd, 1040, theta), oracle.rope(k, 1, hd, 1000, theta))
    assert math.isclose(d1, d2, rel_tol=1e-9)


# ------------------------------------------------------------------ silu

def test_silu_matches_library(oracle):
    zs = np.linspace(-40, 40, 801)
    got = np.array([oracle.silu(float(z)) for z in zs])
    np.testing.assert_allclose(got, zs * scipy.special.expit(zs), rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0


# ------------------------------------------------------------- attention

def _kv(nkv, max_seq, hd, seed):
    k = synth.gaussian_bf16((nkv, max_seq, hd), 1.0, seed, "k", "cpu")
    v = synth.gaussian_bf16((nkv, max_seq, hd), 1.0, seed, "v", "cpu")
    return k, v


def test_attention_single_position_returns_v(oracle):
    nq, nkv, hd = 4, 2, 64
    k, v = _kv(nkv, 8, hd, 1)
    q = np.random.default_rng(1).standard_normal(nq * hd)
    o = oracle.attention(q, k, v, nq, nkv, hd, 1).reshape(nq, hd)
    for i in range(nq):
        np.testing.assert_array_equal(o[i], v[i // 2, 0].double().numpy())


def test_attention_equal_keys_mean_and_unit_sum(oracle):
    nq, nkv, hd, ctx = 2, 1, 64, 9
    k, v = _kv(nkv, 16, hd, 2)
    k[:, :ctx] = k[:, :1]
    q = np.random.default_rng(2).standard_normal(nq * hd)
    o = oracle.attention(q, k, v, nq, nkv, hd, ctx).reshape(nq, hd)
    mean_v = v[0, :ctx].double().mean(0).numpy()
    np.testing.assert_allclose(o[0], mean_v, rtol=1e-12, atol=1e-14)
    # probabilities sum to one: V of ones gives ones
    ones = torch.ones_like(v)
    o1 = oracle.attention(q, k, ones, nq, nkv, hd, ctx)
    np.testing.assert_allclose(o1, 1.0, rtol=1e-14)


@pytest.mark.parametrize("nq,nkv", [(4, 4), (8, 2), (4, 1)])
def test_attention_matches_library_sdpa(oracle, nq, nkv):
    hd, ctx, max_seq = 64, 23, 40
    k, v = _kv(nkv, max_seq, hd, 3)
    # positions at or beyond ctx must not matter
    k[:, ctx:] = 1e4
    q = np.random.default_rng(3).standard_normal(nq * hd)
    got = oracle.attention(q, k, v, nq, nkv, hd, ctx).reshape(nq, hd)
    qt = torch.from_numpy(q).view(1, nq, 1, hd)
    kt = k[:, :ctx].double().repeat_interleave(nq // nkv, 0).unsqueeze(0)
    vt = v[:, :ctx].double().repeat_interleave(nq // nkv, 0).unsqueeze(0)
    ref = F.scaled_dot_product_attention(qt, kt, vt)[0, :, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------- decoder

def _tiny_cfg(**kw):
    return wc.ModelConfig(**{**wc.TINY.__dict__, **kw})


def test_decoder_zero_layers_closed_form(oracle):
    """All layer weights zero: attention and FFN add nothing, so the logits
    are W_lm (rmsnorm(E[token]) * w_final)."""
    cfg = wc.TINY
    w = synth.model_weights(cfg, seed=5, zero_layers=True)
    w.final_norm = synth.gaussian_bf16((cfg.hidden,), 1.0, 9, "fn", "cpu")
    m = oracle.OracleModel(w, 8)
    kv = synth.empty_kv_cache(cfg, 8)
    tok = 321
    logits = m.decode_step(kv, tok, 0)
    e = w.embed[tok].double().numpy()
    h = e / np.sqrt(np.mean(e * e) + cfg.rms_eps) * w.final_norm.double().numpy()
    ref = w.lm_head.w.double().numpy() @ h
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-13)
    assert not kv.float().abs().sum().item()


def _restated_step(cfg, w, kv, token, pos):
    """The decoder written with torch float64 library routines (rms_norm,
    linear, silu, scaled_dot_product_attention), used only as a pin."""
    hd, nq, nkv = cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    deq = lambda lin: torch.from_numpy(oracle_dequant(lin))  # noqa: E731
    x = w.embed[token].double()
    half = hd // 2
    inv = torch.tensor([cfg.rope_theta ** (-2.0 * i / hd) for i in range(half)], dtype=torch.float64)
    ang = pos * inv
    cos = torch.cat([torch.cos(ang), torch.cos(ang)])
    sin = torch.cat([torch.sin(ang), torch.sin(ang)])

    def rope(t):
        t = t.view(-1, hd)
        rot = torch.cat([-t[:, half:], t[:, :half]], 1)
        return (t * cos + rot * sin).reshape(-1)

    for li, lw in enumerate(w.layers):
        h = F.rms_norm(x, (cfg.hidden,), lw["attn_norm"].double(), cfg.rms_eps)
        q = rope(F.linear(h, deq(lw["wq"])))
        k = rope(F.linear(h, deq(lw["wk"])))
        v = F.linear(h, deq(lw["wv"]))
        kv[li, 0, :, pos] = k.view(nkv, hd).float().to(torch.bfloat16)
        kv[li, 1, :, pos] = v.view(nkv, hd).float().to(torch.bfloat16)
        kt = kv[li, 0, :, :pos + 1].double().repeat_interleave(nq // nkv, 0).unsqueeze(0)
        vt = kv[li, 1, :, :pos + 1].double().repeat_interleave(nq // nkv, 0).unsqueeze(0)
        o = F.scaled_dot_product_attention(q.view(1, nq, 1, hd), kt, vt)[0, :, 0].reshape(-1)
        x = x + F.linear(o, deq(lw["wo"]))
        h = F.rms_norm(x, (cfg.hidden,), lw["ffn_norm"].double(), cfg.rms_eps)
        a = F.silu(F.linear(h, deq(lw["wg"]))) * F.linear(h, deq(lw["wu"]))
        x = x + F.linear(a, deq(lw["wd"]))
    h = F.rms_norm(x, (cfg.hidden,), w.final_norm.double(), cfg.rms_eps)
    return F.linear(h, deq(w.lm_head_linear())).numpy()


_ORC = None


def oracle_dequant(lin):
    return _ORC.dequant(lin)


@pytest.mark.parametrize("variant", ["untied-bf16", "tied-bf16", "int8", "int4"])
def test_decoder_matches_library_restatement(oracle, variant):
    global _ORC
    _ORC = oracle
    if variant == "untied-bf16":
        cfg = _tiny_cfg()
    elif variant == "tied-bf16":
        cfg = _tiny_cfg(tied_embeddings=True, n_kv_heads=4)
    elif variant == "int8":
        cfg = _tiny_cfg(weight_format="int8", n_kv_heads=1)
    else:
        cfg = _tiny_cfg(weight_format="int4", ffn=768)
    w = synth.model_weights(cfg, seed=1)
    # non-unit norm weights so that swapped norms are caught
    for li, lw in enumerate(w.layers):
        lw["attn_norm"] = synth.gaussian_bf16((cfg.hidden,), 0.3, 20 + li, "an", "cpu") + 1
        lw["ffn_norm"] = synth.gaussian_bf16((cfg.hidden,), 0.3, 40 + li, "fn", "cpu") + 1
    max_seq = 12
    m = oracle.OracleModel(w, max_seq)
    kv_o = synth.empty_kv_cache(cfg, max_seq)
    kv_r = synth.empty_kv_cache(cfg, max_seq)
    toks = synth.prompt_tokens(cfg, 9, seed=4).tolist()
    for pos, tok in enumerate(toks):
        lo = m.decode_step(kv_o, tok, pos)
        lr = _restated_step(cfg, w, kv_r, tok, pos)
        # the restatement rounds K,V through binary32 first; allow rare 1-ulp
        # bf16 differences and their small downstream effect
        np.testing.assert_allclose(lo, lr, rtol=0, atol=2e-3 * max(1.0, np.abs(lr).max()))
        close = np.abs(lo - lr) <= 1e-9 * np.abs(lr).max()
        assert close.mean() > 0.9
    a, b = bf16_bits(kv_o), bf16_bits(kv_r)
    ulp = np.abs(a.astype(np.int32) - b.astype(np.int32))
    assert ulp.max() <= 1 and (ulp == 0).mean() > 0.999


def test_decoder_thread_count_independent(oracle):
    cfg = wc.TINY
    w = synth.model_weights(cfg, seed=2)
    m = oracle.OracleModel(w, 6)
    outs = []
    for threads in (1, 3):
        oracle.set_threads(threads)
        kv = synth.empty_kv_cache(cfg, 6)
        for pos, tok in enumerate([5, 900, 17]):
            lg = m.decode_step(kv, tok, pos)
        outs.append((lg, bf16_bits(kv)))
    oracle.set_threads(os.cpu_count() or 1)
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])


def test_decoder_rejects_bad_arguments(oracle):
    cfg = wc.TINY
    w = synth.model_weights(cfg, seed=2)
    m = oracle.OracleModel(w, 4)
    kv = synth.empty_kv_cache(cfg, 4)
    with pytest.raises(ValueError):
        m.decode_step(kv, cfg.vocab, 0)
    with pytest.raises(ValueError):
        m.decode_step(kv, 0, 4)
    with pytest.raises(ValueError):
        m.decode_step(kv, -1, 0)


def test_prefill_equals_sequential_steps_and_leaves_tail(oracle):
    cfg = wc.TINY
    w = synth.model_weights(cfg, seed=6)
    m = oracle.OracleModel(w, 10)
    toks = [3, 4, 5, 6]
    kv1 = synth.empty_kv_cache(cfg, 10)
    m.prefill(kv1, toks)
    kv2 = synth.empty_kv_cache(cfg, 10)
    for p, t in enumerate(toks):
        m.decode_step(kv2, t, p, logits=False)
    assert np.array_equal(bf16_bits(kv1), bf16_bits(kv2))
    assert not kv1[:, :, :, len(toks):].float().abs().sum().item()


@pytest.mark.parametrize("variant", ["tiny", "int4", "mha"])
def test_batched_prefill_equals_sequential_decode(oracle, variant):
    """The batched causal prefill (a separate, layer-major loop nest) leaves
    the cache that token-by-token decode steps leave, bit for bit, also
    when it continues a history (start_pos > 0), and the decode step that
    follows sees the same logits."""
    base = dict(wc.TINY.__dict__)
    if variant == "int4":
        base.update(weight_format="int4", ffn=768)
    elif variant == "mha":
        base.update(n_kv_heads=4)
    cfg = wc.ModelConfig(**base)
    w = synth.model_weights(cfg, seed=9)
    m = oracle.OracleModel(w, 24)
    toks = synth.prompt_tokens(cfg, 20).tolist()
    seq = synth.empty_kv_cache(cfg, 24)
    for p, t in enumerate(toks):
        m.decode_step(seq, t, p, logits=False)
    bat = synth.empty_kv_cache(cfg, 24)
    m.prefill_batched(bat, toks[:7], 0)
    m.prefill_batched(bat, toks[7:], 7)
    assert np.array_equal(bf16_bits(seq), bf16_bits(bat))
    assert bat[:, :, :, :20].float().abs().sum().item() > 0
    assert not bat[:, :, :, 20:].float().abs().sum().item()
    a = m.decode_step(seq, 5, 20)
    b = m.decode_step(bat, 5, 20)
    assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        m.prefill_batched(bat, [cfg.vocab], 0)
    with pytest.raises(ValueError):
        m.prefill_batched(bat, [1, 2, 3, 4, 5], 20)   # beyond max_seq


def test_decode_step_is_layers_then_logits(oracle):
    """The sampled halves compose to the full step exactly (same arithmetic)."""
    for cfg in (wc.TINY, wc.ModelConfig(**{**wc.TINY.__dict__, "weight_format": "int4", "ffn": 768}),
                wc.ModelConfig(**{**wc.TINY.__dict__, "weight_format": "int8"})):
        w = synth.model_weights(cfg, seed=8)
        m = oracle.OracleModel(w, 6)
        kv1, kv2 = synth.empty_kv_cache(cfg, 6), synth.empty_kv_cache(cfg, 6)
        for pos, tok in enumerate([11, 500, 7]):
            full = m.decode_step(kv1, tok, pos)
            x = m.embed(tok)
            m.decode_layers(kv2, x, pos, 0, 1)
            m.decode_layers(kv2, x, pos, 1, cfg.n_layers)
            part = m.logits_rows(x, 0, 300)
            m.logits_rows(x, 300, cfg.vocab, part)
            assert np.array_equal(full, part)
        assert np.array_equal(bf16_bits(kv1), bf16_bits(kv2))
