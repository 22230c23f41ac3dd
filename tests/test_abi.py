"""The C ABI: the library loads, exports every declared entry point, and its
host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re

import pytest

from workload import configs as wc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def amk():
    from decode_megakernel_gb300 import build
    build.build()
    from decode_megakernel_gb300 import amk as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "amk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(amk_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(amk):
    names = declared_functions()
    assert len(names) >= 17
    lib = C.CDLL(amk.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(amk):
    for s in range(8):
        assert amk.status_string(s) and amk.status_string(s) != "unknown status"
    assert amk.status_string(99) == "unknown status"


def cfg_of(amk, **over):
    base = dict(wc.TINY.__dict__)
    base.update(over)
    return amk.make_config(wc.ModelConfig(**base), 64)


@pytest.mark.parametrize("over,expect", [
    ({}, 0),
    (dict(head_dim=96, hidden=384), 2),
    (dict(n_kv_heads=3), 2),
    (dict(n_heads=16, n_kv_heads=1), 2),     # group * head_dim = 1024 > 512
    (dict(weight_format="int4"), 2),         # ffn 688 is not a multiple of 128
    (dict(weight_format="int4", ffn=768), 0),
    (dict(weight_format="int8"), 0),
    (dict(ffn=30000), 2),                    # in_features beyond register-resident tiles
])
def test_check_config(amk, over, expect):
    assert amk.amk_check_config(cfg_of(amk, **over)) == expect


def test_check_config_invalid(amk):
    c = cfg_of(amk)
    c.n_layers = 0
    assert amk.amk_check_config(c) == amk.AMK_ERR_INVALID_ARG
    c = cfg_of(amk)
    c.weight_format = 7
    assert amk.amk_check_config(c) == amk.AMK_ERR_INVALID_ARG


def test_sizes(amk):
    c = amk.make_config(wc.LLAMA_8B_BF16, 2176)
    assert amk.amk_kv_cache_bytes(c) == 32 * 2 * 8 * 2176 * 128 * 2
    sc = amk.make_schedule_config(num_ctas=152)
    ws = amk.amk_workspace_bytes(c, sc)
    # the tiled weights dominate: at least the model's bytes
    assert ws >= wc.weight_bytes_per_token(wc.LLAMA_8B_BF16)
    assert ws < 1.1 * wc.weight_bytes_per_token(wc.LLAMA_8B_BF16) + c.vocab * c.hidden * 2
    bad = cfg_of(amk, head_dim=96, hidden=384)
    assert amk.amk_workspace_bytes(bad, sc) == 0


def test_prefill_chunk_sizes_the_workspace(amk):
    """bf16 weights get the tensor-core prefill's chunk buffers (x fp32,
    normed rows and attention / SwiGLU rows as three bf16 parts, rotated q
    fp32, the token ids); prefill_chunk = -1 and int8 / int4 weights do not."""
    c = amk.make_config(wc.LLAMA_8B_BF16, 2176)
    base = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152, prefill_chunk=-1))
    dflt = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152))
    m = wc.LLAMA_8B_BF16
    qd = m.n_heads * m.head_dim
    per_tok = m.hidden * 4 + 3 * m.hidden * 2 + 3 * max(qd, m.ffn) * 2 + qd * 4
    expect = 2048 * per_tok + 2176 * 4
    assert expect <= dflt - base <= expect + 10 * 256
    # a chunk is whole 128-token tiles, and no more than the cache holds
    c1 = amk.make_config(wc.LLAMA_8B_BF16, 200)
    small = amk.amk_workspace_bytes(c1, amk.make_schedule_config(num_ctas=152, prefill_chunk=-1))
    big = amk.amk_workspace_bytes(c1, amk.make_schedule_config(num_ctas=152, prefill_chunk=5000))
    assert 256 * per_tok <= big - small <= 256 * per_tok + 200 * 4 + 10 * 256
    c8 = amk.make_config(wc.LLAMA_8B_INT8, 2176)
    assert (amk.amk_workspace_bytes(c8, amk.make_schedule_config(num_ctas=152)) ==
            amk.amk_workspace_bytes(c8, amk.make_schedule_config(num_ctas=152, prefill_chunk=-1)))
    assert amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152, prefill_chunk=-2)) == 0
    # two or three bf16 parts per prefill activation (0: default); nothing else
    for parts, ok in [(0, True), (2, True), (3, True), (1, False), (4, False), (-1, False)]:
        ws = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152, prefill_parts=parts))
        assert (ws == dflt) if ok else (ws == 0)
    # prefill GEMM tiles of 256 or 224 weight rows (0: chosen per matrix); nothing else
    for rows, ok in [(0, True), (256, True), (224, True), (128, False), (192, False), (-1, False)]:
        ws = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152, prefill_tile_rows=rows))
        assert (ws == dflt) if ok else (ws == 0)


def test_host_argument_checks_need_no_gpu(amk):
    c = cfg_of(amk)
    st, ctx = amk.amk_load_weights(c, amk.amk_weights(), 0, 0, 0, 0)
    assert st == amk.AMK_ERR_INVALID_ARG and not ctx.value
    assert amk.lib.amk_decode_step(None, 0, 0, None) == amk.AMK_ERR_INVALID_ARG
    assert amk.lib.amk_prefill(None, None, 0, 0) == amk.AMK_ERR_INVALID_ARG
    assert amk.lib.amk_sync(None) == amk.AMK_ERR_INVALID_ARG
    assert amk.lib.amk_set_kv_length(None, 0) == amk.AMK_ERR_INVALID_ARG
    assert amk.lib.amk_kv_length(None) == -1
    amk.amk_free(None)
    st, _ = amk.amk_debug_watchdog_probe(0, 0, 100)
    assert st == amk.AMK_ERR_INVALID_ARG
    assert amk.amk_debug_dequant(9, 1, 1, 1, 4, 8, 1, 0) == amk.AMK_ERR_INVALID_ARG
    assert "NULL" in amk.last_error() or amk.last_error()


def test_validate_rejects_garbage(amk):
    st, rep = amk.amk_validate_serialized(b"\x00" * 80)
    assert st == amk.AMK_ERR_SCHEDULE_INVALID and "malformed" in rep
    st, rep = amk.amk_validate_serialized(b"\x01" * 7)
    assert st == amk.AMK_ERR_INVALID_ARG


def test_staging_bytes_is_the_largest_group(amk):
    """amk_weights_staging_bytes: the largest group of matrices packed
    together (QKV, O, gate + up, down, the untied LM head), every tensor of
    it (codes, fp16 scales, packed 4-bit zero points) rounded up to 256
    bytes; the tied LM head packs from the workspace's embedding copy."""
    def tensors(fmt, rows, cols):
        if fmt == "bf16":
            return [rows * cols * 2]
        if fmt == "int8":
            return [rows * cols, rows * 2]
        ng = cols // 128
        return [rows * cols // 2, rows * ng * 2, rows * ((ng + 1) // 2)]

    def group(fmt, shapes):
        return sum(-(-b // 256) * 256 for r, k in shapes for b in tensors(fmt, r, k))

    for m in (wc.LLAMA_8B_BF16, wc.LLAMA_1B, wc.LLAMA_8B_INT8, wc.LLAMA_8B_INT4):
        H, F, qd, kvd = m.hidden, m.ffn, m.q_dim, m.kv_dim
        f = m.weight_format
        want = max(group(f, [(qd, H), (kvd, H), (kvd, H)]), group(f, [(H, qd)]), group(f, [(F, H), (F, H)]),
                   group(f, [(H, F)]))
        if not m.tied_embeddings:
            want = max(want, group(m.lm_head_format, [(m.vocab, H)]))
        assert amk.amk_weights_staging_bytes(amk.make_config(m, 256)) == want, m.name
    bad = cfg_of(amk, head_dim=96, hidden=384)
    assert amk.amk_weights_staging_bytes(bad) == 0


def test_staged_load_checks_its_buffer(amk):
    """A NULL staging buffer is refused before anything touches a GPU."""
    c = cfg_of(amk)
    st, ctx = amk.amk_load_weights_staged(c, amk.amk_weights(), 256, 1 << 20, 256, 0,
                                          amk.make_schedule_config(num_ctas=4), 0, 0)
    assert st == amk.AMK_ERR_INVALID_ARG and not ctx.value


def test_ring_slots_knob(amk):
    """ring_slots caps the decode ring's copies in flight: 0 (the default),
    1..12 and larger values (acting as 12) are accepted and leave the
    workspace unchanged; a negative value is refused."""
    c = amk.make_config(wc.LLAMA_8B_BF16, 2176)
    dflt = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152))
    assert dflt > 0
    for rs, ok in [(0, True), (1, True), (6, True), (12, True), (20, True), (-1, False)]:
        ws = amk.amk_workspace_bytes(c, amk.make_schedule_config(num_ctas=152, ring_slots=rs))
        assert (ws == dflt) if ok else (ws == 0), rs
