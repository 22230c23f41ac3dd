"""Model shapes, workloads and byte accounting for batch-1 Llama decode.

This module holds no arithmetic of the decode step itself: it names the
shapes of the five synthetic workloads and counts the bytes one decode step
must move.  Both the CUDA path and the oracle take their shapes from here.

The problem statement of AutoMegaKernel (AMK summaries, "Problem statement"):
single-stream batch-1 decode is bandwidth bound and its latency floor is
t_min = weight_bytes / HBM bandwidth.  ``step_bytes`` extends the numerator
with the KV-cache bytes a step must read, which is what a step at context
length ``pos + 1`` actually streams.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

FORMAT_BF16 = "bf16"
FORMAT_INT8 = "int8"      # symmetric per-output-row int8, fp16 scale per row
FORMAT_INT4 = "int4"      # asymmetric group-128 int4, fp16 scale + 4-bit zero per group
FORMATS = (FORMAT_BF16, FORMAT_INT8, FORMAT_INT4)
FORMAT_CODE = {FORMAT_BF16: 0, FORMAT_INT8: 1, FORMAT_INT4: 2}

INT4_GROUP = 128


@dataclass(frozen=True)
class ModelConfig:
    """Shape of a Llama-family decoder (HF Llama conventions)."""

    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    tied_embeddings: bool = False
    weight_format: str = FORMAT_BF16
    # the untied LM head follows the weight format unless this is set
    lm_head_bf16: bool = False

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def linear_shapes(self):
        """(name, out_features, in_features) of every per-layer linear map."""
        h, f = self.hidden, self.ffn
        return [
            ("wq", self.q_dim, h),
            ("wk", self.kv_dim, h),
            ("wv", self.kv_dim, h),
            ("wo", h, self.q_dim),
            ("wg", f, h),
            ("wu", f, h),
            ("wd", h, f),
        ]

    @property
    def lm_head_format(self) -> str:
        if self.tied_embeddings or self.lm_head_bf16:
            return FORMAT_BF16
        return self.weight_format


@dataclass(frozen=True)
class Workload:
    """A model plus the decode schedule one run exercises."""

    model: ModelConfig
    prompt_len: int
    decode_steps: int
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def name(self) -> str:
        return self.model.name

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.decode_steps

    def decode_positions(self):
        return list(range(self.prompt_len, self.prompt_len + self.decode_steps))


def matrix_bytes(fmt: str, rows: int, cols: int) -> int:
    """Bytes of one weight matrix in its stored format (codes + scales + zeros)."""
    if fmt == FORMAT_BF16:
        return rows * cols * 2
    if fmt == FORMAT_INT8:
        return rows * cols + rows * 2
    if fmt == FORMAT_INT4:
        assert cols % INT4_GROUP == 0, "int4 needs in_features % 128 == 0"
        groups = cols // INT4_GROUP
        return rows * cols // 2 + rows * groups * 2 + rows * ((groups + 1) // 2)
    raise ValueError(fmt)


def weight_bytes_per_token(m: ModelConfig) -> int:
    """Bytes of weights one decode step streams: all linear maps, the norm
    vectors, one embedding row and the LM head."""
    total = 0
    for _, out_f, in_f in m.linear_shapes():
        total += matrix_bytes(m.weight_format, out_f, in_f)
    total *= m.n_layers
    total += m.n_layers * 2 * m.hidden * 2          # attn + ffn RMSNorm weights (bf16)
    total += m.hidden * 2                           # final RMSNorm weight
    total += m.hidden * 2                           # one embedding row (bf16)
    total += matrix_bytes(m.lm_head_format, m.vocab, m.hidden)
    return total


def kv_bytes_per_position(m: ModelConfig) -> int:
    """bf16 K and V of one position over all layers."""
    return m.n_layers * 2 * m.n_kv_heads * m.head_dim * 2


def kv_read_bytes(m: ModelConfig, pos: int) -> int:
    """KV bytes a step at position ``pos`` reads (context = pos + 1)."""
    return (pos + 1) * kv_bytes_per_position(m)


def step_bytes(m: ModelConfig, pos: int) -> int:
    """Algorithmic bytes of one decode step at ``pos``: weights + KV read."""
    return weight_bytes_per_token(m) + kv_read_bytes(m, pos)


def step_flops(m: ModelConfig, pos: int) -> int:
    """2 flops per weight multiply-add plus the attention score/value work."""
    lin = sum(o * i for _, o, i in m.linear_shapes()) * m.n_layers + m.vocab * m.hidden
    attn = 4 * (pos + 1) * m.n_heads * m.head_dim * m.n_layers
    return 2 * lin + attn


def prefill_flops(m: ModelConfig, n: int, start: int = 0) -> int:
    """Algorithmic flops of a prefill of n tokens at positions start..: the
    QKV products of every layer; causal attention (scores and values, 2
    flops per multiply-add) and the O / gate-up / down products of every
    layer but the last (their output feeds no K,V)."""
    shapes = {name: o * i for name, o, i in m.linear_shapes()}
    qkv = shapes["wq"] + shapes["wk"] + shapes["wv"]
    rest = shapes["wo"] + shapes["wg"] + shapes["wu"] + shapes["wd"]
    lin = qkv * m.n_layers + rest * (m.n_layers - 1)
    ctx = sum(start + t + 1 for t in range(n))   # positions each token attends to
    attn = 4 * ctx * m.n_heads * m.head_dim * (m.n_layers - 1)
    return 2 * lin * n + attn


def _llama8b(fmt: str, name: str, **kw) -> ModelConfig:
    return ModelConfig(
        name=name, n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128,
        ffn=14336, vocab=128256, rms_eps=1e-5, rope_theta=500000.0,
        tied_embeddings=False, weight_format=fmt, **kw)


TINY = ModelConfig(
    name="tiny", n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
    ffn=688, vocab=1024, rms_eps=1e-5, rope_theta=10000.0, tied_embeddings=False)

LLAMA_1B = ModelConfig(
    name="llama3.2-1b", n_layers=16, hidden=2048, n_heads=32, n_kv_heads=8, head_dim=64,
    ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=500000.0, tied_embeddings=True)

LLAMA_8B_BF16 = _llama8b(FORMAT_BF16, "llama3.1-8b-bf16")
LLAMA_8B_INT8 = _llama8b(FORMAT_INT8, "llama3.1-8b-int8")
LLAMA_8B_INT4 = _llama8b(FORMAT_INT4, "llama3.1-8b-int4")

WORKLOADS = {
    "tiny": Workload(TINY, prompt_len=16, decode_steps=32,
                     description="2L H256 4/2 heads hd64 F688 V1024, untied; 16 prompt + 32 decode"),
    "llama1b": Workload(LLAMA_1B, prompt_len=512, decode_steps=128,
                        description="Llama-3.2-1B shape, tied; KV 512 + 128 decode"),
    "llama8b-bf16": Workload(LLAMA_8B_BF16, prompt_len=2048, decode_steps=128,
                             description="Llama-3.1-8B shape bf16; KV 2048 + 128 decode"),
    "llama8b-int8": Workload(LLAMA_8B_INT8, prompt_len=2048, decode_steps=128,
                             description="8B shape, int8 per-row weights; KV 2048 + 128 decode"),
    "llama8b-int4": Workload(LLAMA_8B_INT4, prompt_len=16384, decode_steps=64,
                             description="8B shape, int4 g128 weights; KV 16384 + 64 decode"),
}


# Profiling cases: the per-layer shapes of the 8B workloads with only four
# layers (about 1 GB on the device with the 16K-position history), so that
# a many-pass counter capture of one decode launch stays small.  Not bench
# lines; the decode kernel runs them with the same tiles and schedule rules.
PROFILE_WORKLOADS = {
    "llama8b-int4-4l": Workload(replace(LLAMA_8B_INT4, name="llama8b-int4-4l", n_layers=4),
                                prompt_len=16384, decode_steps=64,
                                description="4 layers of the 8B int4 shape; KV 16384 + 64 decode"),
    "llama8b-int8-4l": Workload(replace(LLAMA_8B_INT8, name="llama8b-int8-4l", n_layers=4),
                                prompt_len=2048, decode_steps=128,
                                description="4 layers of the 8B int8 shape; KV 2048 + 128 decode"),
    "llama8b-bf16-4l": Workload(replace(LLAMA_8B_BF16, name="llama8b-bf16-4l", n_layers=4),
                                prompt_len=2048, decode_steps=128,
                                description="4 layers of the 8B bf16 shape; KV 2048 + 128 decode"),
}


def workload(name: str) -> Workload:
    if name in PROFILE_WORKLOADS:
        return PROFILE_WORKLOADS[name]
    return WORKLOADS[name]


def mean_step_bytes(w: Workload) -> float:
    pos = w.decode_positions()
    return sum(step_bytes(w.model, p) for p in pos) / len(pos)


def with_format(m: ModelConfig, fmt: str, **kw) -> ModelConfig:
    return replace(m, weight_format=fmt, name=f"{m.name}-{fmt}", **kw)
