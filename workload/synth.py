"""Seeded synthetic inputs for batch-1 Llama decode.

Everything a decode step consumes that is not computed by it comes from
here: weights, weight quantisation codes, prompt / decode tokens and, for the
full-size parity cases, a synthetic KV cache.  Both the CUDA path and the
oracle receive the very same tensors produced by these functions; neither
computes any of them.  Nothing in this module dequantises, normalises,
rotates or attends: that arithmetic belongs to the two implementations.

Recipe (random-weight stand-ins for the pages' SmolLM2/TinyLlama checkpoints,
which the AMK summaries use under "Experimental results"):
  * every linear weight and the embedding: N(0, 0.02^2), drawn in fp32 by a
    per-tensor seeded torch generator and rounded to bf16 (RNE);
  * RMSNorm weights: 1.0;
  * int8 (per output row, symmetric): s = fp16(max|w| / 127),
    q = clamp(rint(w / s), -127, 127);
  * int4 (group of 128 along in_features, asymmetric): s = fp16((max-min)/15),
    z = clamp(rint(-min / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15);
    two codes per byte (low nibble = even k), zeros two groups per byte
    (low nibble = even group);
  * tokens: uniform in [0, vocab);
  * synthetic KV (parity at full size): N(0, (0.02*sqrt(hidden))^2) in bf16,
    the spread of k = W_k * rmsnorm(x) under the weight recipe above.
"""
from __future__ import annotations

import math
import zlib

import torch

from .configs import FORMAT_BF16, FORMAT_INT4, FORMAT_INT8, INT4_GROUP, ModelConfig

WEIGHT_STD = 0.02
WEIGHT_SEED = 0
PROMPT_SEED = 1
DECODE_SEED = 2
KV_SEED = 3


def tensor_seed(seed: int, name: str) -> int:
    """Per-tensor seed: generating one tensor never depends on another."""
    return (seed * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF


def _generator(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(tensor_seed(seed, name))
    return g


def gaussian_bf16(shape, std: float, seed: int, name: str, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded once to bf16."""
    g = _generator(seed, name, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(torch.bfloat16)


def uniform_tokens(n: int, vocab: int, seed: int, name: str = "tokens") -> torch.Tensor:
    """``n`` token ids, uniform in [0, vocab), int32 on the host."""
    g = _generator(seed, name, "cpu")
    return torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32)


# --------------------------------------------------------------------------
# quantisation codes (inputs of the int8 / int4 workloads)
# --------------------------------------------------------------------------

def quantize_int8_rows(w: torch.Tensor):
    """Per-output-row symmetric int8 codes of a bf16 [out, in] matrix.

    Returns (codes int8 [out, in], scales fp16 [out])."""
    wf = w.float()
    amax = wf.abs().amax(dim=1)
    s16 = (amax / 127.0).to(torch.float16)
    sf = s16.float()
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    q = torch.round(wf / safe[:, None]).clamp_(-127, 127)
    q = torch.where(sf[:, None] > 0, q, torch.zeros_like(q))
    return q.to(torch.int8), s16


def quantize_int4_g128(w: torch.Tensor):
    """Asymmetric group-128 int4 codes of a bf16 [out, in] matrix.

    Returns (codes uint8 [out, in/2], scales fp16 [out, in/128],
    zeros uint8 [out, ceil(in/256)])."""
    out_f, in_f = w.shape
    if in_f % INT4_GROUP:
        raise ValueError("int4 group-128 needs in_features % 128 == 0")
    ng = in_f // INT4_GROUP
    wf = w.float().view(out_f, ng, INT4_GROUP)
    mn = wf.amin(-1)
    mx = wf.amax(-1)
    s16 = ((mx - mn) / 15.0).to(torch.float16)
    sf = s16.float()
    degenerate = sf == 0
    # a constant group: scale 1, zero point chosen so that q encodes the value
    s16 = torch.where(degenerate, torch.ones_like(s16), s16)
    sf = s16.float()
    z = torch.round(-mn / sf).clamp_(0, 15)
    q = (torch.round(wf / sf[..., None]) + z[..., None]).clamp_(0, 15)
    q = q.view(out_f, in_f).to(torch.uint8)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).contiguous()
    zq = z.to(torch.uint8)
    if ng % 2:
        zq = torch.cat([zq, torch.zeros(out_f, 1, dtype=torch.uint8, device=zq.device)], 1)
    zeros = (zq[:, 0::2] | (zq[:, 1::2] << 4)).contiguous()
    return codes, s16.contiguous(), zeros


class Linear:
    """One weight matrix in its stored format.

    bf16: ``w`` bf16 [out, in].  int8: ``w`` int8 [out, in] + ``scales``
    fp16 [out].  int4: ``w`` uint8 [out, in/2] + ``scales`` fp16
    [out, in/128] + ``zeros`` uint8 [out, ceil(in/256)]."""

    def __init__(self, fmt, out_features, in_features, w, scales=None, zeros=None):
        self.fmt = fmt
        self.out_features = out_features
        self.in_features = in_features
        self.w = w
        self.scales = scales
        self.zeros = zeros

    def tensors(self):
        return [t for t in (self.w, self.scales, self.zeros) if t is not None]

    def to(self, device):
        return Linear(self.fmt, self.out_features, self.in_features,
                      self.w.to(device),
                      None if self.scales is None else self.scales.to(device),
                      None if self.zeros is None else self.zeros.to(device))

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in self.tensors())


def make_linear(fmt: str, w_bf16: torch.Tensor) -> Linear:
    out_f, in_f = w_bf16.shape
    if fmt == FORMAT_BF16:
        return Linear(fmt, out_f, in_f, w_bf16.contiguous())
    if fmt == FORMAT_INT8:
        q, s = quantize_int8_rows(w_bf16)
        return Linear(fmt, out_f, in_f, q, s)
    if fmt == FORMAT_INT4:
        q, s, z = quantize_int4_g128(w_bf16)
        return Linear(fmt, out_f, in_f, q, s, z)
    raise ValueError(fmt)


class ModelWeights:
    """All weights of one synthetic model, in the HF layout."""

    def __init__(self, cfg: ModelConfig, embed, final_norm, lm_head, layers):
        self.cfg = cfg
        self.embed = embed              # bf16 [vocab, hidden]
        self.final_norm = final_norm    # bf16 [hidden]
        self.lm_head = lm_head          # Linear, or None when tied to ``embed``
        self.layers = layers            # list of dict: attn_norm, ffn_norm, wq..wd (Linear)

    def lm_head_linear(self) -> Linear:
        if self.lm_head is not None:
            return self.lm_head
        return Linear(FORMAT_BF16, self.cfg.vocab, self.cfg.hidden, self.embed)

    def to(self, device):
        layers = []
        for lw in self.layers:
            d = {}
            for k, v in lw.items():
                d[k] = v.to(device)
            layers.append(d)
        return ModelWeights(self.cfg, self.embed.to(device), self.final_norm.to(device),
                            None if self.lm_head is None else self.lm_head.to(device), layers)

    def nbytes(self):
        n = self.embed.numel() * 2 + self.final_norm.numel() * 2
        if self.lm_head is not None:
            n += self.lm_head.nbytes()
        for lw in self.layers:
            for k, v in lw.items():
                n += v.nbytes() if isinstance(v, Linear) else v.numel() * v.element_size()
        return n


def model_weights(cfg: ModelConfig, seed: int = WEIGHT_SEED, device="cpu",
                  zero_layers: bool = False) -> ModelWeights:
    """Seeded random weights of ``cfg``.

    ``zero_layers`` sets every per-layer linear weight to zero (norm weights
    stay 1): a degenerate model whose logits have a closed form."""
    h = cfg.hidden
    ones = torch.ones(h, dtype=torch.bfloat16, device=device)
    embed = gaussian_bf16((cfg.vocab, h), WEIGHT_STD, seed, "embed", device)
    layers = []
    for li in range(cfg.n_layers):
        lw = {"attn_norm": ones.clone(), "ffn_norm": ones.clone()}
        for name, out_f, in_f in cfg.linear_shapes():
            if zero_layers:
                w = torch.zeros((out_f, in_f), dtype=torch.bfloat16, device=device)
            else:
                w = gaussian_bf16((out_f, in_f), WEIGHT_STD, seed, f"layers.{li}.{name}", device)
            lw[name] = make_linear(cfg.weight_format, w)
            del w
        layers.append(lw)
    lm_head = None
    if not cfg.tied_embeddings:
        w = gaussian_bf16((cfg.vocab, h), WEIGHT_STD, seed, "lm_head", device)
        lm_head = make_linear(cfg.lm_head_format, w)
        del w
    return ModelWeights(cfg, embed, ones.clone(), lm_head, layers)


def kv_std(cfg: ModelConfig) -> float:
    return WEIGHT_STD * math.sqrt(cfg.hidden)


def kv_cache_shape(cfg: ModelConfig, max_seq: int):
    """KV cache layout: bf16 [n_layers][2 (K, V)][n_kv_heads][max_seq][head_dim]."""
    return (cfg.n_layers, 2, cfg.n_kv_heads, max_seq, cfg.head_dim)


def empty_kv_cache(cfg: ModelConfig, max_seq: int, device="cpu") -> torch.Tensor:
    return torch.zeros(kv_cache_shape(cfg, max_seq), dtype=torch.bfloat16, device=device)


def synthetic_kv_cache(cfg: ModelConfig, n_positions: int, max_seq: int,
                       seed: int = KV_SEED, device="cpu") -> torch.Tensor:
    """A KV cache whose positions [0, n_positions) hold seeded bf16 values.

    Stands in for a prefilled cache when the oracle cannot afford the
    prefill itself (full-size parity cases)."""
    kv = empty_kv_cache(cfg, max_seq, device)
    std = kv_std(cfg)
    for li in range(cfg.n_layers):
        blk = gaussian_bf16((2, cfg.n_kv_heads, n_positions, cfg.head_dim), std, seed,
                            f"kv.{li}", device)
        kv[li, :, :, :n_positions, :] = blk
        del blk
    return kv


def prompt_tokens(cfg: ModelConfig, n: int, seed: int = PROMPT_SEED) -> torch.Tensor:
    return uniform_tokens(n, cfg.vocab, seed, "prompt")


def decode_tokens(cfg: ModelConfig, n: int, seed: int = DECODE_SEED) -> torch.Tensor:
    return uniform_tokens(n, cfg.vocab, seed, "decode")
