"""ctypes binding of the CPU oracle (TEST INFRASTRUCTURE ONLY).

Only tests/, the smoke check and the benchmark's CPU-baseline / reference
legs import this module.  It never imports the CUDA package and the CUDA
package never imports it.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import build as _build

ORC_BF16, ORC_INT8, ORC_INT4 = 0, 1, 2
_FMT = {"bf16": ORC_BF16, "int8": ORC_INT8, "int4": ORC_INT4}


class OrcLinear(C.Structure):
    _fields_ = [("format", C.c_int32), ("w", C.c_void_p),
                ("scales", C.c_void_p), ("zeros", C.c_void_p)]


class OrcLayer(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p)] + [
        (n, OrcLinear) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")]


class OrcWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p),
                ("lm_head", OrcLinear), ("layers", C.POINTER(OrcLayer))]


class OrcConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("max_seq", C.c_int64),
                ("rms_eps", C.c_double), ("rope_theta", C.c_double)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        dp = C.POINTER(C.c_double)
        L.orc_bf16_to_double.restype = C.c_double
        L.orc_bf16_to_double.argtypes = [C.c_uint16]
        L.orc_bf16_from_double.restype = C.c_uint16
        L.orc_bf16_from_double.argtypes = [C.c_double]
        L.orc_fp16_to_double.restype = C.c_double
        L.orc_fp16_to_double.argtypes = [C.c_uint16]
        L.orc_dequant_row.argtypes = [C.POINTER(OrcLinear), C.c_int64, C.c_int64, C.c_int64, dp]
        L.orc_linear_apply.argtypes = [C.POINTER(OrcLinear), C.c_int64, C.c_int64, dp, dp]
        L.orc_rmsnorm.argtypes = [dp, C.c_void_p, C.c_int64, C.c_double, dp]
        L.orc_rope.argtypes = [dp, C.c_int32, C.c_int32, C.c_int64, C.c_double]
        L.orc_silu.restype = C.c_double
        L.orc_silu.argtypes = [C.c_double]
        L.orc_attention.argtypes = [dp, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                    C.c_int64, C.c_int64, dp]
        L.orc_decode_step.restype = C.c_int
        L.orc_decode_step.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), C.c_void_p,
                                      C.c_int32, C.c_int64, dp]
        L.orc_decode_layers.restype = C.c_int
        L.orc_decode_layers.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), C.c_void_p,
                                        dp, C.c_int64, C.c_int32, C.c_int32]
        L.orc_logits_rows.restype = C.c_int
        L.orc_logits_rows.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), dp, dp,
                                      C.c_int64, C.c_int64]
        L.orc_prefill.restype = C.c_int
        L.orc_prefill.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), C.c_void_p,
                                  C.POINTER(C.c_int32), C.c_int64, C.c_int64]
        L.orc_prefill_batched.restype = C.c_int
        L.orc_prefill_batched.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), C.c_void_p,
                                          C.POINTER(C.c_int32), C.c_int64, C.c_int64]
        L.orc_set_threads.argtypes = [C.c_int]
        L.orc_get_threads.restype = C.c_int
        _lib = L
    return _lib


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return C.c_void_p(t.data_ptr())


def make_linear(lin, keep: list) -> OrcLinear:
    """OrcLinear view of a workload.synth.Linear held on the host."""
    for t in lin.tensors():
        keep.append(t)
    return OrcLinear(_FMT[lin.fmt], _ptr(lin.w), _ptr(lin.scales), _ptr(lin.zeros))


# ------------------------------------------------------------ per-op calls

def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(bits)


def bf16_from_double(v: float) -> int:
    return lib().orc_bf16_from_double(v)


def fp16_to_double(bits: int) -> float:
    return lib().orc_fp16_to_double(bits)


def dequant(lin) -> np.ndarray:
    """Every element of a stored linear map as exact doubles [out, in]."""
    keep = []
    ol = make_linear(lin, keep)
    out = np.empty((lin.out_features, lin.in_features), dtype=np.float64)
    for r in range(lin.out_features):
        lib().orc_dequant_row(C.byref(ol), lin.out_features, lin.in_features, r,
                              _dp(out[r]))
    return out


def linear(lin, x: np.ndarray) -> np.ndarray:
    keep = []
    ol = make_linear(lin, keep)
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(lin.out_features, dtype=np.float64)
    lib().orc_linear_apply(C.byref(ol), lin.out_features, lin.in_features, _dp(x), _dp(y))
    return y


def rmsnorm(x: np.ndarray, w_bf16=None, eps: float = 1e-5) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_dp(x), _ptr(w_bf16), x.size, eps, _dp(out))
    return out


def rope(v: np.ndarray, n_heads: int, head_dim: int, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True).reshape(-1)
    lib().orc_rope(_dp(v), n_heads, head_dim, pos, theta)
    return v


def silu(z: float) -> float:
    return lib().orc_silu(z)


def attention(q: np.ndarray, k_bf16: torch.Tensor, v_bf16: torch.Tensor, n_heads: int,
              n_kv_heads: int, head_dim: int, ctx: int) -> np.ndarray:
    """q [n_heads*head_dim] doubles; k, v bf16 [n_kv_heads, max_seq, head_dim]."""
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(-1)
    max_seq = k_bf16.shape[1]
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    lib().orc_attention(_dp(q), _ptr(k_bf16), _ptr(v_bf16), n_heads, n_kv_heads, head_dim,
                        max_seq, ctx, _dp(out))
    return out


# ------------------------------------------------------------ whole model

class OracleModel:
    """The oracle decoder over host copies of a workload.synth.ModelWeights."""

    def __init__(self, weights, max_seq: int):
        cfg = weights.cfg
        self.cfg = cfg
        self.max_seq = int(max_seq)
        self._keep = []
        w = weights.to("cpu") if weights.embed.device.type != "cpu" else weights
        self._w = w
        self._layers = (OrcLayer * cfg.n_layers)()
        for li, lw in enumerate(w.layers):
            L = self._layers[li]
            L.attn_norm = _ptr(lw["attn_norm"])
            L.ffn_norm = _ptr(lw["ffn_norm"])
            for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                setattr(L, n, make_linear(lw[n], self._keep))
        self._weights = OrcWeights(_ptr(w.embed), _ptr(w.final_norm),
                                   make_linear(w.lm_head_linear(), self._keep),
                                   C.cast(self._layers, C.POINTER(OrcLayer)))
        self._cfg = OrcConfig(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads,
                              cfg.head_dim, cfg.ffn, cfg.vocab, self.max_seq,
                              cfg.rms_eps, cfg.rope_theta)

    def _check_kv(self, kv: torch.Tensor):
        c = self.cfg
        exp = (c.n_layers, 2, c.n_kv_heads, self.max_seq, c.head_dim)
        if tuple(kv.shape) != exp or kv.dtype != torch.bfloat16 or kv.device.type != "cpu" \
                or not kv.is_contiguous():
            raise ValueError(f"oracle KV cache must be contiguous host bf16 {exp}")

    def decode_step(self, kv: torch.Tensor, token: int, pos: int, logits: bool = True):
        self._check_kv(kv)
        out = np.empty(self.cfg.vocab, dtype=np.float64) if logits else None
        rc = lib().orc_decode_step(C.byref(self._cfg), C.byref(self._weights),
                                   C.c_void_p(kv.data_ptr()), int(token), int(pos),
                                   _dp(out) if logits else None)
        if rc != 0:
            raise ValueError("oracle decode step rejected its arguments")
        return out

    def embed(self, token: int) -> np.ndarray:
        return self._w.embed[int(token)].double().numpy().copy()

    def decode_layers(self, kv: torch.Tensor, x: np.ndarray, pos: int, l0: int, l1: int):
        """Layers [l0, l1) of a decode step, in place on the residual x."""
        self._check_kv(kv)
        assert x.dtype == np.float64 and x.flags["C_CONTIGUOUS"] and x.size == self.cfg.hidden
        rc = lib().orc_decode_layers(C.byref(self._cfg), C.byref(self._weights),
                                     C.c_void_p(kv.data_ptr()), _dp(x), int(pos), int(l0), int(l1))
        if rc != 0:
            raise ValueError("oracle decode_layers rejected its arguments")

    def logits_rows(self, x: np.ndarray, r0: int, r1: int, out: np.ndarray | None = None):
        """Final norm + LM-head rows [r0, r1) (written into out[r0:r1])."""
        out = np.zeros(self.cfg.vocab, dtype=np.float64) if out is None else out
        rc = lib().orc_logits_rows(C.byref(self._cfg), C.byref(self._weights), _dp(x), _dp(out),
                                   int(r0), int(r1))
        if rc != 0:
            raise ValueError("oracle logits_rows rejected its arguments")
        return out

    def prefill(self, kv: torch.Tensor, tokens, start_pos: int = 0):
        """Sequential decode steps without logits (orc_prefill)."""
        self._check_kv(kv)
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        rc = lib().orc_prefill(C.byref(self._cfg), C.byref(self._weights),
                               C.c_void_p(kv.data_ptr()),
                               t.ctypes.data_as(C.POINTER(C.c_int32)), t.size, int(start_pos))
        if rc != 0:
            raise ValueError("oracle prefill rejected its arguments")

    def prefill_batched(self, kv: torch.Tensor, tokens, start_pos: int = 0):
        """The batched causal prefill (orc_prefill_batched): layer-major over
        all the prompt's tokens."""
        self._check_kv(kv)
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        rc = lib().orc_prefill_batched(C.byref(self._cfg), C.byref(self._weights),
                                       C.c_void_p(kv.data_ptr()),
                                       t.ctypes.data_as(C.POINTER(C.c_int32)), t.size, int(start_pos))
        if rc != 0:
            raise ValueError("oracle batched prefill rejected its arguments")


def library_path() -> str:
    return os.path.abspath(_build.LIB)
