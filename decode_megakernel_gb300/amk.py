"""ctypes binding of libamk.so (include/amk.h), same names as the C ABI.

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Importing this module loads libamk.so and raises if it is
missing; there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libamk.so")

AMK_OK = 0
AMK_ERR_INVALID_ARG = 1
AMK_ERR_UNSUPPORTED = 2
AMK_ERR_SCHEDULE_INVALID = 3
AMK_ERR_CUDA = 4
AMK_ERR_OOM = 5
AMK_ERR_TIMEOUT = 6
AMK_ERR_DEVICE_CHECK = 7

AMK_FORMAT_BF16, AMK_FORMAT_INT8, AMK_FORMAT_INT4 = 0, 1, 2
FORMAT_CODE = {"bf16": AMK_FORMAT_BF16, "int8": AMK_FORMAT_INT8, "int4": AMK_FORMAT_INT4}


class amk_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("max_seq", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("tied_embeddings", C.c_int32),
                ("weight_format", C.c_int32), ("lm_head_format", C.c_int32)]


class amk_linear(C.Structure):
    _fields_ = [("w", C.c_void_p), ("scales", C.c_void_p), ("zeros", C.c_void_p)]


class amk_layer_weights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p)] + [
        (n, amk_linear) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")]


class amk_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", amk_linear),
                ("layers", C.POINTER(amk_layer_weights))]


class amk_schedule_config(C.Structure):
    _fields_ = [("num_ctas", C.c_int32), ("attn_splits", C.c_int32),
                ("max_rows_per_task", C.c_int32), ("watchdog_ms", C.c_int32),
                ("ring_slots", C.c_int32), ("l2_prefetch_tiles", C.c_int32),
                ("prefill_chunk", C.c_int32), ("prefill_parts", C.c_int32),
                ("prefill_tile_rows", C.c_int32)]


class AmkError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_string(status)} ({status}): {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libamk.so is not built ({LIB_PATH}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = C.CDLL(LIB_PATH)
    P = C.c_void_p
    cfgp = C.POINTER(amk_config)
    schp = C.POINTER(amk_schedule_config)
    sig = {
        "amk_workspace_bytes": (C.c_size_t, [cfgp, schp]),
        "amk_prefill_chunk": (C.c_int32, [P]),
        "amk_check_config": (C.c_int, [cfgp]),
        "amk_kv_cache_bytes": (C.c_size_t, [cfgp]),
        "amk_load_weights": (C.c_int, [cfgp, C.POINTER(amk_weights), P, C.c_size_t, P, P, schp,
                                       C.POINTER(P)]),
        "amk_load_weights_requeued": (C.c_int, [cfgp, C.POINTER(amk_weights), P, C.c_size_t, P, P, schp, P,
                                                C.c_size_t, C.POINTER(P)]),
        "amk_weights_staging_bytes": (C.c_size_t, [cfgp]),
        "amk_load_weights_staged": (C.c_int, [cfgp, C.POINTER(amk_weights), P, C.c_size_t, P, P, schp, P,
                                              C.c_size_t, C.POINTER(P)]),
        "amk_prefill": (C.c_int, [P, C.POINTER(C.c_int32), C.c_int32, C.c_int32]),
        "amk_decode_step": (C.c_int, [P, C.c_int32, C.c_int32, P]),
        "amk_decode_step_host": (C.c_int, [P, C.c_int32, C.c_int32, P]),
        "amk_generate": (C.c_int, [P, C.c_int32, C.c_int32, C.c_int32, P, P]),
        "amk_decode_step_static_scratch": (C.c_int, [P, C.c_int32, C.c_int32, P]),
        "amk_set_kv_length": (C.c_int, [P, C.c_int32]),
        "amk_kv_length": (C.c_int32, [P]),
        "amk_sync": (C.c_int, [P]),
        "amk_free": (None, [P]),
        "amk_status_string": (C.c_char_p, [C.c_int]),
        "amk_last_error": (C.c_char_p, [P]),
        "amk_build_schedule": (C.c_int, [cfgp, schp, P, C.c_size_t, C.POINTER(C.c_size_t)]),
        "amk_validate_serialized": (C.c_int, [P, C.c_size_t, C.c_char_p, C.c_size_t]),
        "amk_validate_requeued": (C.c_int, [cfgp, schp, P, C.c_size_t, C.c_char_p, C.c_size_t]),
        "amk_debug_watchdog_probe": (C.c_int, [P, P, C.c_int32, C.POINTER(C.c_int32)]),
        "amk_debug_trace_bytes": (C.c_size_t, [P, C.POINTER(C.c_int32)]),
        "amk_debug_trace_step": (C.c_int, [P, C.c_int32, C.c_int32, P, P, C.c_size_t]),
        "amk_debug_dequant": (C.c_int, [C.c_int32, C.POINTER(amk_linear), C.c_int32, C.c_int32,
                                        P, P]),
        "amk_debug_hbm_read_probe": (C.c_int, [C.c_int32, P, C.c_size_t, P, C.c_size_t, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def status_string(s: int) -> str:
    return lib.amk_status_string(int(s)).decode()


def last_error(ctx=None) -> str:
    r = lib.amk_last_error(ctx)
    return r.decode() if r else ""


def check(status: int, ctx=None):
    if status != AMK_OK:
        raise AmkError(status, last_error(ctx))


# ------------------------------------------------------------ same-name calls

def amk_workspace_bytes(cfg: amk_config, sched: amk_schedule_config | None = None) -> int:
    return int(lib.amk_workspace_bytes(C.byref(cfg), C.byref(sched) if sched else None))


def amk_check_config(cfg: amk_config) -> int:
    return int(lib.amk_check_config(C.byref(cfg)))


def amk_kv_cache_bytes(cfg: amk_config) -> int:
    return int(lib.amk_kv_cache_bytes(C.byref(cfg)))


def amk_load_weights(cfg, weights, workspace_ptr, workspace_bytes, kv_ptr, stream_ptr, sched=None):
    ctx = C.c_void_p()
    st = lib.amk_load_weights(C.byref(cfg), C.byref(weights), C.c_void_p(workspace_ptr),
                              workspace_bytes, C.c_void_p(kv_ptr), C.c_void_p(stream_ptr),
                              C.byref(sched) if sched else None, C.byref(ctx))
    return st, ctx


def amk_weights_staging_bytes(cfg) -> int:
    return int(lib.amk_weights_staging_bytes(C.byref(cfg)))


def amk_load_weights_staged(cfg, host_weights, workspace_ptr, workspace_bytes, kv_ptr, stream_ptr, sched,
                            staging_ptr, staging_bytes):
    ctx = C.c_void_p()
    st = lib.amk_load_weights_staged(C.byref(cfg), C.byref(host_weights), C.c_void_p(workspace_ptr),
                                     workspace_bytes, C.c_void_p(kv_ptr), C.c_void_p(stream_ptr),
                                     C.byref(sched) if sched else None, C.c_void_p(staging_ptr), staging_bytes,
                                     C.byref(ctx))
    return st, ctx


def amk_load_weights_requeued(cfg, weights, workspace_ptr, workspace_bytes, kv_ptr, stream_ptr, sched,
                              schedule: bytes):
    ctx = C.c_void_p()
    st = lib.amk_load_weights_requeued(C.byref(cfg), C.byref(weights), C.c_void_p(workspace_ptr),
                                       workspace_bytes, C.c_void_p(kv_ptr), C.c_void_p(stream_ptr),
                                       C.byref(sched) if sched else None, schedule, len(schedule),
                                       C.byref(ctx))
    return st, ctx


def amk_prefill(ctx, tokens, start_pos: int) -> int:
    arr = (C.c_int32 * len(tokens))(*[int(t) for t in tokens])
    return int(lib.amk_prefill(ctx, arr, len(tokens), int(start_pos)))


def amk_decode_step(ctx, token: int, pos: int, logits_ptr: int) -> int:
    return int(lib.amk_decode_step(ctx, int(token), int(pos), C.c_void_p(logits_ptr)))


def amk_decode_step_host(ctx, token: int, pos: int, logits_host_ptr: int) -> int:
    return int(lib.amk_decode_step_host(ctx, int(token), int(pos), C.c_void_p(logits_host_ptr)))


def amk_generate(ctx, first_token: int, pos: int, n_steps: int, tokens_dev_ptr: int,
                 logits_dev_ptr: int = 0) -> int:
    return int(lib.amk_generate(ctx, int(first_token), int(pos), int(n_steps),
                                C.c_void_p(tokens_dev_ptr), C.c_void_p(logits_dev_ptr or None)))


def amk_decode_step_static_scratch(ctx, token: int, pos: int, logits_ptr: int) -> int:
    """amk_decode_step with the per-step scratch in the library's fixed
    device array: for callers that cannot allocate device memory."""
    return int(lib.amk_decode_step_static_scratch(ctx, int(token), int(pos),
                                                  C.c_void_p(logits_ptr)))


def amk_set_kv_length(ctx, n: int) -> int:
    return int(lib.amk_set_kv_length(ctx, int(n)))


def amk_kv_length(ctx) -> int:
    return int(lib.amk_kv_length(ctx))


def amk_prefill_chunk(ctx) -> int:
    return int(lib.amk_prefill_chunk(ctx))


def amk_sync(ctx) -> int:
    return int(lib.amk_sync(ctx))


def amk_free(ctx) -> None:
    lib.amk_free(ctx)


def amk_build_schedule(cfg: amk_config, sched: amk_schedule_config | None = None) -> bytes:
    need = C.c_size_t(0)
    sp = C.byref(sched) if sched else None
    check(lib.amk_build_schedule(C.byref(cfg), sp, None, 0, C.byref(need)))
    buf = C.create_string_buffer(need.value)
    check(lib.amk_build_schedule(C.byref(cfg), sp, buf, need.value, C.byref(need)))
    return buf.raw[:need.value]


def amk_validate_serialized(blob: bytes):
    rep = C.create_string_buffer(512)
    st = lib.amk_validate_serialized(blob, len(blob), rep, 512)
    return int(st), rep.value.decode()


def amk_validate_requeued(cfg: amk_config, sched: amk_schedule_config | None, blob: bytes):
    rep = C.create_string_buffer(512)
    st = lib.amk_validate_requeued(C.byref(cfg), C.byref(sched) if sched else None, blob, len(blob), rep, 512)
    return int(st), rep.value.decode()


def amk_debug_watchdog_probe(scratch_ptr: int, stream_ptr: int, limit_us: int):
    dst = C.c_int32(-1)
    st = lib.amk_debug_watchdog_probe(C.c_void_p(scratch_ptr), C.c_void_p(stream_ptr),
                                      int(limit_us), C.byref(dst))
    return int(st), int(dst.value)


def amk_debug_trace_bytes(ctx):
    stride = C.c_int32(0)
    n = int(lib.amk_debug_trace_bytes(ctx, C.byref(stride)))
    return n, int(stride.value)


def amk_debug_trace_step(ctx, token: int, pos: int, logits_ptr: int, trace_ptr: int,
                         trace_bytes: int) -> int:
    return int(lib.amk_debug_trace_step(ctx, int(token), int(pos), C.c_void_p(logits_ptr),
                                        C.c_void_p(trace_ptr), int(trace_bytes)))


def amk_debug_dequant(fmt: int, w_ptr, s_ptr, z_ptr, out_features, in_features, out_ptr,
                      stream_ptr) -> int:
    lin = amk_linear(w_ptr, s_ptr, z_ptr)
    return int(lib.amk_debug_dequant(int(fmt), C.byref(lin), int(out_features), int(in_features),
                                     C.c_void_p(out_ptr), C.c_void_p(stream_ptr)))


def amk_debug_hbm_read_probe(mode: int, buf_ptr: int, nbytes: int, out_ptr: int, out_words: int,
                             stream_ptr: int) -> int:
    return int(lib.amk_debug_hbm_read_probe(int(mode), C.c_void_p(buf_ptr), int(nbytes),
                                            C.c_void_p(out_ptr), int(out_words), C.c_void_p(stream_ptr)))


# ------------------------------------------------------------ marshalling helpers

def make_config(model, max_seq: int) -> amk_config:
    """amk_config from any object with the HF-style shape attributes."""
    lm_fmt = getattr(model, "lm_head_format", model.weight_format)
    return amk_config(model.n_layers, model.hidden, model.n_heads, model.n_kv_heads,
                      model.head_dim, model.ffn, model.vocab, int(max_seq), float(model.rms_eps),
                      float(model.rope_theta), int(bool(model.tied_embeddings)),
                      FORMAT_CODE[model.weight_format], FORMAT_CODE[lm_fmt])


def make_schedule_config(num_ctas=0, attn_splits=0, max_rows_per_task=0, watchdog_ms=0,
                         ring_slots=0, l2_prefetch_tiles=0, prefill_chunk=0, prefill_parts=0,
                         prefill_tile_rows=0):
    return amk_schedule_config(num_ctas, attn_splits, max_rows_per_task, watchdog_ms,
                               ring_slots, l2_prefetch_tiles, prefill_chunk, prefill_parts,
                               prefill_tile_rows)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _linear(lin):
    return amk_linear(_ptr(lin.w), _ptr(lin.scales), _ptr(lin.zeros))


class Decoder:
    """One loaded model: owns (through torch) its workspace and KV cache.

    ``weights`` holds tensors with attributes embed, final_norm, lm_head
    (or None when tied) and layers (dicts of attn_norm, ffn_norm and wq..wd
    objects carrying .w / .scales / .zeros): device tensors, or host tensors
    (then loaded through a device staging buffer, amk_load_weights_staged,
    onto `device`)."""

    def __init__(self, weights, max_seq: int, stream: torch.cuda.Stream | None = None,
                 sched: amk_schedule_config | None = None, kv_cache: torch.Tensor | None = None,
                 schedule: bytes | None = None, device: torch.device | None = None):
        """schedule: optional serialised re-queueing of the lowering's tasks
        (amk_load_weights_requeued); None loads the library's own lowering."""
        cfg = weights.cfg
        self.model = cfg
        self.cfg = make_config(cfg, max_seq)
        self.sched = sched
        self.stream = stream or torch.cuda.current_stream()
        nbytes = amk_workspace_bytes(self.cfg, sched)
        if nbytes == 0:
            raise AmkError(AMK_ERR_UNSUPPORTED, last_error())
        host = weights.embed.device.type == "cpu"
        dev = (device or torch.device("cuda", torch.cuda.current_device())) if host else weights.embed.device
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        if kv_cache is None:
            kv_cache = torch.zeros((cfg.n_layers, 2, cfg.n_kv_heads, max_seq, cfg.head_dim),
                                   dtype=torch.bfloat16, device=dev)
        self.kv = kv_cache
        layers = (amk_layer_weights * cfg.n_layers)()
        for i, lw in enumerate(weights.layers):
            layers[i].attn_norm = _ptr(lw["attn_norm"])
            layers[i].ffn_norm = _ptr(lw["ffn_norm"])
            for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                setattr(layers[i], n, _linear(lw[n]))
        w = amk_weights(_ptr(weights.embed), _ptr(weights.final_norm),
                        _linear(weights.lm_head) if weights.lm_head is not None else amk_linear(),
                        C.cast(layers, C.POINTER(amk_layer_weights)))
        if host:
            if schedule is not None:
                raise ValueError("a re-queued schedule needs device weights")
            sb = amk_weights_staging_bytes(self.cfg)
            staging = torch.empty(max(sb, 256), dtype=torch.uint8, device=dev)
            st, ctx = amk_load_weights_staged(self.cfg, w, self.workspace.data_ptr(), nbytes,
                                              self.kv.data_ptr(), self.stream.cuda_stream, sched,
                                              staging.data_ptr(), sb)
            del staging
        elif schedule is None:
            st, ctx = amk_load_weights(self.cfg, w, self.workspace.data_ptr(), nbytes,
                                       self.kv.data_ptr(), self.stream.cuda_stream, sched)
        else:
            st, ctx = amk_load_weights_requeued(self.cfg, w, self.workspace.data_ptr(), nbytes,
                                                self.kv.data_ptr(), self.stream.cuda_stream, sched,
                                                bytes(schedule))
        check(st)
        self.ctx = ctx

    def prefill(self, tokens, start_pos: int = 0):
        check(amk_prefill(self.ctx, list(tokens), start_pos), self.ctx)

    def decode_step(self, token: int, pos: int, logits: torch.Tensor):
        assert logits.dtype == torch.float32 and logits.is_cuda and logits.numel() >= self.model.vocab
        check(amk_decode_step(self.ctx, token, pos, logits.data_ptr()), self.ctx)

    def decode_step_host(self, token: int, pos: int, logits_host: torch.Tensor):
        assert logits_host.dtype == torch.float32 and not logits_host.is_cuda
        check(amk_decode_step_host(self.ctx, token, pos, logits_host.data_ptr()), self.ctx)

    def generate(self, first_token: int, pos: int, n_steps: int, tokens: torch.Tensor,
                 logits: torch.Tensor | None = None):
        """Greedy decoding on the device (amk_generate): tokens (int32 cuda
        [n_steps]) receives the argmax of each step's logits."""
        assert tokens.dtype == torch.int32 and tokens.is_cuda and tokens.numel() >= n_steps
        lp = 0
        if logits is not None:
            assert logits.dtype == torch.float32 and logits.is_cuda
            lp = logits.data_ptr()
        check(amk_generate(self.ctx, first_token, pos, n_steps, tokens.data_ptr(), lp), self.ctx)

    @property
    def prefill_chunk(self) -> int:
        """Tokens per tensor-core prefill chunk (0: prefill by decode steps)."""
        return amk_prefill_chunk(self.ctx)

    def set_kv_length(self, n: int):
        check(amk_set_kv_length(self.ctx, n), self.ctx)

    def sync(self):
        check(amk_sync(self.ctx), self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            amk_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
