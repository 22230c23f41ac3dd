/*
 * amk.h: C ABI of the GB300 batch-1 decode megakernel library (libamk.so).
 *
 * The library runs one autoregressive decode step of a Llama-family decoder
 * at batch 1 (RMSNorm, QKV / O / gate-up / down / LM-head matrix-vector
 * products, RoPE, GQA attention over a bf16 KV cache, SwiGLU) as ONE
 * persistent CUDA kernel launch per token on an sm_103a GPU.  This is the
 * path the AutoMegaKernel pages target ("Problem statement": single-stream
 * batch-1 decode is bandwidth bound with floor t_min = weight_bytes / HBM
 * bandwidth; launching one kernel per operator and round-tripping
 * activations through HBM misses that floor).
 *
 * Conventions for every entry point:
 *   - Device memory is allocated by the caller (for example through
 *     PyTorch) and only borrowed by the library; the library allocates no
 *     device memory of its own.  Host memory it owns is freed by amk_free.
 *   - Pointers named *_dev are device pointers, *_host host pointers.
 *   - Functions return an amk_status and never abort the process.  Device
 *     work is stream ordered and asynchronous: failures that happen on the
 *     device (watchdog timeout, device-side check) are reported by the next
 *     amk_sync().  After AMK_ERR_TIMEOUT or AMK_ERR_DEVICE_CHECK the context
 *     is poisoned: every later call returns the same status and the caller
 *     must amk_free it (and may load a fresh context).
 *   - Calls on one context must not overlap from several host threads.
 */
#ifndef AMK_H
#define AMK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    AMK_OK = 0,
    AMK_ERR_INVALID_ARG = 1,       /* a NULL pointer, a size or an index out of range */
    AMK_ERR_UNSUPPORTED = 2,       /* a model variant the kernel does not implement */
    AMK_ERR_SCHEDULE_INVALID = 3,  /* the task schedule failed validation: nothing launched */
    AMK_ERR_CUDA = 4,              /* a CUDA runtime call failed (see amk_last_error) */
    AMK_ERR_OOM = 5,               /* the caller's workspace is smaller than required */
    AMK_ERR_TIMEOUT = 6,           /* a device-side wait hit the watchdog; context poisoned */
    AMK_ERR_DEVICE_CHECK = 7       /* a device-side consistency check failed; context poisoned */
} amk_status;

enum { AMK_FORMAT_BF16 = 0, AMK_FORMAT_INT8 = 1, AMK_FORMAT_INT4 = 2 };

/*
 * Model shape (HuggingFace Llama conventions).
 * Supported (else AMK_ERR_UNSUPPORTED, the analogue of the pages' rejection
 * of unsupported variants such as biased projections, AMK "Key
 * contributions" 2): no biases; head_dim 64 or 128; n_heads a multiple of
 * n_kv_heads with (n_heads / n_kv_heads) * head_dim <= 512; in_features of
 * every matrix <= 16384 (after padding to the kernel's tile); int4 needs
 * hidden, n_heads*head_dim and ffn to be multiples of 128.
 */
typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
    int32_t max_seq;          /* KV cache capacity in positions */
    float rms_eps;
    float rope_theta;         /* rotate-half RoPE base; no frequency scaling */
    int32_t tied_embeddings;  /* 1: the LM head is the embedding matrix */
    int32_t weight_format;    /* AMK_FORMAT_* of the 7 per-layer matrices */
    int32_t lm_head_format;   /* AMK_FORMAT_* of an untied LM head (ignored when tied) */
} amk_config;

/*
 * One weight matrix W [out_features][in_features] (nn.Linear layout), device
 * pointers, in one of three formats:
 *   BF16: w = bf16 [out][in]; scales = zeros = NULL.
 *   INT8: w = int8 [out][in]; scales = fp16 [out]; W = q * s_row.
 *   INT4: w = uint8 [out][in/2], two codes per byte, low nibble = even k;
 *         scales = fp16 [out][in/128];
 *         zeros = uint8 [out][ceil(in/256)], two 4-bit zero points per byte,
 *         low nibble = even group; W = (q - z_group) * s_group.
 * (int8 / int4 weight-only formats: AMK "Key contributions" 4.)
 */
typedef struct {
    const void* w;
    const void* scales;
    const void* zeros;
} amk_linear;

typedef struct {
    const void* attn_norm;    /* bf16 [hidden] */
    const void* ffn_norm;     /* bf16 [hidden] */
    amk_linear wq, wk, wv, wo, wg, wu, wd;
} amk_layer_weights;

typedef struct {
    const void* embed;                 /* bf16 [vocab][hidden] */
    const void* final_norm;            /* bf16 [hidden] */
    amk_linear lm_head;                /* ignored when tied_embeddings */
    const amk_layer_weights* layers;   /* HOST array [n_layers] of device pointers */
} amk_weights;

/*
 * Schedule knobs (the pages' ScheduleConfig, AMK "Layer 2": tiling, SM
 * assignment).  Zero selects the default for every field.
 */
typedef struct {
    int32_t num_ctas;           /* persistent CTAs (default: one per SM) */
    int32_t attn_splits;        /* context splits per KV head (default: num_ctas / n_kv_heads) */
    int32_t max_rows_per_task;  /* rows of one GEMV task (default and maximum 256) */
    int32_t watchdog_ms;        /* device wait limit before AMK_ERR_TIMEOUT (default 2000) */
    int32_t ring_slots;         /* copies in flight per CTA, 1..12.  Each CTA streams the
                                   weight tiles of its GEMV tasks and the K,V history stages
                                   of its attention tasks, in queue order, through one ring
                                   of 12 shared-memory slots of 17 KB; a copy is issued once
                                   its slot is free and the copy ring_slots before it has
                                   landed.  0 (default): 6; values above 12 act as 12 */
    int32_t l2_prefetch_tiles;  /* weight tiles a CTA may prefetch into L2 beyond its full
                                   ring while its consumers run attention, the split merge
                                   or the O projection (-1: off; 0: default) */
    int32_t prefill_chunk;      /* tokens per chunk of the tensor-core prefill (bf16 weights):
                                   0: default 2048 (at most max_seq rounded up to 128);
                                   -1: prefill through the decode kernel, one launch per
                                   token (always so for int8 / int4 weights) */
    int32_t prefill_parts;      /* bf16 parts per activation operand of the prefill GEMMs:
                                   0 or 2: two (activations to 2^-18 relative, the default);
                                   3: three (fp32-level products, 1.5x the tensor work) */
    int32_t prefill_tile_rows;  /* weight rows per prefill GEMM tile (the MMA's N): 0 (default):
                                   per matrix 256 or 224, whichever covers a full chunk in
                                   fewer tile-rows when every SM runs one tile at a time;
                                   256 or 224: that width for every matrix */
} amk_schedule_config;

typedef struct amk_ctx amk_ctx;

/*
 * Bytes of device workspace amk_load_weights needs for this model (repacked
 * weights, tagged activation words, task table, status words).  Host only when
 * sched->num_ctas > 0; otherwise it reads the SM count of the current
 * device.  Returns 0 for an unsupported or invalid configuration.
 */
size_t amk_workspace_bytes(const amk_config* cfg, const amk_schedule_config* sched);

/* Shape check alone (host only): AMK_OK, AMK_ERR_INVALID_ARG or AMK_ERR_UNSUPPORTED. */
amk_status amk_check_config(const amk_config* cfg);

/* Bytes of the KV cache the caller allocates: bf16 [n_layers][2 (K,V)][n_kv_heads][max_seq][head_dim]. */
size_t amk_kv_cache_bytes(const amk_config* cfg);

/*
 * Build, validate and upload the task schedule, then repack the weights into
 * the workspace (tile-major, RoPE pairs and gate/up rows interleaved).
 *   workspace_dev  caller-owned, >= amk_workspace_bytes, 256-byte aligned;
 *   kv_cache_dev   caller-owned, amk_kv_cache_bytes, 16-byte aligned; its
 *                  content is kept: positions [0, n) become valid through
 *                  amk_prefill, amk_decode_step or amk_set_kv_length;
 *   stream         cudaStream_t (NULL = legacy default stream) that every
 *                  launch of this context is ordered on.
 * The schedule is checked (one writer per element and version, every read
 * satisfiable, acyclic, readers ordered before the next version's writer,
 * no stale word old enough for its 4-bit tag to alias, race-free untagged
 * buffers, output coverage; the conditions of AMK "The safety gate" for
 * counters fused with the data) before anything is
 * launched: a failure returns AMK_ERR_SCHEDULE_INVALID.
 * Synchronous: on return the caller's weight buffers are no longer needed.
 */
amk_status amk_load_weights(const amk_config* cfg, const amk_weights* weights,
                            void* workspace_dev, size_t workspace_bytes, void* kv_cache_dev,
                            void* stream, const amk_schedule_config* sched, amk_ctx** out);

/*
 * amk_load_weights with the task queues of a given schedule: the schedule
 * search's way to run a structural edit of the lowering (which CTA runs a
 * task, and in which order), the pages' "SM assignment" choices of the
 * ScheduleConfig (AMK "Layer 2").  schedule (host, schedule_bytes bytes)
 * is a serialised schedule in the format of amk_build_schedule that holds
 * exactly the tasks of this model's own lowering for (cfg, sched), matched
 * by type, layer and parameters, in any queues and order, with each
 * queue's LM-head tasks after its body and only there.  The library takes
 * the task set and every task's memory accesses from its own lowering and
 * only the placement from the given schedule, then runs the safety gate on
 * the result: a schedule that is malformed, holds other tasks, or fails the
 * gate (for example a queue order that deadlocks) returns
 * AMK_ERR_SCHEDULE_INVALID with the reason, and nothing is launched.
 * Everything else is as amk_load_weights (same workspace size).
 */
amk_status amk_load_weights_requeued(const amk_config* cfg, const amk_weights* weights,
                                     void* workspace_dev, size_t workspace_bytes, void* kv_cache_dev,
                                     void* stream, const amk_schedule_config* sched,
                                     const void* schedule, size_t schedule_bytes, amk_ctx** out);

/*
 * Bytes of the device staging buffer amk_load_weights_staged needs for this
 * model: the largest group of matrices repacked together (QKV, O, gate + up,
 * down, or the untied LM head) in their stored formats, each tensor rounded
 * up to 256 bytes; 0 for an unsupported config.  Host only.
 */
size_t amk_weights_staging_bytes(const amk_config* cfg);

/*
 * amk_load_weights with the weights in HOST memory (every pointer of
 * host_weights, the layer table included, is host memory; page-locked
 * memory copies fastest): the embedding and the norms are copied straight
 * into the workspace, and each group of matrices is copied into staging_dev
 * (caller-owned device memory, 256-byte aligned, at least
 * amk_weights_staging_bytes) and repacked from there, so the device holds
 * the packed model plus one staging buffer instead of the caller's copy of
 * the model as well.  The call returns after the stream has finished the
 * copies: staging_dev and the host weights may be freed when it returns.
 * Errors as amk_load_weights; a NULL, misaligned or too small staging
 * buffer is AMK_ERR_INVALID_ARG.
 */
amk_status amk_load_weights_staged(const amk_config* cfg, const amk_weights* host_weights, void* workspace_dev,
                                   size_t workspace_bytes, void* kv_cache_dev, void* stream,
                                   const amk_schedule_config* sched, void* staging_dev, size_t staging_bytes,
                                   amk_ctx** out);

/*
 * Fill the KV cache with the K,V rows of host_tokens at positions
 * start_pos .. start_pos + n - 1 (start_pos <= the valid KV length,
 * start_pos + n <= max_seq, every token in [0, vocab)); no logits.
 * With bf16 weights (and prefill_chunk >= 0) the tokens go through the
 * tensor-core prefill in chunks of prefill_chunk tokens: per layer an
 * RMSNorm, a QKV GEMM with RoPE and the KV append fused, causal GQA
 * attention over the cache, and the O / gate-up / down GEMMs with the
 * residual adds and SwiGLU fused (tcgen05 MMAs with fp32 accumulation, the
 * activations split into bf16 hi + lo halves).  Otherwise each token is one
 * decode step with the LM head skipped.  Asynchronous; host_tokens may be
 * reused once the call returns.
 */
amk_status amk_prefill(amk_ctx* ctx, const int32_t* host_tokens, int32_t n, int32_t start_pos);

/*
 * One decode step: token at position pos (0 <= pos <= valid KV length,
 * pos < max_seq; a smaller pos rolls the context back) writes K,V of pos
 * into the cache and fp32 logits [vocab] into logits_dev.  One persistent
 * kernel launch; asynchronous.
 */
amk_status amk_decode_step(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_dev);

/* The same step with the logits copied to host memory (pinned memory is
 * fastest); waits for the step to finish and reports device failures. */
amk_status amk_decode_step_host(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_host);

/*
 * The same decode step as amk_decode_step, for callers that cannot call
 * cudaMalloc: code that runs inside a host application whose allocator
 * owns all device memory and only lends it weight and cache buffers, or a
 * loop that is not allowed to allocate once it has started.  Such a caller
 * still passes its inputs (the loaded context, token, position) and its
 * output (logits_dev, fp32 [vocab], device memory); the scratch the step
 * needs besides them (the tagged activation words and attention partials,
 * status word) comes from a fixed array inside libamk.so instead
 * of the context's workspace.  The AMK pages have no counterpart to this
 * entry point.
 *   - Size limit: the array holds 1 MiB on every GPU that loads the library,
 *     kept until the process exits.  A model whose per-step scratch exceeds
 *     it (roughly: n_kv_heads * attn_splits * group * (head_dim + 2) * 4
 *     bytes of partials plus 4 * (2 * hidden + n_heads * head_dim +
 *     n_kv_heads * (group + 2) * head_dim + ffn))
 *     is rejected with AMK_ERR_OOM and a message giving both sizes.
 *   - Allocation: none.  No cudaMalloc, cudaFree or allocating library call.
 *   - Set-up: every call looks up the array's device address
 *     (cudaGetSymbolAddress) in the current device's context, so that an
 *     address never outlives its context (for example across a
 *     cudaDeviceReset); the first call on a device may load the library's
 *     device code, so make it before any stream capture.  The context's
 *     device must be the current device.
 *   - Sharing: every call uses the same array and finds the previous call's
 *     contents there; the call zeroes the whole scratch plan itself (each
 *     call runs with the tags of a context's first launch, so old words
 *     would carry the awaited tags).
 *     Calls that overlap on the GPU (other streams, other threads, other
 *     contexts on the same device) race on the array and must not be made.
 *   - Synchronous: returns after the step has finished, with the device
 *     status of that step (AMK_ERR_TIMEOUT / AMK_ERR_DEVICE_CHECK poison the
 *     context as for amk_sync, and so does a CUDA error while waiting for
 *     the step: AMK_ERR_CUDA).  Checks and KV bookkeeping are those of
 *     amk_decode_step.
 */
amk_status amk_decode_step_static_scratch(amk_ctx* ctx, int32_t token, int32_t pos,
                                          float* logits_dev);

/*
 * Greedy decoding on the device: n_steps decode steps from position pos
 * with no host round trip between them: the argmax of each step's
 * logits is the next step's token.  Step 0 consumes first_token;
 * each LM-head task also records the (max logit, row) of its rows, and
 * step i + 1 takes as its token the argmax of step i's records (the larger
 * logit wins, the smaller token id on a tie, as torch.argmax).  tokens_dev
 * (device, int32 [n_steps], 4-byte aligned) receives the generated tokens:
 * tokens_dev[i] = argmax of step i's logits.  logits_dev: NULL, or device
 * fp32 [vocab] that holds the last step's logits on completion.  Checks as
 * amk_decode_step for (first_token, pos); pos + n_steps <= max_seq.
 * Asynchronous: n_steps + 1 launches on the context's stream (the last
 * reduces the final step's records); the valid KV length becomes
 * pos + n_steps.  Device failures surface at amk_sync; a step whose
 * logits have no finite maximum reports AMK_ERR_DEVICE_CHECK.
 */
amk_status amk_generate(amk_ctx* ctx, int32_t first_token, int32_t pos, int32_t n_steps,
                        int32_t* tokens_dev, float* logits_dev);

/* Tokens per chunk of the context's tensor-core prefill; 0 when
 * amk_prefill runs decode steps (int8 / int4 weights, or prefill_chunk
 * -1); -1 for a NULL context. */
int32_t amk_prefill_chunk(const amk_ctx* ctx);

/* Declare KV positions [0, n) valid (a cache filled by the caller). */
amk_status amk_set_kv_length(amk_ctx* ctx, int32_t n);
int32_t amk_kv_length(const amk_ctx* ctx);

/* Wait for the context's stream and report device-side failures. */
amk_status amk_sync(amk_ctx* ctx);

/* Release host state.  Does not free caller memory.  NULL is accepted. */
void amk_free(amk_ctx* ctx);

const char* amk_status_string(amk_status s);
/* Last error message of a context, or of the most recent failing call on this thread when ctx is NULL. */
const char* amk_last_error(const amk_ctx* ctx);

/*
 * Schedule introspection (host only).  amk_build_schedule lowers a config
 * to the task DAG the kernel would run (AMK "Layer 2": a typed Schedule IR;
 * here its counters are fused with the data as version-tagged words, each
 * access naming the version it writes or waits for) and serialises it as
 * int64 words
 * into buf (cap bytes); *needed receives the size.  The format is
 * documented in decode_megakernel_gb300/csrc/schedule.hpp.
 * amk_validate_serialized runs the safety gate on such a buffer (which may
 * come from anywhere) and writes a one-line report; AMK_OK means accepted.
 */
amk_status amk_build_schedule(const amk_config* cfg, const amk_schedule_config* sched,
                              void* buf, size_t cap, size_t* needed);
amk_status amk_validate_serialized(const void* buf, size_t bytes, char* report, size_t cap);

/*
 * The host-side half of amk_load_weights_requeued (host only when
 * sched->num_ctas > 0): checks that the serialised schedule in buf re-queues
 * exactly the tasks of this model's lowering, rebuilds it with the
 * lowering's own accesses and runs the safety gate on it; writes a
 * one-line report.  AMK_OK means amk_load_weights_requeued would accept it.
 */
amk_status amk_validate_requeued(const amk_config* cfg, const amk_schedule_config* sched, const void* buf,
                                 size_t bytes, char* report, size_t cap);

/*
 * Watchdog probe (test aid): launches a small grid of the decode kernel's
 * bounded poll on a tagged word that nothing ever writes, with the given
 * limit, and returns the status the device reported (expected
 * AMK_ERR_TIMEOUT) in *device_status.  scratch_dev: >= 256 bytes of
 * caller device memory.  Nothing hangs: every wait is time bounded.
 */
amk_status amk_debug_watchdog_probe(void* scratch_dev, void* stream, int32_t limit_us,
                                    int32_t* device_status);

/*
 * Per-task timestamps of one decode step (tuning aid, in the spirit of the
 * region timing of the Argus page, "Case 3").  amk_debug_trace_bytes gives
 * the int64 buffer size and, in *stride, the longest task queue S.  The
 * buffer is [num_ctas][1 + S][16]: row 0 of a CTA holds its start and end
 * %globaltimer (ns) and clock64, and its task count; row 1 + i holds, for
 * its i-th task: consumer begin, inputs arrived (thread 0's tagged poll
 * done), work done, outputs stored (%globaltimer ns); producer first and
 * last copy issued (ns) and clock64 cycles blocked on a full ring; task
 * type | layer << 8; consumer clock64 cycles spent waiting for ring data;
 * for attention tasks, the ends of the stage loop and of the warp merge
 * with the partial stored (ns).  Row 0 word 5 holds the CTA's SM id.  amk_debug_trace_step runs
 * amk_decode_step with the recording on and waits for it.  trace_dev:
 * caller device memory, 8-byte aligned.
 */
size_t amk_debug_trace_bytes(const amk_ctx* ctx, int32_t* stride);
amk_status amk_debug_trace_step(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_dev,
                                int64_t* trace_dev, size_t trace_bytes);

/*
 * Dequantisation check (test aid): writes the fp32 values the kernel's
 * weight decoder produces for matrix `lin` of the given format and shape
 * into out_dev [out_features][in_features].  Used to check that int8 / int4
 * decoding is bit exact.
 */
amk_status amk_debug_dequant(int32_t format, const amk_linear* lin, int32_t out_features,
                             int32_t in_features, float* out_dev, void* stream);

/*
 * Read-only HBM stream probe (measurement aid).  The decode step's floor is
 * set by how fast the GPU can stream bytes it only reads (AMK "Problem
 * statement": t_min = weight_bytes / HBM bandwidth); a copy benchmark moves
 * every byte twice and may settle at a different rate.  This launches one
 * pass over buf_dev (bytes: a non-zero multiple of 16384, 16-byte aligned),
 * asynchronously on `stream`, so that the caller can time it with events:
 *   mode 0: one CTA per SM keeps eight 16 KB cp.async.bulk copies in flight
 *           into shared memory (the decode kernel's producer without its
 *           consumers);
 *   mode 1: 128-bit non-caching global loads from four CTAs per SM.
 * out_dev (device, >= 8 * SM-count uint32 words) receives per-CTA checksum
 * and failure words (a nonzero failure word: a copy did not land within
 * 2 s).  Errors: AMK_ERR_INVALID_ARG for a bad mode, size or alignment,
 * AMK_ERR_CUDA for a failed launch.
 */
amk_status amk_debug_hbm_read_probe(int32_t mode, const void* buf_dev, size_t bytes, uint32_t* out_dev,
                                    size_t out_words, void* stream);

#ifdef __cplusplus
}
#endif
#endif
