// Host side of the C ABI declared in include/amk.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/amk.h"
#include "device_model.hpp"
#include "prefill.hpp"
#include "schedule.hpp"

using namespace amk;

// Default ring copies in flight per SM: six 17 KB tiles, 102 KB (plain
// streaming on GB300 peaks at 96-128 KB in flight per SM; 8B bf16 decode
// at 3 / 4 / 5 / 6 / 7 / 8 / 10 / 12 copies: 358.8 / 379.2 / 385.5 / 386.1 /
// 385.7 / 383.8 / 382.1 / 380.6 tok/s, the quantised and 1B workloads
// within 0.3 % from 4 to 12)
constexpr int kDefaultRingSlots = 6;

// Default L2 prefetch budget during the attention chain (tiles of 16 KB).
constexpr int kDefaultPrefetchTiles = 0;

struct amk_ctx {
  amk_config cfg{};
  ModelGeom geom;
  cudaStream_t stream = nullptr;
  int device = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  void* kv = nullptr;
  DevModel dm{};
  const void* kernel = nullptr;
  int smem = 0;
  uint32_t tag_base = 0;  // tag base of the latest launch (see next_tag_base)
  int32_t kv_len = 0;
  float* logits_stage = nullptr;
  uint64_t timeout_ns = 0;
  amk_status poisoned = AMK_OK;
  int32_t max_queue = 0;  // longest per-CTA task queue (trace sizing)
  int32_t n_lm = 0;       // LM-head tasks: argmax pairs per step
  uint32_t* amax[2] = {nullptr, nullptr};  // per-step argmax pairs, double buffered
  // tensor-core prefill (bf16 weights): chunk buffers and tensor maps
  struct Prefill {
    int32_t chunk = 0;        // tokens per chunk; 0: prefill by decode steps
    int32_t parts = kPfDefaultParts;   // bf16 parts of the GEMM activations
    float* x = nullptr;       // residual rows [chunk][hidden]
    uint16_t* h1[kPfParts] = {};  // normed rows, bf16 parts [chunk][hidden]
    uint16_t* h2[kPfParts] = {};  // attention output [chunk][qd] or SwiGLU [chunk][ffn], bf16 parts
    float* q = nullptr;       // rotated queries [chunk][qd]
    int32_t* tokens = nullptr;  // [max_seq]
    CUtensorMap a_h1[kPfParts], a_o[kPfParts], a_a[kPfParts];   // activation operands (parts)
    std::vector<CUtensorMap> w[M_NUM];     // weight operands per layer (QKV, O, gate/up, down)
    int32_t tile_rows = 0;                 // schedule knob: 0 = chosen per matrix
    int32_t bn[M_NUM] = {};                // GEMM tile width per matrix (the weight maps' box rows)
    CUtensorMap kv_attn;                   // the KV cache in boxes of 64 dims x kTcKeys positions
  } pf;
  std::string err;
};

namespace {

thread_local std::string g_last_error;

amk_status fail(amk_ctx* ctx, amk_status st, const std::string& msg) {
  if (ctx) ctx->err = msg;
  g_last_error = msg;
  return st;
}

amk_status cuda_fail(amk_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, AMK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define AMK_CUDA(ctx, call)                                      \
  do {                                                           \
    cudaError_t e_ = (call);                                     \
    if (e_ != cudaSuccess) return cuda_fail((ctx), e_, #call);   \
  } while (0)

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace layout: every region 256-byte aligned.
struct Layout {
  size_t w[M_NUM] = {};
  size_t scales[M_NUM] = {};
  size_t mats = 0, embed = 0, attn_norm = 0, ffn_norm = 0, final_norm = 0, rope = 0;
  size_t xres = 0, xmid = 0, qkv = 0, o = 0, a = 0, part = 0, status = 0, logits = 0, amax = 0;
  size_t tasks = 0, queue_off = 0, queue_body = 0;
  size_t pf_x = 0, pf_h1[kPfParts] = {}, pf_h2[kPfParts] = {}, pf_q = 0, pf_tok = 0;
  size_t total = 0;
};

}  // namespace

namespace amk {

// Per-step scratch regions (256-byte aligned) from one base: tagged x_res,
// x_mid, qkv, o, a, attention partials, then 64 bytes of status words.
StepScratchPlan step_scratch_plan(const ModelGeom& g) {
  const amk_config& c = g.cfg;
  StepScratchPlan plan;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t qd = (size_t)c.n_heads * c.head_dim;
  plan.xres = take((size_t)c.hidden * 4);
  plan.xmid = take((size_t)c.hidden * 4);
  plan.qkv = take((size_t)c.n_kv_heads * (g.group + 2) * c.head_dim * 4);
  plan.o = take(qd * 4);
  plan.a = take((size_t)c.ffn * 4);
  plan.part = take((size_t)c.n_kv_heads * g.splits * g.part_stride * 4);
  plan.status = take(64);
  plan.total = off;
  return plan;
}

}  // namespace amk

namespace {

Layout make_layout(const ModelGeom& g, const Schedule& s) {
  const amk_config& c = g.cfg;
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  for (int k = 0; k < M_NUM; ++k) {
    const int layers = k == M_LM ? 1 : c.n_layers;
    L.w[k] = take((size_t)g.mat[k].bytes * layers);
  }
  for (int k = 0; k < M_NUM; ++k) {
    const int layers = k == M_LM ? 1 : c.n_layers;
    L.scales[k] = g.mat[k].fmt == AMK_FORMAT_INT8 ? take((size_t)g.mat[k].rows_padded * 2 * layers) : 0;
  }
  L.mats = take(sizeof(DevMat) * M_NUM);
  L.embed = take((size_t)c.vocab * c.hidden * 2);
  L.attn_norm = take((size_t)c.n_layers * c.hidden * 2);
  L.ffn_norm = take((size_t)c.n_layers * c.hidden * 2);
  L.final_norm = take((size_t)c.hidden * 2);
  L.rope = take((size_t)c.max_seq * (c.head_dim / 2) * sizeof(float) * 2);
  // per-step scratch (tagged words), then the status words: the same
  // regions in the same order as step_scratch_plan
  StepScratchPlan sp = step_scratch_plan(g);
  const size_t base = take(sp.total);
  L.xres = base + sp.xres;
  L.xmid = base + sp.xmid;
  L.qkv = base + sp.qkv;
  L.o = base + sp.o;
  L.a = base + sp.a;
  L.part = base + sp.part;
  L.status = base + sp.status;
  L.logits = take((size_t)c.vocab * 4);
  L.amax = take((size_t)s.buffers[B_AMAX].size * 4 * 2);
  size_t n_queued = 0;
  for (const auto& q : s.queues) n_queued += q.size();
  L.tasks = take(n_queued * sizeof(DevTask));
  L.queue_off = take((s.queues.size() + 1) * 4);
  L.queue_body = take(s.queues.size() * 4);
  if (g.prefill_chunk > 0) {
    const size_t P = (size_t)g.prefill_chunk, qd = (size_t)c.n_heads * c.head_dim;
    L.pf_x = take(P * c.hidden * 4);
    for (int i = 0; i < kPfParts; ++i) L.pf_h1[i] = take(P * c.hidden * 2);
    for (int i = 0; i < kPfParts; ++i) L.pf_h2[i] = take(P * std::max<size_t>(qd, c.ffn) * 2);
    L.pf_q = take(P * qd * 4);
    L.pf_tok = take((size_t)c.max_seq * 4);
  }
  L.total = off;
  return L;
}

amk_status resolve_ctas(const amk_schedule_config* sched, BuildOptions* opt, std::string* why) {
  *opt = BuildOptions{};
  if (sched) {
    opt->num_ctas = sched->num_ctas;
    opt->attn_splits = sched->attn_splits;
    opt->max_rows_per_task = sched->max_rows_per_task;
    if (sched->num_ctas < 0 || sched->attn_splits < 0 || sched->max_rows_per_task < 0 ||
        sched->watchdog_ms < 0 || sched->ring_slots < 0 || sched->l2_prefetch_tiles < -1 ||
        sched->prefill_chunk < -1 || (sched->prefill_parts != 0 && sched->prefill_parts != 2 &&
                                      sched->prefill_parts != 3) ||
        (sched->prefill_tile_rows != 0 && sched->prefill_tile_rows != kPfBN &&
         sched->prefill_tile_rows != kPfBNNarrow)) {
      *why = "schedule knob out of range";
      return AMK_ERR_INVALID_ARG;
    }
  }
  if (opt->num_ctas == 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      *why = std::string("no CUDA device to size the schedule: ") + cudaGetErrorString(e);
      return AMK_ERR_CUDA;
    }
    opt->num_ctas = sms;
  }
  return AMK_OK;
}

int lm_format(const amk_config& c) { return c.tied_embeddings ? AMK_FORMAT_BF16 : c.lm_head_format; }

// tag_base of a launch: version v of the step carries tag 1 + (tag_base + v - 1) mod kTagPeriod.
// Launch e of a context has tag_base (e * n_layers) mod kTagPeriod, so that
// the tags of consecutive launches continue one another.  The context keeps
// the base itself, advanced modulo kTagPeriod at every launch, rather than
// a launch counter: a counter would wrap after 2^32 launches to a value
// whose base breaks that continuity (2^32 is 1 mod 15), letting a reader
// accept the previous launch's words.
uint32_t next_tag_base(amk_ctx* ctx) {
  ctx->tag_base = (ctx->tag_base + (uint32_t)(ctx->cfg.n_layers % kTagPeriod)) % (uint32_t)kTagPeriod;
  return ctx->tag_base;
}

amk_status plan(const amk_config* cfg, const amk_schedule_config* sched, ModelGeom* g,
                Schedule* s, std::string* why) {
  if (!cfg) {
    *why = "config is NULL";
    return AMK_ERR_INVALID_ARG;
  }
  BuildOptions opt;
  amk_status st = resolve_ctas(sched, &opt, why);
  if (st != AMK_OK) return st;
  st = plan_geometry(*cfg, opt, g, why);
  if (st != AMK_OK) return st;
  // tensor-core prefill: bf16 weights only; chunk rounded up to whole
  // 128-token GEMM tiles and to no more than the cache holds
  {
    const int32_t want = sched ? sched->prefill_chunk : 0;
    g->prefill_chunk = 0;
    if (cfg->weight_format == AMK_FORMAT_BF16 && want >= 0) {
      const int64_t chunk = want > 0 ? want : kPfDefaultChunk;
      const int64_t cap = ((int64_t)cfg->max_seq + kPfBM - 1) / kPfBM * kPfBM;
      g->prefill_chunk = (int32_t)std::min<int64_t>((chunk + kPfBM - 1) / kPfBM * kPfBM, cap);
    }
  }
  if (!decode_kernel_for(cfg->weight_format, lm_format(*cfg))) {
    *why = "no kernel for this weight / LM-head format pair";
    return AMK_ERR_UNSUPPORTED;
  }
  if (s) *s = build_schedule(*g);
  return AMK_OK;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// The KV cache as a 2-D tensor for TMA: rows of head_dim bf16 (one row per
// layer, K/V, KV head and position), boxes of 64 dims x the positions of
// one KV stage, 128-byte swizzle (conflict-free ldmatrix reads).  The
// driver's encoder is reached through the runtime's entry-point query.
// A bf16 tensor map with 128-byte swizzle (rank <= 4; strides of dims
// 1.. in bytes).  The driver's encoder is reached through the runtime's
// entry-point query.
amk_status encode_bf16_map(amk_ctx* ctx, const char* what, CUtensorMap* out, void* base, int rank,
                           const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                CUtensorMapFloatOOBfill);
  static void* fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || !fn || q != cudaDriverEntryPointSuccess) {
      fn = nullptr;
      return fail(ctx, AMK_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    }
  }
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = reinterpret_cast<EncodeFn>(fn)(
      out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, base, dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (%s) failed: %d", what, (int)r);
    return fail(ctx, AMK_ERR_CUDA, buf);
  }
  return AMK_OK;
}

// The KV cache as a 2-D tensor for TMA: rows of head_dim bf16 (one row per
// layer, K/V, KV head and position), boxes of 64 dims x the positions of
// one KV stage, 128-byte swizzle (conflict-free ldmatrix reads).
amk_status encode_kv_map(amk_ctx* ctx, const amk_config& c, void* kv, CUtensorMap* out, int box_rows = 0) {
  const int pps = box_rows > 0 ? box_rows : (kStageBytes / 2) / (c.head_dim * 2);
  const cuuint64_t dims[2] = {(cuuint64_t)c.head_dim,
                              (cuuint64_t)c.n_layers * 2 * c.n_kv_heads * c.max_seq};
  const cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)pps};
  return encode_bf16_map(ctx, "KV cache", out, kv, 2, dims, strides, box);
}

// Tensor maps of the tensor-core prefill.  Activation operands (each of
// the kPfParts bf16 parts): [chunk][K] row major, boxes of 64 k x 128 tokens.  Weight operands: the
// decode kernel's packed tiles of one layer's matrix as a 4-D tensor
// {Kt, Rt, nkt, row blocks}, boxes {64, Rt, 1, bn / Rt}, so that one box
// is a bn-row x 64-k slice in plain row order; bn (256 or 224 rows, both
// multiples of every Rt) per matrix from prefill_gemm_bn for a full chunk
// on this device's SMs.
amk_status encode_prefill_maps(amk_ctx* ctx, const DevMat* mats) {
  const amk_config& c = ctx->cfg;
  auto& pf = ctx->pf;
  const cuuint64_t P = (cuuint64_t)pf.chunk, qd = (cuuint64_t)c.n_heads * c.head_dim;
  auto act = [&](CUtensorMap* m, void* base, cuuint64_t K) {
    const cuuint64_t dims[2] = {K, P};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kPfBK, (cuuint32_t)kPfBM};
    return encode_bf16_map(ctx, "prefill activations", m, base, 2, dims, strides, box);
  };
  for (int i = 0; i < kPfParts; ++i) {
    amk_status st = act(&pf.a_h1[i], pf.h1[i], (cuuint64_t)c.hidden);
    if (st == AMK_OK) st = act(&pf.a_o[i], pf.h2[i], qd);
    if (st == AMK_OK) st = act(&pf.a_a[i], pf.h2[i], (cuuint64_t)c.ffn);
    if (st != AMK_OK) return st;
  }
  if (c.head_dim % 64 == 0) {   // the tensor-core attention's K,V blocks
    amk_status st = encode_kv_map(ctx, c, ctx->kv, &pf.kv_attn, kTcKeys);
    if (st != AMK_OK) return st;
  }
  int sms = 0;
  AMK_CUDA(ctx, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device));
  for (int k : {M_QKV, M_O, M_GU, M_DOWN}) {
    const DevMat& m = mats[k];
    pf.bn[k] = pf.tile_rows ? pf.tile_rows : prefill_gemm_bn(m.rows, pf.chunk, sms);
    if (pf.bn[k] % m.Rt != 0) pf.bn[k] = kPfBN;
    pf.w[k].resize(c.n_layers);
    const cuuint64_t dims[4] = {(cuuint64_t)m.Kt, (cuuint64_t)m.Rt, (cuuint64_t)m.nkt,
                                (cuuint64_t)(m.rows_padded / m.Rt)};
    const cuuint64_t strides[3] = {(cuuint64_t)m.Kt * 2, (cuuint64_t)m.stage_bytes,
                                   (cuuint64_t)m.nkt * m.stage_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)kPfBK, (cuuint32_t)m.Rt, 1, (cuuint32_t)(pf.bn[k] / m.Rt)};
    for (int l = 0; l < c.n_layers; ++l) {
      void* base = const_cast<uint8_t*>(m.base) + (int64_t)l * m.layer_bytes;
      amk_status st = encode_bf16_map(ctx, "prefill weights", &pf.w[k][l], base, 4, dims, strides, box);
      if (st != AMK_OK) return st;
    }
  }
  return AMK_OK;
}

// Bytes of a linear map's tensors in its stored format (amk_linear): codes,
// fp16 scales, packed 4-bit zero points.
struct LinearBytes {
  size_t w = 0, s = 0, z = 0;
};
LinearBytes linear_bytes(int fmt, int64_t rows, int64_t cols) {
  LinearBytes b;
  if (fmt == AMK_FORMAT_BF16) {
    b.w = (size_t)(rows * cols * 2);
  } else if (fmt == AMK_FORMAT_INT8) {
    b.w = (size_t)(rows * cols);
    b.s = (size_t)(rows * 2);
  } else {
    const int64_t ng = cols / 128;
    b.w = (size_t)(rows * cols / 2);
    b.s = (size_t)(rows * ng * 2);
    b.z = (size_t)(rows * ((ng + 1) / 2));
  }
  return b;
}

size_t align256z(size_t v) { return (v + 255) & ~(size_t)255; }

// The linear maps packed together (the groups of launch_pack_matrix), as
// (rows, cols, format) per member; the staging a host-memory load needs is
// the largest group's bytes, each tensor 256-byte aligned.
struct LinearShape {
  int64_t rows, cols;
};
size_t group_staging_bytes(int fmt, std::initializer_list<LinearShape> members) {
  size_t t = 0;
  for (const LinearShape& m : members) {
    const LinearBytes b = linear_bytes(fmt, m.rows, m.cols);
    t += align256z(b.w) + align256z(b.s) + align256z(b.z);
  }
  return t;
}
size_t staging_bytes_of(const amk_config& c) {
  const int64_t H = c.hidden, F = c.ffn, qd = (int64_t)c.n_heads * c.head_dim, kvd = (int64_t)c.n_kv_heads * c.head_dim;
  const int f = c.weight_format;
  size_t m = std::max({group_staging_bytes(f, {{qd, H}, {kvd, H}, {kvd, H}}), group_staging_bytes(f, {{H, qd}}),
                       group_staging_bytes(f, {{F, H}, {F, H}}), group_staging_bytes(f, {{H, F}})});
  if (!c.tied_embeddings) m = std::max(m, group_staging_bytes(lm_format(c), {{c.vocab, H}}));
  return m;
}

// present and aligned for the kernel's vector loads (bf16 rows are read 16
// bytes, int8 rows 8 bytes, int4 rows 4 bytes, fp16 scales 2 bytes at a time)
bool linear_ok(const amk_linear& l, int fmt) {
  if (!l.w) return false;
  if (fmt == AMK_FORMAT_BF16) return aligned(l.w, 16);
  if (fmt == AMK_FORMAT_INT8) return aligned(l.w, 8) && l.scales && aligned(l.scales, 2);
  return aligned(l.w, 4) && l.scales && aligned(l.scales, 2) && l.zeros;
}

// Launch parameters of one step; greedy-decoding and trace fields off.
StepParams make_params(const amk_ctx* ctx, const DevModel& dm, int32_t token, int32_t pos,
                       float* logits, int skip_lm, uint32_t tag_base) {
  StepParams p;
  p.m = dm;
  p.logits = logits;
  p.token = token;
  p.pos = pos;
  p.tag_base = tag_base;
  p.skip_lm = skip_lm;
  p.timeout_ns = ctx->timeout_ns;
  p.trace = nullptr;
  p.trace_stride = 0;
  p.n_lm = ctx->n_lm;
  p.amax = nullptr;
  p.token_src = nullptr;
  p.token_out = nullptr;
  return p;
}

amk_status launch_params(amk_ctx* ctx, StepParams& p) {
  void* args[] = {&p};
  cudaError_t e = cudaLaunchCooperativeKernel(ctx->kernel, dim3(ctx->geom.num_ctas),
                                              dim3(kThreads), args, (size_t)ctx->smem, ctx->stream);
  if (e != cudaSuccess) {
    ctx->poisoned = AMK_ERR_CUDA;
    return cuda_fail(ctx, e, "cudaLaunchCooperativeKernel");
  }
  return AMK_OK;
}

amk_status launch_step(amk_ctx* ctx, int32_t token, int32_t pos, float* logits, int skip_lm) {
  StepParams p = make_params(ctx, ctx->dm, token, pos, logits, skip_lm, next_tag_base(ctx));
  return launch_params(ctx, p);
}

amk_status step_checks(amk_ctx* ctx, int32_t token, int32_t pos) {
  if (!ctx) return fail(nullptr, AMK_ERR_INVALID_ARG, "context is NULL");
  if (ctx->poisoned != AMK_OK) return fail(ctx, ctx->poisoned, "context is poisoned: " + ctx->err);
  if (token < 0 || token >= ctx->cfg.vocab) return fail(ctx, AMK_ERR_INVALID_ARG, "token out of range");
  if (pos < 0 || pos >= ctx->cfg.max_seq) return fail(ctx, AMK_ERR_INVALID_ARG, "pos out of range");
  if (pos > ctx->kv_len)
    return fail(ctx, AMK_ERR_INVALID_ARG, "pos is beyond the valid KV length (positions must be sequential)");
  return AMK_OK;
}

amk_status read_status(amk_ctx* ctx) {
  uint32_t st[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(st, ctx->dm.status, sizeof st, cudaMemcpyDeviceToHost, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) {
    ctx->poisoned = AMK_ERR_CUDA;
    return cuda_fail(ctx, e, "reading the device status");
  }
  if (st[0] == ST_OK) return AMK_OK;
  char buf[160];
  snprintf(buf, sizeof buf, "device %s at CTA %u, task %u, site %u",
           st[0] == ST_TIMEOUT ? "watchdog timeout" : "check failure", st[1], st[2], st[3]);
  ctx->poisoned = st[0] == ST_TIMEOUT ? AMK_ERR_TIMEOUT : AMK_ERR_DEVICE_CHECK;
  return fail(ctx, ctx->poisoned, buf);
}

}  // namespace

// Internal entry points for decode variants that keep a context's weights
// and KV cache but place the per-step scratch somewhere else
// (static_scratch.cu).  They reuse the context's checks and kernel.
namespace amk {

amk_status internal_begin_step(amk_ctx* ctx, int32_t token, int32_t pos, const float* logits,
                               DevModel* dm, StepScratchPlan* plan) {
  amk_status st = step_checks(ctx, token, pos);
  if (st != AMK_OK) return st;
  if (!logits) return fail(ctx, AMK_ERR_INVALID_ARG, "logits pointer is NULL");
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != ctx->device)
    return fail(ctx, AMK_ERR_INVALID_ARG, "the context's device is not the current device");
  *dm = ctx->dm;
  *plan = step_scratch_plan(ctx->geom);
  plan->stream = ctx->stream;
  plan->device = ctx->device;
  return AMK_OK;
}

// A launch on scratch that the caller zeroed: it runs with the tag base of
// a context's first launch (tag 0, which zeroed words carry, is never a
// version's tag).
amk_status internal_launch_fresh(amk_ctx* ctx, const DevModel& dm, int32_t token, int32_t pos,
                                 float* logits) {
  const uint32_t base = (uint32_t)(ctx->cfg.n_layers % kTagPeriod);
  StepParams p = make_params(ctx, dm, token, pos, logits, 0, base);
  return launch_params(ctx, p);
}

amk_status internal_end_step(amk_ctx* ctx, int32_t pos, const uint32_t status[4]) {
  ctx->kv_len = pos + 1;
  if (status[0] == ST_OK) return AMK_OK;
  char buf[160];
  snprintf(buf, sizeof buf, "device %s at CTA %u, task %u, site %u",
           status[0] == ST_TIMEOUT ? "watchdog timeout" : "check failure", status[1], status[2],
           status[3]);
  ctx->poisoned = status[0] == ST_TIMEOUT ? AMK_ERR_TIMEOUT : AMK_ERR_DEVICE_CHECK;
  return fail(ctx, ctx->poisoned, buf);
}

amk_status internal_fail(amk_ctx* ctx, amk_status st, const char* msg) { return fail(ctx, st, msg); }

// A CUDA call of a step failed after its launch: the context is poisoned as
// amk_sync does in that case.
amk_status internal_poison(amk_ctx* ctx, cudaError_t e, const char* what) {
  ctx->poisoned = AMK_ERR_CUDA;
  return cuda_fail(ctx, e, what);
}

}  // namespace amk

extern "C" {

const char* amk_status_string(amk_status s) {
  switch (s) {
    case AMK_OK: return "ok";
    case AMK_ERR_INVALID_ARG: return "invalid argument";
    case AMK_ERR_UNSUPPORTED: return "unsupported model variant";
    case AMK_ERR_SCHEDULE_INVALID: return "schedule rejected by the validator";
    case AMK_ERR_CUDA: return "CUDA error";
    case AMK_ERR_OOM: return "workspace too small";
    case AMK_ERR_TIMEOUT: return "device watchdog timeout";
    case AMK_ERR_DEVICE_CHECK: return "device check failed";
  }
  return "unknown status";
}

const char* amk_last_error(const amk_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_last_error.c_str();
}

amk_status amk_check_config(const amk_config* cfg) {
  if (!cfg) return fail(nullptr, AMK_ERR_INVALID_ARG, "config is NULL");
  ModelGeom g;
  BuildOptions opt;
  opt.num_ctas = 1;
  std::string why;
  amk_status st = plan_geometry(*cfg, opt, &g, &why);
  if (st != AMK_OK) return fail(nullptr, st, why);
  if (!decode_kernel_for(cfg->weight_format, lm_format(*cfg)))
    return fail(nullptr, AMK_ERR_UNSUPPORTED, "no kernel for this weight / LM-head format pair");
  return AMK_OK;
}

size_t amk_kv_cache_bytes(const amk_config* cfg) {
  if (!cfg || cfg->n_layers <= 0 || cfg->n_kv_heads <= 0 || cfg->max_seq <= 0 || cfg->head_dim <= 0)
    return 0;
  return (size_t)cfg->n_layers * 2 * cfg->n_kv_heads * cfg->max_seq * cfg->head_dim * 2;
}

size_t amk_workspace_bytes(const amk_config* cfg, const amk_schedule_config* sched) {
  ModelGeom g;
  Schedule s;
  std::string why;
  if (plan(cfg, sched, &g, &s, &why) != AMK_OK) {
    g_last_error = why;
    return 0;
  }
  return make_layout(g, s).total;
}

amk_status amk_validate_requeued(const amk_config* cfg, const amk_schedule_config* sched, const void* buf,
                                size_t bytes, char* report, size_t cap) {
  auto put = [&](const std::string& m) {
    if (report && cap) {
      size_t n = m.size() < cap - 1 ? m.size() : cap - 1;
      std::memcpy(report, m.data(), n);
      report[n] = 0;
    }
  };
  ModelGeom g;
  Schedule own, given, mine;
  std::string why;
  amk_status st = plan(cfg, sched, &g, &own, &why);
  if (st != AMK_OK) {
    put(why);
    return fail(nullptr, st, why);
  }
  if (!buf || bytes % sizeof(int64_t) ||
      !deserialize(static_cast<const int64_t*>(buf), bytes / sizeof(int64_t), &given, &why)) {
    why = "malformed schedule: " + (why.empty() ? std::string("buffer is NULL or not whole int64 words") : why);
    put(why);
    return fail(nullptr, AMK_ERR_SCHEDULE_INVALID, why);
  }
  if (!requeue(own, given, &mine, &why)) {
    why = "schedule does not re-queue this model's tasks: " + why;
    put(why);
    return fail(nullptr, AMK_ERR_SCHEDULE_INVALID, why);
  }
  Report r = validate(mine);
  put(r.msg);
  if (!r.ok) return fail(nullptr, AMK_ERR_SCHEDULE_INVALID, r.msg);
  return AMK_OK;
}

amk_status amk_build_schedule(const amk_config* cfg, const amk_schedule_config* sched, void* buf,
                              size_t cap, size_t* needed) {
  ModelGeom g;
  Schedule s;
  std::string why;
  amk_status st = plan(cfg, sched, &g, &s, &why);
  if (st != AMK_OK) return fail(nullptr, st, why);
  std::vector<int64_t> words = serialize(s);
  const size_t bytes = words.size() * sizeof(int64_t);
  if (needed) *needed = bytes;
  if (!buf) return AMK_OK;
  if (cap < bytes) return fail(nullptr, AMK_ERR_INVALID_ARG, "buffer too small for the schedule");
  std::memcpy(buf, words.data(), bytes);
  return AMK_OK;
}

amk_status amk_validate_serialized(const void* buf, size_t bytes, char* report, size_t cap) {
  auto put = [&](const std::string& m) {
    if (report && cap) {
      size_t n = m.size() < cap - 1 ? m.size() : cap - 1;
      std::memcpy(report, m.data(), n);
      report[n] = 0;
    }
  };
  if (!buf || bytes % sizeof(int64_t)) {
    put("buffer is NULL or not whole int64 words");
    return fail(nullptr, AMK_ERR_INVALID_ARG, "bad serialised schedule buffer");
  }
  Schedule s;
  std::string why;
  if (!deserialize(static_cast<const int64_t*>(buf), bytes / sizeof(int64_t), &s, &why)) {
    put("malformed: " + why);
    return fail(nullptr, AMK_ERR_SCHEDULE_INVALID, why);
  }
  Report r = validate(s);
  put(r.msg);
  if (!r.ok) return fail(nullptr, AMK_ERR_SCHEDULE_INVALID, r.msg);
  return AMK_OK;
}

}  // extern "C"

namespace {

// amk_load_weights, optionally with the lowering's tasks re-queued as a
// given serialised schedule assigns them (amk_load_weights_requeued)
// staging != NULL: the weights are in host memory; each group of matrices
// is copied into the staging buffer and repacked from there (the device
// never holds the caller's copy of the model).
amk_status load_impl(const amk_config* cfg, const amk_weights* weights, void* workspace_dev,
                     size_t workspace_bytes, void* kv_cache_dev, void* stream,
                     const amk_schedule_config* sched, const void* requeue_buf, size_t requeue_bytes,
                     amk_ctx** out, void* staging = nullptr, size_t staging_bytes = 0) {
  if (!out) return fail(nullptr, AMK_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg || !weights || !workspace_dev || !kv_cache_dev)
    return fail(nullptr, AMK_ERR_INVALID_ARG, "NULL config, weights, workspace or KV cache");
  if (((uintptr_t)workspace_dev & 255) || ((uintptr_t)kv_cache_dev & 15))
    return fail(nullptr, AMK_ERR_INVALID_ARG, "workspace must be 256-byte and KV cache 16-byte aligned");

  amk_ctx* ctx = new (std::nothrow) amk_ctx;
  if (!ctx) return fail(nullptr, AMK_ERR_OOM, "host allocation failed");
  auto bail = [&](amk_status st) {
    g_last_error = ctx->err;
    delete ctx;
    return st;
  };

  Schedule s;
  std::string why;
  amk_status st = plan(cfg, sched, &ctx->geom, &s, &why);
  if (st != AMK_OK) return bail(fail(ctx, st, why));
  const amk_config& c = *cfg;
  const ModelGeom& g = ctx->geom;
  if (requeue_buf) {
    Schedule given, mine;
    if (requeue_bytes % sizeof(int64_t) ||
        !deserialize(static_cast<const int64_t*>(requeue_buf), requeue_bytes / sizeof(int64_t), &given, &why))
      return bail(fail(ctx, AMK_ERR_SCHEDULE_INVALID, "malformed schedule: " + why));
    if (!requeue(s, given, &mine, &why))
      return bail(fail(ctx, AMK_ERR_SCHEDULE_INVALID, "schedule does not re-queue this model's tasks: " + why));
    s = std::move(mine);
  }

  // the safety gate: nothing is launched for a schedule that fails it
  Report rep = validate(s);
  if (!rep.ok) return bail(fail(ctx, AMK_ERR_SCHEDULE_INVALID, "schedule rejected: " + rep.msg));

  // weights present for every matrix (device pointers also aligned for the
  // pack kernels' vector loads; host pointers are copied to aligned staging)
  const int lmf = lm_format(c);
  const bool host = staging != nullptr;
  auto lin_ok = [&](const amk_linear& l, int fmt) {
    if (!host) return linear_ok(l, fmt);
    return l.w && (fmt == AMK_FORMAT_BF16 || l.scales) && (fmt != AMK_FORMAT_INT4 || l.zeros);
  };
  if (host && (((uintptr_t)staging & 255) || staging_bytes < staging_bytes_of(c)))
    return bail(fail(ctx, AMK_ERR_INVALID_ARG, "staging buffer misaligned or smaller than amk_weights_staging_bytes"));
  if (!weights->embed || !weights->final_norm || !weights->layers ||
      (!host && (!aligned(weights->embed, 16) || !aligned(weights->final_norm, 2))))
    return bail(fail(ctx, AMK_ERR_INVALID_ARG, "missing or misaligned embedding, final norm or layer table"));
  if (!c.tied_embeddings && !lin_ok(weights->lm_head, lmf))
    return bail(fail(ctx, AMK_ERR_INVALID_ARG, "missing LM-head weights"));
  for (int l = 0; l < c.n_layers; ++l) {
    const amk_layer_weights& lw = weights->layers[l];
    if (!lw.attn_norm || !lw.ffn_norm || (!host && (!aligned(lw.attn_norm, 2) || !aligned(lw.ffn_norm, 2))))
      return bail(fail(ctx, AMK_ERR_INVALID_ARG, "missing or misaligned norm weights"));
    for (const amk_linear* lin : {&lw.wq, &lw.wk, &lw.wv, &lw.wo, &lw.wg, &lw.wu, &lw.wd})
      if (!lin_ok(*lin, c.weight_format))
        return bail(fail(ctx, AMK_ERR_INVALID_ARG, "missing or misaligned linear weights / scales / zeros"));
  }

  Layout L = make_layout(g, s);
  if (workspace_bytes < L.total) {
    char buf[128];
    snprintf(buf, sizeof buf, "workspace has %zu bytes, needs %zu", workspace_bytes, L.total);
    return bail(fail(ctx, AMK_ERR_OOM, buf));
  }

  ctx->cfg = c;
  ctx->stream = (cudaStream_t)stream;
  ctx->ws = (uint8_t*)workspace_dev;
  ctx->ws_bytes = workspace_bytes;
  ctx->kv = kv_cache_dev;
  ctx->timeout_ns = (uint64_t)(sched && sched->watchdog_ms > 0 ? sched->watchdog_ms : 2000) * 1000000ull;
  if (cudaGetDevice(&ctx->device) != cudaSuccess) return bail(fail(ctx, AMK_ERR_CUDA, "cudaGetDevice failed"));

  // kernel and co-residency of one CTA per SM
  ctx->kernel = decode_kernel_for(c.weight_format, lmf);
  ctx->smem = decode_smem_bytes();
  {
    cudaError_t e = cudaFuncSetAttribute(ctx->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ctx->smem);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "cudaFuncSetAttribute"));
    int per_sm = 0, sms = 0, coop = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ctx->kernel, kThreads, ctx->smem);
    if (e != cudaSuccess) return bail(cuda_fail(ctx, e, "occupancy query"));
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, ctx->device);
    if (!coop) return bail(fail(ctx, AMK_ERR_UNSUPPORTED, "device lacks cooperative launch"));
    if (per_sm < 1 || g.num_ctas > per_sm * sms)
      return bail(fail(ctx, AMK_ERR_UNSUPPORTED, "num_ctas exceeds co-resident CTAs"));
  }

  // device model
  uint8_t* ws = ctx->ws;
  DevMat mats[M_NUM];
  for (int k = 0; k < M_NUM; ++k) {
    const MatGeom& m = g.mat[k];
    DevMat& d = mats[k];
    d.base = ws + L.w[k];
    d.scales = L.scales[k] ? (const uint16_t*)(ws + L.scales[k]) : nullptr;
    d.layer_bytes = m.bytes;
    d.rb_bytes = m.rb_bytes;
    d.stage_bytes = (int32_t)(m.tile_bytes + m.side_bytes);
    d.fmt = m.fmt;
    d.rows = m.rows;
    d.rows_padded = m.rows_padded;
    d.K = m.K;
    d.Kp = m.Kp;
    d.Kt = m.Kt;
    d.nkt = m.nkt;
    d.Rt = m.Rt;
    d.cpr_shift = m.cpr_shift;
  }
  DevModel& dm = ctx->dm;
  dm.mat = (const DevMat*)(ws + L.mats);
  dm.n_layers = c.n_layers;
  dm.hidden = c.hidden;
  dm.n_heads = c.n_heads;
  dm.n_kv_heads = c.n_kv_heads;
  dm.head_dim = c.head_dim;
  dm.ffn = c.ffn;
  dm.vocab = c.vocab;
  dm.max_seq = c.max_seq;
  dm.group = g.group;
  dm.splits = g.splits;
  dm.part_stride = g.part_stride;
  dm.num_ctas = g.num_ctas;
  dm.rms_eps = c.rms_eps;
  dm.ring_slots = sched && sched->ring_slots > 0 ? std::min<int32_t>(sched->ring_slots, kRingSlots)
                                                 : kDefaultRingSlots;
  dm.prefetch_tiles = !sched || sched->l2_prefetch_tiles == 0 ? kDefaultPrefetchTiles
                      : sched->l2_prefetch_tiles < 0          ? 0
                                                              : std::min(sched->l2_prefetch_tiles, 1024);
  dm.pad0 = 0;
  dm.embed = (const uint16_t*)(ws + L.embed);
  dm.final_norm = (const uint16_t*)(ws + L.final_norm);
  dm.attn_norm = (const uint16_t*)(ws + L.attn_norm);
  dm.ffn_norm = (const uint16_t*)(ws + L.ffn_norm);
  dm.rope = (const float2*)(ws + L.rope);
  dm.kv = (uint16_t*)kv_cache_dev;
  dm.xres = (uint32_t*)(ws + L.xres);
  dm.xmid = (uint32_t*)(ws + L.xmid);
  dm.qkv = (uint32_t*)(ws + L.qkv);
  dm.o = (uint32_t*)(ws + L.o);
  dm.a = (uint32_t*)(ws + L.a);
  dm.part = (uint32_t*)(ws + L.part);
  dm.status = (uint32_t*)(ws + L.status);
  dm.tasks = (const DevTask*)(ws + L.tasks);
  dm.queue_off = (const int32_t*)(ws + L.queue_off);
  dm.queue_body = (const int32_t*)(ws + L.queue_body);
  {
    amk_status kst = encode_kv_map(ctx, c, kv_cache_dev, &dm.kv_map);
    if (kst != AMK_OK) return bail(kst);
  }
  ctx->logits_stage = (float*)(ws + L.logits);

  // task table, queue order per CTA
  std::vector<DevTask> tasks;
  std::vector<int32_t> qoff(s.queues.size() + 1, 0), qbody(s.queues.size(), 0);
  for (size_t q = 0; q < s.queues.size(); ++q) {
    qoff[q] = (int32_t)tasks.size();
    qbody[q] = s.body_len[q];
    for (int32_t id : s.queues[q]) {
      const Task& t = s.tasks[id];
      DevTask d{};
      d.type = (int16_t)t.type;
      d.layer = (int16_t)t.layer;
      d.a0 = (int32_t)t.a[0];
      d.a1 = (int32_t)t.a[1];
      d.a2 = (int32_t)t.a[2];
      d.a3 = (int32_t)t.a[3];
      tasks.push_back(d);
    }
  }
  qoff[s.queues.size()] = (int32_t)tasks.size();
  for (const auto& q : s.queues) ctx->max_queue = std::max<int32_t>(ctx->max_queue, (int32_t)q.size());
  ctx->n_lm = (int32_t)(s.buffers[B_AMAX].size / 2);
  ctx->amax[0] = (uint32_t*)(ws + L.amax);
  ctx->amax[1] = ctx->amax[0] + 2 * ctx->n_lm;

  // rotate-half RoPE table, computed in double and rounded to float
  const int half = c.head_dim / 2;
  std::vector<float> rope((size_t)c.max_seq * half * 2);
  for (int pos = 0; pos < c.max_seq; ++pos)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)pos * std::pow((double)c.rope_theta, -2.0 * i / c.head_dim);
      rope[((size_t)pos * half + i) * 2 + 0] = (float)std::cos(ang);
      rope[((size_t)pos * half + i) * 2 + 1] = (float)std::sin(ang);
    }

  cudaStream_t st_ = ctx->stream;
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.mats, mats, sizeof mats, cudaMemcpyHostToDevice, st_));
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.tasks, tasks.data(), tasks.size() * sizeof(DevTask),
                                cudaMemcpyHostToDevice, st_));
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.queue_off, qoff.data(), qoff.size() * 4, cudaMemcpyHostToDevice, st_));
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.queue_body, qbody.data(), qbody.size() * 4, cudaMemcpyHostToDevice, st_));
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.rope, rope.data(), rope.size() * 4, cudaMemcpyHostToDevice, st_));
  // tagged scratch and status start zeroed: tag 0 is never a version's tag
  AMK_CUDA(ctx, cudaMemsetAsync(ws + L.xres, 0, L.status + 64 - L.xres, st_));

  // weights: embedding (row major copy), norms, tiled matrices.  Copies
  // take the direction from the pointers (host or device memory); with
  // host weights each group of matrices goes through the staging buffer,
  // whose next fill is ordered on the stream after the pack that read it.
  const size_t H2 = (size_t)c.hidden * 2;
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.embed, weights->embed, (size_t)c.vocab * H2, cudaMemcpyDefault, st_));
  AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.final_norm, weights->final_norm, H2, cudaMemcpyDefault, st_));
  const int64_t qd = (int64_t)c.n_heads * c.head_dim, kvd = (int64_t)c.n_kv_heads * c.head_dim;
  // the group's linears with device pointers: the caller's, or copies in staging
  auto staged = [&](int fmt, std::initializer_list<std::pair<const amk_linear*, LinearShape>> members,
                    amk_linear* dst) -> amk_status {
    size_t off = 0;
    int i = 0;
    for (const auto& mb : members) {
      dst[i] = *mb.first;
      if (host) {
        const LinearBytes b = linear_bytes(fmt, mb.second.rows, mb.second.cols);
        uint8_t* base = (uint8_t*)staging;
        AMK_CUDA(ctx, cudaMemcpyAsync(base + off, mb.first->w, b.w, cudaMemcpyDefault, st_));
        dst[i].w = base + off;
        off += align256z(b.w);
        if (b.s) {
          AMK_CUDA(ctx, cudaMemcpyAsync(base + off, mb.first->scales, b.s, cudaMemcpyDefault, st_));
          dst[i].scales = base + off;
          off += align256z(b.s);
        }
        if (b.z) {
          AMK_CUDA(ctx, cudaMemcpyAsync(base + off, mb.first->zeros, b.z, cudaMemcpyDefault, st_));
          dst[i].zeros = base + off;
          off += align256z(b.z);
        }
      }
      ++i;
    }
    return AMK_OK;
  };
  const int64_t Hh = c.hidden, Ff = c.ffn;
  for (int l = 0; l < c.n_layers; ++l) {
    const amk_layer_weights& lw = weights->layers[l];
    const int f = c.weight_format;
    amk_linear d[3];
    AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.attn_norm + l * H2, lw.attn_norm, H2, cudaMemcpyDefault, st_));
    AMK_CUDA(ctx, cudaMemcpyAsync(ws + L.ffn_norm + l * H2, lw.ffn_norm, H2, cudaMemcpyDefault, st_));
    if ((st = staged(f, {{&lw.wq, {qd, Hh}}, {&lw.wk, {kvd, Hh}}, {&lw.wv, {kvd, Hh}}}, d)) != AMK_OK) return bail(st);
    launch_pack_matrix(M_QKV, f, mats[M_QKV], l, d[0].w, d[0].scales, d[0].zeros, d[1].w, d[1].scales, d[1].zeros,
                       d[2].w, d[2].scales, d[2].zeros, c.n_heads, c.n_kv_heads, c.head_dim, st_);
    if ((st = staged(f, {{&lw.wo, {Hh, qd}}}, d)) != AMK_OK) return bail(st);
    launch_pack_matrix(M_O, f, mats[M_O], l, d[0].w, d[0].scales, d[0].zeros, nullptr, nullptr, nullptr, nullptr,
                       nullptr, nullptr, c.n_heads, c.n_kv_heads, c.head_dim, st_);
    if ((st = staged(f, {{&lw.wg, {Ff, Hh}}, {&lw.wu, {Ff, Hh}}}, d)) != AMK_OK) return bail(st);
    launch_pack_matrix(M_GU, f, mats[M_GU], l, d[0].w, d[0].scales, d[0].zeros, d[1].w, d[1].scales, d[1].zeros,
                       nullptr, nullptr, nullptr, c.n_heads, c.n_kv_heads, c.head_dim, st_);
    if ((st = staged(f, {{&lw.wd, {Hh, Ff}}}, d)) != AMK_OK) return bail(st);
    launch_pack_matrix(M_DOWN, f, mats[M_DOWN], l, d[0].w, d[0].scales, d[0].zeros, nullptr, nullptr, nullptr,
                       nullptr, nullptr, nullptr, c.n_heads, c.n_kv_heads, c.head_dim, st_);
    AMK_CUDA(ctx, cudaGetLastError());
  }
  if (c.tied_embeddings) {   // from the workspace's row-major copy of the embedding
    launch_pack_matrix(M_LM, AMK_FORMAT_BF16, mats[M_LM], 0, ws + L.embed, nullptr, nullptr,
                       nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, c.n_heads,
                       c.n_kv_heads, c.head_dim, st_);
  } else {
    amk_linear d[1];
    if ((st = staged(lmf, {{&weights->lm_head, {(int64_t)c.vocab, Hh}}}, d)) != AMK_OK) return bail(st);
    launch_pack_matrix(M_LM, lmf, mats[M_LM], 0, d[0].w, d[0].scales, d[0].zeros, nullptr, nullptr, nullptr,
                       nullptr, nullptr, nullptr, c.n_heads, c.n_kv_heads, c.head_dim, st_);
  }
  AMK_CUDA(ctx, cudaGetLastError());
  if (g.prefill_chunk > 0) {
    auto& pf = ctx->pf;
    pf.chunk = g.prefill_chunk;
    pf.parts = sched && sched->prefill_parts ? sched->prefill_parts : kPfDefaultParts;
    pf.tile_rows = sched ? sched->prefill_tile_rows : 0;
    pf.x = (float*)(ws + L.pf_x);
    for (int i = 0; i < kPfParts; ++i) {
      pf.h1[i] = (uint16_t*)(ws + L.pf_h1[i]);
      pf.h2[i] = (uint16_t*)(ws + L.pf_h2[i]);
    }
    pf.q = (float*)(ws + L.pf_q);
    pf.tokens = (int32_t*)(ws + L.pf_tok);
    amk_status pst = encode_prefill_maps(ctx, mats);
    if (pst != AMK_OK) return bail(pst);
  }
  AMK_CUDA(ctx, cudaStreamSynchronize(st_));
  ctx->kv_len = 0;
  *out = ctx;
  return AMK_OK;
}

}  // namespace

extern "C" {

amk_status amk_load_weights(const amk_config* cfg, const amk_weights* weights, void* workspace_dev,
                            size_t workspace_bytes, void* kv_cache_dev, void* stream,
                            const amk_schedule_config* sched, amk_ctx** out) {
  return load_impl(cfg, weights, workspace_dev, workspace_bytes, kv_cache_dev, stream, sched, nullptr, 0, out);
}

size_t amk_weights_staging_bytes(const amk_config* cfg) {
  if (!cfg || amk_check_config(cfg) != AMK_OK) return 0;
  return staging_bytes_of(*cfg);
}

amk_status amk_load_weights_staged(const amk_config* cfg, const amk_weights* host_weights, void* workspace_dev,
                                   size_t workspace_bytes, void* kv_cache_dev, void* stream,
                                   const amk_schedule_config* sched, void* staging_dev, size_t staging_bytes,
                                   amk_ctx** out) {
  if (!staging_dev) {
    if (out) *out = nullptr;
    return fail(nullptr, AMK_ERR_INVALID_ARG, "staging buffer is NULL");
  }
  return load_impl(cfg, host_weights, workspace_dev, workspace_bytes, kv_cache_dev, stream, sched, nullptr, 0, out,
                   staging_dev, staging_bytes);
}

amk_status amk_load_weights_requeued(const amk_config* cfg, const amk_weights* weights, void* workspace_dev,
                                     size_t workspace_bytes, void* kv_cache_dev, void* stream,
                                     const amk_schedule_config* sched, const void* schedule,
                                     size_t schedule_bytes, amk_ctx** out) {
  if (!schedule) {
    if (out) *out = nullptr;
    return fail(nullptr, AMK_ERR_INVALID_ARG, "schedule is NULL");
  }
  return load_impl(cfg, weights, workspace_dev, workspace_bytes, kv_cache_dev, stream, sched, schedule,
                   schedule_bytes, out);
}

namespace {

// The tensor-core prefill of tokens (already on the device) at positions
// start_pos .. start_pos + n - 1, chunk by chunk, layer by layer.
amk_status prefill_tensor_cores(amk_ctx* ctx, int32_t n, int32_t start_pos) {
  const amk_config& c = ctx->cfg;
  const ModelGeom& geo = ctx->geom;
  auto& pf = ctx->pf;
  const DevModel& dm = ctx->dm;
  cudaStream_t s = ctx->stream;
  const int qd = c.n_heads * c.head_dim;
  const size_t H = (size_t)c.hidden;
  PrefillGemm g{};
  g.hd = c.head_dim;
  g.group = geo.group;
  g.n_kv = c.n_kv_heads;
  g.max_seq = c.max_seq;
  g.x = pf.x;
  g.ldx = c.hidden;
  g.q = pf.q;
  g.ldq = qd;
  g.kv = dm.kv;
  g.rope = dm.rope;
  for (int i = 0; i < kPfParts; ++i) g.out[i] = pf.h2[i];
  g.ldo = c.ffn;
  g.parts = pf.parts;
  g.status = dm.status;
  g.timeout_ns = ctx->timeout_ns;
  {
    int sms = 0;
    AMK_CUDA(ctx, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device));
    g.ctas = sms;
  }
  PrefillAttn at{};
  at.q = pf.q;
  at.ldq = qd;
  at.kv = dm.kv;
  at.n_kv = c.n_kv_heads;
  at.max_seq = c.max_seq;
  at.group = geo.group;
  at.hd = c.head_dim;
  for (int i = 0; i < kPfParts; ++i) at.o[i] = pf.h2[i];
  at.ldo = qd;
  at.parts = pf.parts;
  at.status = dm.status;
  at.timeout_ns = ctx->timeout_ns;
  const CUtensorMap* kv_attn = c.head_dim % 64 == 0 ? &pf.kv_attn : nullptr;
  auto gemm = [&](int epi, int kind, int layer, const CUtensorMap* a) {
    const MatGeom& m = geo.mat[kind];
    g.N = m.rows;
    g.nk = m.Kp / kPfBK;
    g.Kt = m.Kt;
    g.Rt = m.Rt;
    g.layer = layer;
    return launch_prefill_gemm(epi, a, &pf.w[kind][layer], pf.bn[kind], g, s);
  };
  for (int32_t c0 = 0; c0 < n; c0 += pf.chunk) {
    const int T = std::min<int32_t>(pf.chunk, n - c0);
    g.T = at.T = T;
    g.s0 = at.s0 = start_pos + c0;
    AMK_CUDA(ctx, launch_prefill_embed(pf.tokens + c0, T, dm.embed, c.hidden, pf.x, s));
    for (int l = 0; l < c.n_layers; ++l) {
      AMK_CUDA(ctx, launch_prefill_norm(pf.x, T, c.hidden, dm.attn_norm + l * H, c.rms_eps, pf.h1, pf.parts, s));
      AMK_CUDA(ctx, gemm(PE_QKV, M_QKV, l, pf.a_h1));
      if (l == c.n_layers - 1) break;   // the rest of the last layer feeds no K,V
      at.layer = l;
      AMK_CUDA(ctx, launch_prefill_attn(at, kv_attn, s));
      AMK_CUDA(ctx, gemm(PE_RESID, M_O, l, pf.a_o));
      AMK_CUDA(ctx, launch_prefill_norm(pf.x, T, c.hidden, dm.ffn_norm + l * H, c.rms_eps, pf.h1, pf.parts, s));
      AMK_CUDA(ctx, gemm(PE_SWIGLU, M_GU, l, pf.a_h1));
      AMK_CUDA(ctx, gemm(PE_RESID, M_DOWN, l, pf.a_a));
    }
  }
  return AMK_OK;
}

}  // namespace

amk_status amk_prefill(amk_ctx* ctx, const int32_t* host_tokens, int32_t n, int32_t start_pos) {
  if (!ctx) return fail(nullptr, AMK_ERR_INVALID_ARG, "context is NULL");
  if (n < 0 || (n > 0 && !host_tokens)) return fail(ctx, AMK_ERR_INVALID_ARG, "bad token array");
  if (start_pos < 0 || (int64_t)start_pos + n > ctx->cfg.max_seq)
    return fail(ctx, AMK_ERR_INVALID_ARG, "prefill runs past max_seq");
  if (ctx->pf.chunk > 0 && n > 0) {
    amk_status st = step_checks(ctx, host_tokens[0], start_pos);
    if (st != AMK_OK) return st;
    for (int32_t i = 0; i < n; ++i)
      if (host_tokens[i] < 0 || host_tokens[i] >= ctx->cfg.vocab)
        return fail(ctx, AMK_ERR_INVALID_ARG, "token out of range");
    AMK_CUDA(ctx, cudaMemcpyAsync(ctx->pf.tokens, host_tokens, (size_t)n * 4, cudaMemcpyHostToDevice,
                                  ctx->stream));
    st = prefill_tensor_cores(ctx, n, start_pos);
    if (st != AMK_OK) return st;
    ctx->kv_len = start_pos + n;
    return AMK_OK;
  }
  for (int32_t i = 0; i < n; ++i) {
    amk_status st = step_checks(ctx, host_tokens[i], start_pos + i);
    if (st != AMK_OK) return st;
    st = launch_step(ctx, host_tokens[i], start_pos + i, nullptr, 1);
    if (st != AMK_OK) return st;
    ctx->kv_len = start_pos + i + 1;
  }
  return AMK_OK;
}

amk_status amk_decode_step(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_dev) {
  amk_status st = step_checks(ctx, token, pos);
  if (st != AMK_OK) return st;
  if (!logits_dev) return fail(ctx, AMK_ERR_INVALID_ARG, "logits pointer is NULL");
  st = launch_step(ctx, token, pos, logits_dev, 0);
  if (st == AMK_OK) ctx->kv_len = pos + 1;
  return st;
}

amk_status amk_decode_step_host(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_host) {
  amk_status st = step_checks(ctx, token, pos);
  if (st != AMK_OK) return st;
  if (!logits_host) return fail(ctx, AMK_ERR_INVALID_ARG, "logits pointer is NULL");
  st = launch_step(ctx, token, pos, ctx->logits_stage, 0);
  if (st != AMK_OK) return st;
  ctx->kv_len = pos + 1;
  cudaError_t e = cudaMemcpyAsync(logits_host, ctx->logits_stage, (size_t)ctx->cfg.vocab * 4,
                                  cudaMemcpyDeviceToHost, ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "logits copy");
  return amk_sync(ctx);
}

amk_status amk_generate(amk_ctx* ctx, int32_t first_token, int32_t pos, int32_t n_steps,
                        int32_t* tokens_dev, float* logits_dev) {
  amk_status st = step_checks(ctx, first_token, pos);
  if (st != AMK_OK) return st;
  if (n_steps < 1 || (int64_t)pos + n_steps > ctx->cfg.max_seq)
    return fail(ctx, AMK_ERR_INVALID_ARG, "n_steps must be >= 1 and pos + n_steps <= max_seq");
  if (!tokens_dev || ((uintptr_t)tokens_dev & 3) || (logits_dev && ((uintptr_t)logits_dev & 3)))
    return fail(ctx, AMK_ERR_INVALID_ARG, "tokens_dev NULL or misaligned, or logits_dev misaligned");
  float* logits = logits_dev ? logits_dev : ctx->logits_stage;
  for (int32_t i = 0; i < n_steps; ++i) {
    StepParams p = make_params(ctx, ctx->dm, first_token, pos + i, logits, 0, next_tag_base(ctx));
    p.amax = ctx->amax[i & 1];
    if (i > 0) {
      p.token_src = ctx->amax[(i - 1) & 1];
      p.token_out = tokens_dev + (i - 1);
    }
    st = launch_params(ctx, p);
    if (st != AMK_OK) return st;
    ctx->kv_len = pos + i + 1;
  }
  launch_argmax_pairs(ctx->amax[(n_steps - 1) & 1], ctx->n_lm, tokens_dev + (n_steps - 1), ctx->stream);
  AMK_CUDA(ctx, cudaGetLastError());
  return AMK_OK;
}

amk_status amk_set_kv_length(amk_ctx* ctx, int32_t n) {
  if (!ctx) return fail(nullptr, AMK_ERR_INVALID_ARG, "context is NULL");
  if (n < 0 || n > ctx->cfg.max_seq) return fail(ctx, AMK_ERR_INVALID_ARG, "KV length out of range");
  ctx->kv_len = n;
  return AMK_OK;
}

int32_t amk_prefill_chunk(const amk_ctx* ctx) { return ctx ? ctx->pf.chunk : -1; }

int32_t amk_kv_length(const amk_ctx* ctx) { return ctx ? ctx->kv_len : -1; }

amk_status amk_sync(amk_ctx* ctx) {
  if (!ctx) return fail(nullptr, AMK_ERR_INVALID_ARG, "context is NULL");
  if (ctx->poisoned != AMK_OK) return fail(ctx, ctx->poisoned, ctx->err);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) {
    ctx->poisoned = AMK_ERR_CUDA;
    return cuda_fail(ctx, e, "cudaStreamSynchronize");
  }
  return read_status(ctx);
}

void amk_free(amk_ctx* ctx) { delete ctx; }

size_t amk_debug_trace_bytes(const amk_ctx* ctx, int32_t* stride) {
  if (!ctx) return 0;
  if (stride) *stride = ctx->max_queue;
  return (size_t)ctx->geom.num_ctas * (1 + (size_t)ctx->max_queue) * kTraceWords * sizeof(int64_t);
}

amk_status amk_debug_trace_step(amk_ctx* ctx, int32_t token, int32_t pos, float* logits_dev,
                                int64_t* trace_dev, size_t trace_bytes) {
  amk_status st = step_checks(ctx, token, pos);
  if (st != AMK_OK) return st;
  if (!logits_dev || !trace_dev || ((uintptr_t)trace_dev & 7) ||
      trace_bytes < amk_debug_trace_bytes(ctx, nullptr))
    return fail(ctx, AMK_ERR_INVALID_ARG, "bad logits or trace buffer (see amk_debug_trace_bytes)");
  AMK_CUDA(ctx, cudaMemsetAsync(trace_dev, 0, amk_debug_trace_bytes(ctx, nullptr), ctx->stream));
  StepParams p = make_params(ctx, ctx->dm, token, pos, logits_dev, 0, next_tag_base(ctx));
  p.trace = trace_dev;
  p.trace_stride = ctx->max_queue;
  st = launch_params(ctx, p);
  if (st != AMK_OK) return st;
  ctx->kv_len = pos + 1;
  return amk_sync(ctx);
}

amk_status amk_debug_watchdog_probe(void* scratch_dev, void* stream, int32_t limit_us,
                                    int32_t* device_status) {
  if (!scratch_dev || !device_status || limit_us <= 0 || limit_us > 10000000)
    return fail(nullptr, AMK_ERR_INVALID_ARG, "bad watchdog probe arguments");
  cudaStream_t s = (cudaStream_t)stream;
  AMK_CUDA(nullptr, cudaMemsetAsync(scratch_dev, 0, 256, s));
  launch_watchdog_probe((uint32_t*)scratch_dev, (uint64_t)limit_us * 1000ull, stream);
  AMK_CUDA(nullptr, cudaGetLastError());
  uint32_t st[4];
  AMK_CUDA(nullptr, cudaMemcpyAsync(st, (uint32_t*)scratch_dev + 16, sizeof st, cudaMemcpyDeviceToHost, s));
  AMK_CUDA(nullptr, cudaStreamSynchronize(s));
  *device_status = st[0] == ST_OK ? AMK_OK : st[0] == ST_TIMEOUT ? AMK_ERR_TIMEOUT : AMK_ERR_DEVICE_CHECK;
  return AMK_OK;
}

amk_status amk_debug_dequant(int32_t format, const amk_linear* lin, int32_t out_features,
                             int32_t in_features, float* out_dev, void* stream) {
  if (!lin || !out_dev || out_features <= 0 || in_features <= 0 || in_features % 8 ||
      !aligned(out_dev, 4))
    return fail(nullptr, AMK_ERR_INVALID_ARG, "bad dequant arguments");
  if (format < AMK_FORMAT_BF16 || format > AMK_FORMAT_INT4 || !linear_ok(*lin, format))
    return fail(nullptr, AMK_ERR_INVALID_ARG, "bad format or missing scales / zeros");
  if (format == AMK_FORMAT_INT4 && in_features % 128)
    return fail(nullptr, AMK_ERR_UNSUPPORTED, "int4 needs in_features % 128 == 0");
  launch_debug_dequant(format, lin->w, lin->scales, lin->zeros, out_features, in_features, out_dev, stream);
  AMK_CUDA(nullptr, cudaGetLastError());
  AMK_CUDA(nullptr, cudaStreamSynchronize((cudaStream_t)stream));
  return AMK_OK;
}

amk_status amk_debug_hbm_read_probe(int32_t mode, const void* buf_dev, size_t bytes, uint32_t* out_dev,
                                    size_t out_words, void* stream) {
  if (mode != 0 && mode != 1)
    return fail(nullptr, AMK_ERR_INVALID_ARG, "hbm read probe: mode must be 0 (bulk ring) or 1 (128-bit loads)");
  if (!buf_dev || !out_dev || !aligned(buf_dev, 16) || !aligned(out_dev, 4) || bytes == 0 ||
      bytes % kHbmProbeTileBytes)
    return fail(nullptr, AMK_ERR_INVALID_ARG,
                "hbm read probe: buffer must be 16-byte aligned and a non-zero multiple of 16384 bytes");
  int dev = 0, sms = 0;
  AMK_CUDA(nullptr, cudaGetDevice(&dev));
  AMK_CUDA(nullptr, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t need = (size_t)2 * (mode == 0 ? sms : 4 * sms);
  if (out_words < need)
    return fail(nullptr, AMK_ERR_INVALID_ARG, "hbm read probe: out buffer needs 8 * SM count words");
  cudaStream_t s = (cudaStream_t)stream;
  AMK_CUDA(nullptr, cudaMemsetAsync(out_dev, 0, need * sizeof(uint32_t), s));
  AMK_CUDA(nullptr, launch_hbm_probe(mode, buf_dev, bytes, out_dev, sms, 2000000000ull, stream));
  return AMK_OK;
}

}  // extern "C"
