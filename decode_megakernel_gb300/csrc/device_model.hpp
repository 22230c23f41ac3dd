// Structures shared by the host library and the persistent decode kernel.
#pragma once

#include <cuda.h>   // CUtensorMap (a plain 128-byte descriptor)
#include <cuda_runtime.h>

#include <cstdint>

#include "schedule.hpp"

namespace amk {

// One task of a CTA's queue as the kernel reads it (32 bytes).  A task's
// inputs are tagged words: it polls them until they carry the version it
// needs, so the task table holds no wait or signal.
struct alignas(16) DevTask {
  int16_t type;
  int16_t layer;
  int32_t a0, a1, a2, a3;   // GEMV: row blocks [a0, a1); ATTN: kv head a0, split a1;
                            // COMBINE: kv head a0, query head a1 within its group
  int32_t pad[3];
};
static_assert(sizeof(DevTask) == 32, "DevTask layout");

// Tiled weight matrix (see MatGeom).  Layer l of a per-layer matrix starts
// at base + l * layer_bytes; int8 row scales (fp16) of layer l start at
// scales + l * rows_padded.
struct DevMat {
  const uint8_t* base;
  const uint16_t* scales;
  int64_t layer_bytes;
  int64_t rb_bytes;
  int32_t stage_bytes;    // tile + side bytes copied per stage
  int32_t fmt, rows, rows_padded, K, Kp, Kt, nkt, Rt, cpr_shift;
};

struct DevModel {
  const DevMat* mat;           // [M_NUM] in device memory (indexed by task kind)
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab, max_seq;
  int32_t group, splits, part_stride, num_ctas;
  float rms_eps;
  int32_t ring_slots;          // ring copies in flight at most (1 <= ring_slots <= kRingSlots)
  int32_t prefetch_tiles;      // weight tiles the producer may prefetch into L2 beyond its full
                               // ring while the consumers are in attention / merge / O tasks
  int32_t pad0;
  const uint16_t* embed;       // bf16 [vocab][hidden], row major
  const uint16_t* final_norm;  // bf16 [hidden]
  const uint16_t* attn_norm;   // bf16 [n_layers][hidden]
  const uint16_t* ffn_norm;    // bf16 [n_layers][hidden]
  const float2* rope;          // (cos, sin) [max_seq][head_dim / 2]
  uint16_t* kv;                // bf16 [n_layers][2][n_kv_heads][max_seq][head_dim]
  // per-step scratch of tagged words (fp32 rounded to 28 bits | 4-bit version tag)
  uint32_t* xres;              // residual stream entering a layer [hidden]
  uint32_t* xmid;              // residual stream after attention [hidden]
  uint32_t* qkv;               // [n_kv_heads][(group + 2) * head_dim]: rotated q heads, k, v
  uint32_t* o;                 // attention output [n_heads * head_dim]
  uint32_t* a;                 // SwiGLU activations [ffn]
  uint32_t* part;              // attention partials [n_kv_heads][splits][part_stride]:
                               // acc [group][head_dim], then (m, l) per head, zero padding
  uint32_t* status;            // [0] code, [1] cta, [2] task, [3] site
  const DevTask* tasks;        // queue of CTA c: tasks[queue_off[c] .. queue_off[c + 1])
  const int32_t* queue_off;    // [num_ctas + 1]
  const int32_t* queue_body;   // [num_ctas]: tasks run when the LM head is skipped
  // TMA descriptor of the KV cache seen as rows of head_dim bf16
  // ([n_layers * 2 * n_kv_heads * max_seq][head_dim]), boxes of 64 dims x
  // (positions per KV stage) with the 128-byte swizzle
  CUtensorMap kv_map;
};

struct StepParams {
  DevModel m;
  float* logits;               // [vocab] fp32 output (unused when skip_lm)
  int32_t token;
  int32_t pos;
  uint32_t tag_base;           // (launch index * n_layers) mod kTagPeriod: version v carries
                               // tag 1 + (tag_base + v - 1) mod kTagPeriod (tag 0 is never written)
  int32_t skip_lm;
  uint64_t timeout_ns;
  // optional per-task timestamps (tuning aid): null, or
  // int64 [num_ctas][1 + trace_stride][kTraceWords], see TraceWord below
  int64_t* trace;
  int32_t trace_stride;
  int32_t n_lm;                // LM-head tasks: argmax pairs per step
  // greedy decoding on the device (all null for a plain step):
  uint32_t* amax;              // [n_lm][2] this step's (max logit bits, row) per LM task
  const uint32_t* token_src;   // the previous step's pairs: this step's token is their argmax
  int32_t* token_out;          // CTA 0 records the token it derived there
};

// Trace record words.  Row 0 of a CTA: start / end %globaltimer and clock64,
// task count, SM id.  Row 1 + i for task i: consumer begin, inputs arrived
// (thread 0's tagged poll done), main loop done, outputs stored; producer
// first / last issue, cycles blocked on a full ring; task type | layer << 8;
// consumer cycles spent waiting for ring data; attention only: chunk loop
// done, partial stored, every thread's inputs arrived.  Producer blocked
// time is in ns.
constexpr int kTraceWords = 16;
enum TraceWord : int {
  TR_C_BEGIN = 0, TR_C_WAITED = 1, TR_C_DONE = 2, TR_C_SIGNALLED = 3,
  TR_P_FIRST = 4, TR_P_LAST = 5, TR_P_BLOCKED = 6, TR_TAG = 7,
  TR_C_STARVED = 8, TR_A_STAGES = 9, TR_A_MERGED = 10, TR_A_INPUTS = 11
};

enum DevStatus : uint32_t {
  ST_OK = 0, ST_TIMEOUT = 1, ST_CHECK = 2
};
enum WaitSite : uint32_t {
  SITE_DATA = 1, SITE_FULL = 2, SITE_EMPTY = 3, SITE_DRAIN = 4, SITE_PROBE = 5, SITE_TOKEN = 6, SITE_SMEM = 7,
  // tensor-core prefill GEMM: TMA producer (stage free), MMA issuer (stage
  // loaded), epilogue (accumulator complete)
  SITE_PF_TMA = 8, SITE_PF_MMA = 9, SITE_PF_EPI = 10
};

// kernel geometry
constexpr int kConsumerWarps = kConsumerThreads / 32;  // 8
constexpr int kThreads = kConsumerThreads + 32;        // + one producer warp
// One ring per CTA carries the weight tiles of its GEMV tasks and the K,V
// history stages of its attention tasks, in the order its consumers take
// them.  Copies in flight are capped per launch (ring_slots); the other
// slots hold landed tiles while the consumers wait at a hand-off.
constexpr int kRingSlots = 12;                         // 17 KB slots
constexpr int kKvChunkStages = 4;                      // KV stages an attention chunk holds at once
constexpr int kSlotBytes = kStageBytes + kSideBytes;   // one slot: a weight tile and its side data
constexpr int kScratchFloats = 4608;                   // GEMV row partials / attention merge
// int8 / int4 GEMV tasks stage each warp's activations (256 floats) above the row
// partials, which take at most kRowsMax rows x 8 warps
constexpr int kActStageOffset = kRowsMax * kConsumerWarps;
static_assert(kActStageOffset + kConsumerWarps * 256 <= kScratchFloats, "activation staging");
constexpr int kSmemBytes = kRingSlots * kSlotBytes + kScratchFloats * 4 + 2 * kRingSlots * 8 + 256;

// Byte offsets of the per-step scratch regions (tagged x_res, x_mid, qkv,
// o, a, attention partials, then the status words) laid out from one base
// address.
struct StepScratchPlan {
  size_t xres = 0, xmid = 0, qkv = 0, o = 0, a = 0, part = 0, status = 0, total = 0;
  void* stream = nullptr;
  int device = 0;
};

// the per-step scratch of a model (amk_api.cpp)
StepScratchPlan step_scratch_plan(const ModelGeom& g);

// launch wrappers (decode_kernel.cu)
int decode_smem_bytes();
// persistent kernel instance for (layer weight format, LM-head format); null if none
const void* decode_kernel_for(int fmt, int lm_fmt);
void launch_pack_matrix(int kind, int fmt, const DevMat& dst, int layer, const void* w0,
                        const void* s0, const void* z0, const void* w1, const void* s1,
                        const void* z1, const void* w2, const void* s2, const void* z2,
                        int n_heads, int n_kv_heads, int head_dim, void* stream);
void launch_watchdog_probe(uint32_t* scratch, uint64_t timeout_ns, void* stream);
// token = argmax over n argmax pairs (the last step of a device greedy loop)
void launch_argmax_pairs(const uint32_t* pairs, int n, int32_t* out, void* stream);
void launch_debug_dequant(int fmt, const void* w, const void* scales, const void* zeros,
                          int rows, int K, float* out, void* stream);
// read-only HBM stream probe (hbm_probe.cu): mode 0 bulk-copy ring, mode 1
// 128-bit loads; out holds 2 words per CTA (sms CTAs, or 4 * sms in mode 1)
constexpr uint64_t kHbmProbeTileBytes = 16384;
cudaError_t launch_hbm_probe(int mode, const void* buf, uint64_t bytes, uint32_t* out, int sms,
                             uint64_t timeout_ns, void* stream);

}  // namespace amk
