// Schedule IR of the persistent decode kernel: geometry, builder, validator.
//
// The AutoMegaKernel pages describe the schedule as a typed task DAG
// synchronised by monotonic counters, walked by one threadblock per SM
// that runs wait -> dispatch -> signal over a local queue (AMK "Layer 0"
// and "Layer 2"), and a safety gate that rejects a schedule before launch
// unless the producer/consumer DAG is acyclic, every wait threshold t
// satisfies 1 <= t <= #producers, the per-SM queue orders are valid,
// multi-producer counters are joined before a consumer reads their data,
// memory accesses respect happens-before, and outputs are reachable with
// referential integrity (AMK "The safety gate").  This file is the
// host-side half of that design for this kernel.
//
// Tagged data instead of counters.  Every value one CTA hands to another
// inside a step is a 32-bit tagged word: an fp32 rounded to 28 bits with
// a 4-bit version tag in the low nibble.  A writer stores the word once per
// version; a reader polls the words it needs until every tag equals the
// version it waits for.  A read of [lo, hi) at version v is thus a wait on
// one counter per element, with one producer and threshold 1, fused with
// the data so that neither a fence nor a separate flag round trip is
// needed.  The gate's conditions carry over element by element:
//   * referential integrity: ids and ranges valid, every task queued once;
//   * each element of a tagged buffer has exactly one writer per version
//     and is written at every version 1..V of the step, all inside the
//     prefill body;  this makes every read satisfiable (1 <= t <= #producers);
//   * tags cycle through kTagPeriod values, so a stale word must never be
//     kTagPeriod or more versions behind the one awaited: when a reader
//     starts (its queue predecessor done), every element it reads must
//     already hold a version within kMaxTagGap of the awaited one;
//   * the graph of queue order plus writer -> reader edges is acyclic and
//     the queues run to completion (no deadlock);
//   * happens-before: the writers of an element are ordered by version and
//     every reader of version v finishes before the writer of v + 1 starts
//     (otherwise it could wait for a tag that is already gone); untagged
//     buffers (KV-cache rows, logits) are race free;
//   * outputs are reachable: every element of an output buffer is written.
//
// Serialised form (int64 little-endian words), used by amk_build_schedule /
// amk_validate_serialized and by the tests that build adversarial schedules:
//   header  [0x414D4B53, version=2, n_tasks, n_queues, n_buffers, n_access,
//            n_queue_items, versions_per_step]
//   buffers n_buffers x [size, kind]        kind: 0 tagged, 1 output, 2 state
//   tasks   n_tasks x [type, layer, queue, access_begin, access_count,
//                      a0, a1, a2, a3]
//   access  n_access x [buffer, lo, hi, write, version]
//   queues  n_queues x [item_begin, item_count, body_count]
//   items   n_queue_items x [task]
// A tagged access names a version in [1, versions_per_step]; an access to
// an output or state buffer names version 0.  body_count is the queue
// prefix that runs when the LM head is skipped (prefill); the remaining
// items of a queue must be skippable.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/amk.h"

namespace amk {

enum TaskType : int32_t {
  T_QKV = 0,      // rmsnorm + QKV GEMV + RoPE + KV append
  T_ATTN = 1,     // split-K GQA attention over one context split of one KV head
  T_OPROJ = 2,    // O GEMV + residual
  T_GATEUP = 3,   // rmsnorm + gate/up GEMV + SwiGLU
  T_DOWN = 4,     // down GEMV + residual
  T_LMHEAD = 5,   // final rmsnorm + LM-head GEMV
  T_COMBINE = 6,  // LSE merge of one query head's attention splits
  T_NUM_TYPES = 7
};

enum BufKind : int32_t { BUF_TAGGED = 0, BUF_OUTPUT = 1, BUF_STATE = 2 };

// matrix kinds of the GEMV tasks
enum MatKind : int32_t { M_QKV = 0, M_O = 1, M_GU = 2, M_DOWN = 3, M_LM = 4, M_NUM = 5 };

struct Access {
  int32_t buffer;
  int64_t lo, hi;
  int32_t write;
  int32_t version;   // tagged buffers: 1..versions_per_step; others 0
};

struct Task {
  int32_t type = 0, layer = 0, queue = -1;
  std::vector<Access> acc;
  int64_t a[4] = {0, 0, 0, 0};
};

struct Buffer { int64_t size = 0; int32_t kind = BUF_TAGGED; };

struct Schedule {
  std::vector<Task> tasks;
  std::vector<std::vector<int32_t>> queues;
  std::vector<int32_t> body_len;   // per queue
  std::vector<Buffer> buffers;
  int32_t versions = 0;            // versions of every tagged buffer per step
};

// Versions per step, and the tag arithmetic: version v of launch e carries
// tag 1 + ((e * V + v - 1) mod kTagPeriod); tag 0 is never written.  A word
// at most kMaxTagGap versions behind the awaited one therefore never shows
// the awaited tag.
constexpr int kMaxVersions = 4096;
constexpr int kTagPeriod = 15;
constexpr int kMaxTagGap = kTagPeriod - 1;

// Tiled layout of one weight matrix in the workspace.  Rows are grouped in
// row blocks of Rt rows; a row block is nkt tiles of [Rt x Kt] elements,
// each tile one TMA stage of kStageBytes; in_features is zero-padded to Kp = nkt*Kt.
struct MatGeom {
  int32_t fmt = 0;
  int32_t rows = 0, rows_padded = 0;  // real rows, rows padded to Rt
  int32_t K = 0, Kp = 0, Kt = 0, nkt = 0, Rt = 0;
  int32_t cpr_shift = 0;              // log2(Kt / 8): threads sharing one row
  int64_t tile_bytes = 0;             // code bytes of one tile (kStageBytes)
  int64_t side_bytes = 0;             // per-tile scale/zero bytes (int4)
  int64_t rb_bytes = 0;               // one row block: nkt * (tile + side)
  int64_t bytes = 0;                  // whole matrix
  int32_t n_rb() const { return rows_padded / Rt; }
};

#ifndef AMK_STAGE_BYTES
#define AMK_STAGE_BYTES 16384
#endif
constexpr int kStageBytes = AMK_STAGE_BYTES;    // one weight tile = one ring stage
constexpr int kSideBytes = kStageBytes / 16;     // int4 scales / zeros of a tile
constexpr int kConsumerThreads = 256;
constexpr int kRowsMax = 256;
constexpr int kMaxHReg = 64;        // activation floats a consumer thread keeps in registers
constexpr int kMaxGroupDim = 512;   // (n_heads / n_kv_heads) * head_dim

struct ModelGeom {
  amk_config cfg{};
  MatGeom mat[M_NUM];
  int32_t num_ctas = 0, splits = 0, group = 0, rows_max = 0;
  int32_t part_stride = 0;   // words of one attention partial: group * (head_dim + 2), rounded up to 4
  int32_t prefill_chunk = 0; // tokens per tensor-core prefill chunk (0: prefill by decode steps)
};

struct BuildOptions {
  int32_t num_ctas = 0;
  int32_t attn_splits = 0;
  int32_t max_rows_per_task = 0;
};

// Shape checks and tile geometry.  Returns AMK_OK or the reason in *why.
amk_status plan_geometry(const amk_config& cfg, const BuildOptions& opt, ModelGeom* g,
                         std::string* why);

// Buffers the validator reasons about.  Tagged (per-step scratch):
//   XRES  residual stream entering a layer (written by down, read by QKV / O / LM head)
//   XMID  residual stream after attention (written by O, read by gate/up and down)
//   QKV   rotated q heads, k and v of the step's position, grouped per KV head:
//         [n_kv_heads][(group + 2) * head_dim]
//   PART  attention partials [n_kv_heads][splits][part_stride]
//   O     attention output [n_heads * head_dim];  A  SwiGLU output [ffn]
// State: KVROW, the KV-cache rows at the step's position [n_layers][2][n_kv_heads * head_dim].
// Output: LOGITS [vocab]; AMAX [n_lm_tasks][2], each LM task's (max logit, its index).
enum BufId : int32_t { B_XRES = 0, B_XMID, B_QKV, B_PART, B_O, B_A, B_KVROW, B_LOGITS, B_AMAX, B_NUM };

// Lower a model to the task DAG (tasks, counters, per-CTA queues, accesses).
Schedule build_schedule(const ModelGeom& g);

struct Report { bool ok = true; std::string msg; };
Report validate(const Schedule& s);

std::vector<int64_t> serialize(const Schedule& s);
bool deserialize(const int64_t* w, size_t n_words, Schedule* out, std::string* why);

// A re-queued lowering: the tasks of `own` (the library's lowering of a
// model, whose accesses describe what the kernel does for each task's
// parameters) placed in the queues, order and body lengths that `given`
// (a serialised schedule from anywhere) assigns them.  `given` must hold
// exactly the tasks of `own`, matched by (type, layer, a0..a3); its own
// access lists are ignored.  Every queue must list its LM-head tasks after
// its body and nothing else there (a step that skips the LM head runs the
// body alone).  Returns false with the reason for anything else; the
// result still has to pass validate() before it may run.
bool requeue(const Schedule& own, const Schedule& given, Schedule* out, std::string* why);

}  // namespace amk
