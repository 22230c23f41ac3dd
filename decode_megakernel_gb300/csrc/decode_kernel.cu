// Persistent batch-1 decode kernel for sm_103a.
//
// One cooperative CTA per SM walks its static task queue, the execution
// model of the AutoMegaKernel "Layer 0" VM (wait -> dispatch -> signal over
// a local queue).  Two departures from the pages' design:
//   * a CTA is split into a producer warp and eight consumer warps.  The
//     producer streams the weight tiles of the CTA's whole queue (1-D TMA
//     bulk copies) and the K,V history of its attention tasks (2-D
//     swizzled TMA boxes) through one shared-memory ring of twelve 17 KB
//     slots, in queue order, with at most six copies in flight (a launch
//     parameter); copies complete on mbarriers.
//     Weights never depend on activations and the history never depends on
//     the current step, so the producer runs ahead across the consumers'
//     waits; this hides the per-tile cross-SM synchronisation cost the
//     pages name as the bottleneck on high-bandwidth GPUs (AMK
//     "Experimental results": training-class GPUs).
//   * the monotonic counters are fused into the data: every value handed
//     between CTAs is a tagged word (fp32 rounded to 28 bits | 4-bit version
//     tag).  A task polls its inputs until they carry the version it needs
//     and its tagged stores are its signal, so a hand-off costs one L2 round
//     trip instead of a release fence, a counter poll and a data load.
// The consumers keep the activation vector in registers, reduce with warp
// shuffles and apply the fused epilogues (RoPE + KV append, residual adds,
// SwiGLU, logits); bf16 GEMVs run on packed FMA, int8 / int4 GEMVs and
// attention on the tensor cores (mma.sync).  Every
// wait is bounded by %globaltimer: on expiry the kernel records a status
// word, lets its own copies land and returns.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_model.hpp"
#include "ptx.cuh"

namespace amk {

// ------------------------------------------------------------------ PTX


__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(tx)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled TMA load of one box (coordinates: x = element, y = row) into
// shared memory, completing on an mbarrier; the tensor map lives in the
// kernel's parameter space.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}


// Tagged words.  A value handed from one CTA to another inside a step is an
// fp32 rounded to nearest-even at bit 4 (28 of its 32 bits kept, i.e. 19
// explicit significand bits) whose low nibble carries the version tag.  A 32-bit store and load are single-copy
// atomic, so a reader that sees the awaited tag also sees that version's
// value: no fence, flag or counter round trip stands between producer and
// consumer.
constexpr uint32_t kTagMask = 0xFu;

__device__ __forceinline__ uint32_t tag_of(const StepParams& p, int version) {
  return 1u + (p.tag_base + (uint32_t)(version + kTagPeriod - 1)) % (uint32_t)kTagPeriod;
}

__device__ __forceinline__ uint32_t tag_word(float v, uint32_t tag) {
  uint32_t b = __float_as_uint(v);
  b += 0x7u + ((b >> 4) & 1u);
  return (b & ~kTagMask) | tag;
}

__device__ __forceinline__ float tag_value(uint32_t w) { return __uint_as_float(w & ~kTagMask); }

// the value a tagged word would carry (same rounding), as a float
__device__ __forceinline__ float tag_round(float v) { return tag_value(tag_word(v, 0u)); }

__device__ __forceinline__ bool tags_are(const uint4& v, uint32_t tag) {
  return ((v.x & kTagMask) == tag) & ((v.y & kTagMask) == tag) & ((v.z & kTagMask) == tag) &
         ((v.w & kTagMask) == tag);
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_v4(uint32_t* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// named barrier 1: the 256 consumer threads only (the producer warp never joins)
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// consumer barrier that also ORs a predicate over all consumer threads
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kConsumerThreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------ shared memory

struct Smem {
  uint8_t ring[kRingSlots][kSlotBytes];   // weight tiles and K,V stages, in queue order
  float scratch[kScratchFloats];
  uint64_t full[kRingSlots];
  uint64_t empty[kRingSlots];
  alignas(16) float misc[32];
  int32_t abort_flag;
  int32_t cur_task;   // queue index of the consumers' current task (read by the producer)
  int32_t token;      // the step's input token
};
static_assert(sizeof(Smem) <= kSmemBytes, "shared memory layout");

// ------------------------------------------------------------- status

__device__ void set_status(uint32_t* status, uint32_t code, uint32_t task, uint32_t site) {
  if (atomicCAS(&status[0], 0u, code) == 0u) {
    status[1] = blockIdx.x;
    status[2] = task;
    status[3] = site;
    __threadfence();
  }
}

// Bounded poll of N 16-byte vectors of tagged words (bit i of `active`
// selects vector i; the others are left alone) until every tag equals
// `tag`.  Only the vectors still stale are reloaded.  Returns false when
// the CTA is aborting, or after timeout_ns, having recorded ST_TIMEOUT and
// raised the abort flag.
template <int N, typename Addr>
__device__ __forceinline__ bool poll_tagged(Addr at, uint4 (&v)[N], uint32_t active, uint32_t tag,
                                            uint32_t* status, volatile int32_t* abort_flag,
                                            uint64_t timeout_ns, uint32_t task) {
  static_assert(N <= 32, "one pending bit per vector");
  uint32_t pending = active;
  uint64_t t0 = 0;
  for (;;) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (pending & (1u << i)) v[i] = ld_relaxed_v4(at(i));
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((pending & (1u << i)) && tags_are(v[i], tag)) pending &= ~(1u << i);
    if (!pending) return true;
    if (*abort_flag) return false;
    const uint64_t now = global_timer();
    if (!t0) {
      t0 = now;
    } else if (now - t0 > timeout_ns) {
      set_status(status, ST_TIMEOUT, task, SITE_DATA);
      *abort_flag = 1;
      return false;
    }
  }
}

// Bounded poll of one tagged word; its value goes to *out.
__device__ __forceinline__ bool poll_word(const uint32_t* ptr, uint32_t tag, float* out,
                                          uint32_t* status, volatile int32_t* abort_flag,
                                          uint64_t timeout_ns, uint32_t task) {
  uint64_t t0 = 0;
  for (;;) {
    const uint32_t w = ld_relaxed(ptr);
    if ((w & kTagMask) == tag) {
      *out = tag_value(w);
      return true;
    }
    if (*abort_flag) return false;
    const uint64_t now = global_timer();
    if (!t0) {
      t0 = now;
    } else if (now - t0 > timeout_ns) {
      set_status(status, ST_TIMEOUT, task, SITE_DATA);
      *abort_flag = 1;
      return false;
    }
  }
}

// Bounded wait for an mbarrier phase.  Gives up when the CTA is aborting.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* status,
                           volatile int32_t* abort_flag, uint64_t timeout_ns, uint32_t task,
                           uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((spin & 15u) == 0u && global_timer() - t0 > timeout_ns) {
      set_status(status, ST_TIMEOUT, task, site);
      *abort_flag = 1;
      return false;
    }
  }
}

// ------------------------------------------------------------ task helpers

__device__ __forceinline__ int mat_kind(int type) {
  switch (type) {
    case T_QKV: return M_QKV;
    case T_OPROJ: return M_O;
    case T_GATEUP: return M_GU;
    case T_DOWN: return M_DOWN;
    default: return M_LM;
  }
}

// context split j of a KV head: cached positions [t0, t1) read from the
// cache history; the current position is handled by the last split
__device__ __forceinline__ void attn_range(int pos, int splits, int j, int* t0, int* t1) {
  const int len = (pos + splits - 1) / splits;
  int a = j * len;
  if (a > pos) a = pos;
  int b = a + len;
  if (b > pos) b = pos;
  *t0 = a;
  *t1 = b;
}

__device__ __forceinline__ int attn_positions_per_stage(int head_dim) {
  return (kStageBytes / 2) / (head_dim * 2);
}

__device__ __forceinline__ const uint16_t* kv_row(const DevModel& m, int layer, int kvsel, int g,
                                                  int t) {
  return m.kv + ((((int64_t)layer * 2 + kvsel) * m.n_kv_heads + g) * m.max_seq + t) *
                    (int64_t)m.head_dim;
}

// -------------------------------------------------------------- producer

__device__ __forceinline__ int64_t* trace_row(const StepParams& p, int i) {
  return p.trace + ((int64_t)blockIdx.x * (1 + p.trace_stride) + 1 + i) * kTraceWords;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The tiles one task streams through the ring, in order.  A weight task's
// tiles are consecutive stage_bytes chunks of one contiguous range; an
// attention task's tile s holds K then V of up to pps cached positions.
struct TaskTiles {
  const uint8_t* k = nullptr;
  const uint8_t* v = nullptr;
  int rk = 0, rv = 0;   // attention: KV-cache tensor rows of position 0 (K, V)
  int64_t stride = 0;   // weights: bytes between tiles
  uint32_t bytes = 0;   // weights: bytes per tile
  int nst = 0;          // number of tiles
  int t0 = 0, t1 = 0, pps = 0, row = 0;  // attention: positions, per stage, bytes per position
  bool attn = false;
};

__device__ __forceinline__ TaskTiles task_tiles(const StepParams& p, const DevTask& t) {
  const DevModel& m = p.m;
  TaskTiles tt;
  if (t.type == T_ATTN) {
    attn_range(p.pos, m.splits, t.a1, &tt.t0, &tt.t1);
    tt.pps = attn_positions_per_stage(m.head_dim);
    tt.row = m.head_dim * 2;
    tt.rk = ((t.layer * 2 + 0) * m.n_kv_heads + t.a0) * m.max_seq;
    tt.rv = ((t.layer * 2 + 1) * m.n_kv_heads + t.a0) * m.max_seq;
    tt.nst = (tt.t1 - tt.t0 + tt.pps - 1) / tt.pps;
    tt.attn = true;
  } else if (t.type == T_COMBINE) {
    tt.nst = 0;
  } else {
    const int kind = mat_kind(t.type);
    const DevMat M = m.mat[kind];
    tt.k = M.base + (kind == M_LM ? 0 : (int64_t)t.layer * M.layer_bytes) + (int64_t)t.a0 * M.rb_bytes;
    tt.stride = M.stage_bytes;
    tt.bytes = (uint32_t)M.stage_bytes;
    tt.nst = (t.a1 - t.a0) * M.nkt;
  }
  return tt;
}

// A cursor over the queue's ring tiles (the producer's copies, or the
// L2 prefetches that run ahead of them).
struct RingCursor {
  int task = 0, tile = 0;
  TaskTiles tt;
  bool valid = false;
  uint32_t slot = 0, phase = 0;
  int64_t blocked = 0;   // trace: ns spent blocked
};

__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Producer: one thread streams the CTA's queue through the ring in the
// order the consumers take it: the weight tiles of GEMV tasks and the K,V
// history stages of attention tasks share the slots.  Neither depends on
// this step's activations, so the producer runs up to a full ring ahead of
// the consumers.  Copy k is issued once its slot is free and copy
// k - ring_slots has landed: a TMA stream runs best with 96-128 KB in flight
// per SM, and the rest of the ring keeps landed tiles for the consumers to
// find when they come out of a hand-off (the attention -> merge -> O chain
// consumes no weights for several microseconds).
__device__ void producer_loop(const StepParams& p, Smem& sm, const DevTask* q, int n) {
  const DevModel& m = p.m;
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_kv = policy_evict_normal();
  volatile int32_t* abort_flag = &sm.abort_flag;
  const uint32_t cap = (uint32_t)m.ring_slots;
  RingCursor c;
  uint32_t seq = 0;                          // copies issued
  uint32_t issued = 0, parity = 0;           // slots that held a copy, parity of each one's last
  bool ok = true;
  uint64_t wait_t0 = 0;
  // L2 prefetch of weight tiles beyond the ring while the consumers are in
  // the attention -> merge -> O chain: pf walks the weight tiles ahead of
  // the copy cursor (off by default).
  RingCursor pf;
  int64_t w_seq = 0, pf_seq = 0;   // weight tiles copied / prefetched so far
  const int64_t pf_budget = m.prefetch_tiles;
  volatile int32_t* cur_task = &sm.cur_task;

  while (ok && c.task < n) {
    if (*abort_flag) { ok = false; break; }
    if (!c.valid) {
      const DevTask& t = q[c.task];
      if (t.type == T_COMBINE) {   // no ring tiles
        ++c.task;
        continue;
      }
      c.tt = task_tiles(p, t);
      c.tile = 0;
      c.valid = true;
      c.blocked = 0;
      if (p.trace) trace_row(p, c.task)[TR_P_FIRST] = (int64_t)global_timer();
    }
    if (c.tile == c.tt.nst) {
      if (p.trace) {
        int64_t* tr = trace_row(p, c.task);
        tr[TR_P_LAST] = (int64_t)global_timer();
        tr[TR_P_BLOCKED] = c.blocked;
      }
      ++c.task;
      c.valid = false;
      continue;
    }
    // what blocks copy seq: its slot still held, or copy seq - cap in flight
    uint64_t* bar = nullptr;
    uint32_t bpar = 0;
    if (!mbar_test_wait(&sm.empty[c.slot], c.phase ^ 1u)) {
      bar = &sm.empty[c.slot];
      bpar = c.phase ^ 1u;
    } else if (seq >= cap) {
      const uint32_t back = seq - cap;
      const uint32_t s2 = back % (uint32_t)kRingSlots, ph2 = (back / (uint32_t)kRingSlots) & 1u;
      if (!mbar_test_wait(&sm.full[s2], ph2)) {
        bar = &sm.full[s2];
        bpar = ph2;
      }
    }
    if (!bar) {
      uint64_t* full = &sm.full[c.slot];
      uint8_t* dst = sm.ring[c.slot];
      if (c.tt.attn) {
        // K then V of positions [p0, p0 + pps): boxes of 64 dims x pps rows,
        // 128-byte swizzled (rows past the split are loaded too and masked)
        const int p0 = c.tt.t0 + c.tile * c.tt.pps;
        const int nbox = m.head_dim / 64;
        mbar_arrive_expect_tx(full, kStageBytes);
        for (int b = 0; b < nbox; ++b) {
          tma_load_2d(dst + b * c.tt.pps * 128, &m.kv_map, 64 * b, c.tt.rk + p0, full, pol_kv);
          tma_load_2d(dst + kStageBytes / 2 + b * c.tt.pps * 128, &m.kv_map, 64 * b, c.tt.rv + p0, full,
                      pol_kv);
        }
      } else {
        mbar_arrive_expect_tx(full, c.tt.bytes);
        bulk_copy_g2s(dst, c.tt.k + (int64_t)c.tile * c.tt.stride, c.tt.bytes, full, pol_w);
        ++w_seq;
      }
      issued |= 1u << c.slot;
      parity = (parity & ~(1u << c.slot)) | (c.phase << c.slot);
      if (++c.slot == (uint32_t)kRingSlots) {
        c.slot = 0;
        c.phase ^= 1u;
      }
      ++c.tile;
      ++seq;
      wait_t0 = 0;
      continue;
    }
    // blocked.  In the attention chain, prefetch the next weight tiles into
    // L2 instead (when enabled).
    if (pf_budget > 0) {
      const int ct = *cur_task;
      const int cty = ct < n ? q[ct].type : T_LMHEAD;
      if (cty == T_ATTN || cty == T_COMBINE || cty == T_OPROJ) {
        if (pf_seq < w_seq) {   // the copies caught up: restart from the copy cursor
          pf = c;
          pf_seq = w_seq;
        }
        bool issued_pf = false;
        while (pf_seq < w_seq + pf_budget && pf.task < n && !issued_pf) {
          if (!pf.valid) {
            const DevTask& t = q[pf.task];
            if (t.type == T_ATTN || t.type == T_COMBINE) {
              ++pf.task;
              continue;
            }
            pf.tt = task_tiles(p, t);
            pf.tile = 0;
            pf.valid = true;
          }
          if (pf.tile == pf.tt.nst || pf.tt.attn) {
            ++pf.task;
            pf.valid = false;
            continue;
          }
          prefetch_l2(pf.tt.k + (int64_t)pf.tile * pf.tt.stride, pf.tt.bytes);
          ++pf.tile;
          ++pf_seq;
          issued_pf = true;
        }
        if (issued_pf) {
          wait_t0 = 0;
          continue;
        }
      }
    }
    // sleep briefly on what blocks, then look again
    const uint64_t now = global_timer();
    if (!wait_t0) {
      wait_t0 = now;
    } else if (now - wait_t0 > p.timeout_ns) {
      set_status(m.status, ST_TIMEOUT, (uint32_t)c.task, SITE_EMPTY);
      *abort_flag = 1;
      ok = false;
      break;
    }
    mbar_try_wait_hint(bar, bpar, 200);
    if (p.trace) c.blocked += (int64_t)(global_timer() - now);
  }
  // Every copy this CTA issued must land before its shared memory goes away.
  // Consumers normally wait for all of them already; when they stop early
  // (a failed wait anywhere) this is what keeps the CTA from exiting with
  // a copy in flight.
  for (int s2 = 0; s2 < kRingSlots; ++s2) {
    if (!(issued & (1u << s2))) continue;
    const uint32_t par = (parity >> s2) & 1u;
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(&sm.full[s2], par)) {
      if (global_timer() - t0 > p.timeout_ns) {
        set_status(m.status, ST_TIMEOUT, 0xFFFFFFFFu, SITE_DRAIN);
        break;
      }
    }
  }
}

// -------------------------------------------------------------- consumers

// weight decoding of one 8-element chunk (shared with the dequant check)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf16x2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// Two int8 codes held offset-binary (u = q + 128) in bytes 0, 1 (sel
// 0x5140) or 2, 3 (sel 0x5342) of w, as an f16 pair of q: each byte goes
// under the f16 exponent of 1024 (the value 1024 + u, exact), then 1152 is
// subtracted (exact: |q| <= 128 needs 8 of f16's 11 significand bits).
__device__ __forceinline__ uint32_t i8x2_f16(uint32_t w_ob, uint32_t sel) {
  const uint32_t biased = __byte_perm(w_ob, 0x64646464u, sel);
  const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&biased), __half2half2(__ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&q);
}
__device__ __forceinline__ uint32_t i8x2_lo(uint32_t w_ob) { return i8x2_f16(w_ob, 0x5140u); }
__device__ __forceinline__ uint32_t i8x2_hi(uint32_t w_ob) { return i8x2_f16(w_ob, 0x5342u); }
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// d += a (16x16, row) * b (16x8, col), f16 in, fp32 accumulate
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One mma A fragment of int4 codes as f16 q - z (see pack_kernel): the
// 32-bit word holds nibbles (row R, k, k+1) at bits 0-3 / 16-19, (R, k+2,
// k+3) at 4-7 / 20-23, (R+2, k, k+1) at 8-11 / 24-27 and (R+2, k+2, k+3) at
// 12-15 / 28-31.  A nibble pair masked in place under the f16 exponent of
// 1024 reads 1024 + q (bits 0-3) or 1024 + 16 q (bits 4-7); then
//   (1024 + q) - (1024 + z) = q - z,   (1024 + 16 q) / 16 - (64 + z) = q - z,
// both exact in f16 (|q - z| <= 15).  zc0 / zc1: f16 pair of 1024 + z for row
// R / R + 2, zf0 / zf1: f16 pair of -(64 + z).
__device__ __forceinline__ void u4_fragment(uint32_t w, uint32_t zc0, uint32_t zf0, uint32_t zc1, uint32_t zf1,
                                            uint32_t (&a)[4]) {
  const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00));   // 1/16
  const uint32_t w8 = w >> 8;
  const uint32_t p0 = (w & 0x000F000Fu) | 0x64006400u, p2 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t p1 = (w8 & 0x000F000Fu) | 0x64006400u, p3 = (w8 & 0x00F000F0u) | 0x64006400u;
  const __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), *reinterpret_cast<const __half2*>(&zc0));
  const __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), *reinterpret_cast<const __half2*>(&zc1));
  const __half2 r2 = __hfma2(*reinterpret_cast<const __half2*>(&p2), sixteenth, *reinterpret_cast<const __half2*>(&zf0));
  const __half2 r3 = __hfma2(*reinterpret_cast<const __half2*>(&p3), sixteenth, *reinterpret_cast<const __half2*>(&zf1));
  a[0] = *reinterpret_cast<const uint32_t*>(&r0);
  a[1] = *reinterpret_cast<const uint32_t*>(&r1);
  a[2] = *reinterpret_cast<const uint32_t*>(&r2);
  a[3] = *reinterpret_cast<const uint32_t*>(&r3);
}
// zero point z (0..15) as the pair constants of u4_fragment
__device__ __forceinline__ uint32_t u4_zc(uint32_t z) { return __byte_perm(z, 0x64u, 0x4040u); }
__device__ __forceinline__ uint32_t u4_zf(uint32_t zc) {
  const __half2 r = __hsub2(__half2half2(__ushort_as_half(0x6380)), *reinterpret_cast<const __half2*>(&zc));   // 960 - (1024 + z)
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float fp16_bits_to_float(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void mbar_arrive32(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for a ring slot's data (consumer side).
__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, const StepParams& p,
                                          volatile int32_t* abort_flag, uint32_t task,
                                          int64_t* starved = nullptr) {
  // try_wait itself blocks for a while before reporting an incomplete
  // phase, so a starvation measurement must time the first call too
  const int64_t c0 = starved ? clock64() : 0;
  if (mbar_try_wait32(bar, parity)) {
    if (starved) *starved += clock64() - c0;
    return true;
  }
  const uint64_t t0 = global_timer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait32(bar, parity)) {
      if (starved) *starved += clock64() - c0;
      return true;
    }
    if (*abort_flag) return false;
    if ((spin & 15u) == 0u && global_timer() - t0 > p.timeout_ns) {
      set_status(p.m.status, ST_TIMEOUT, task, SITE_FULL);
      *abort_flag = 1;
      return false;
    }
  }
}

template <int FMT>
struct Fmt;
// passes per tile = tile bytes / (256 threads x chunk bytes)
template <>
struct Fmt<AMK_FORMAT_BF16> { static constexpr int kChunkBytes = 16, kPasses = kStageBytes / (256 * 16); };
template <>
struct Fmt<AMK_FORMAT_INT8> { static constexpr int kChunkBytes = 8, kPasses = kStageBytes / (256 * 8); };
template <>
struct Fmt<AMK_FORMAT_INT4> { static constexpr int kChunkBytes = 4, kPasses = kStageBytes / (256 * 4); };

// Sum P per-lane values over the warp.  Lanes whose low (5 - log2 P) bits
// are zero return the total of value index (lane >> (5 - log2 P)); the other
// lanes of that group hold the same total.
template <int P>
__device__ __forceinline__ float transpose_reduce(float (&v)[P], int lane) {
#pragma unroll
  for (int n = P, msk = 16; n > 1; n >>= 1, msk >>= 1) {
    const bool up = (lane & msk) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? v[i + n / 2] : v[i];
      const float send = up ? v[i] : v[i + n / 2];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, msk);
    }
  }
#pragma unroll
  for (int msk = 16 / P; msk >= 1; msk >>= 1) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], msk);
  return v[0];
}

// (value, index) argmax: the larger value wins, the smaller index on a tie
__device__ __forceinline__ void amax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// argmax over the 256 consumer threads' (v, i); the result is valid in
// thread 0.  Uses sm.misc[0..16).
__device__ __forceinline__ void block_amax(float& v, int& i, float* misc) {
  const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1)
    amax_merge(v, i, __shfl_xor_sync(0xFFFFFFFFu, v, msk), __shfl_xor_sync(0xFFFFFFFFu, i, msk));
  if (lane == 0) {
    misc[2 * (tid >> 5)] = v;
    misc[2 * (tid >> 5) + 1] = __int_as_float(i);
  }
  consumer_sync();
  if (tid == 0)
    for (int w = 1; w < kConsumerWarps; ++w) amax_merge(v, i, misc[2 * w], __float_as_int(misc[2 * w + 1]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, msk);
  return v;
}

__device__ __forceinline__ void load8_f32(const float* src, float2* d) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(src));
  const float4 b = __ldcg(reinterpret_cast<const float4*>(src) + 1);
  d[0] = make_float2(a.x, a.y);
  d[1] = make_float2(a.z, a.w);
  d[2] = make_float2(b.x, b.y);
  d[3] = make_float2(b.z, b.w);
}

__device__ __forceinline__ void load8_bf16(const uint16_t* src, float2* d) {
  const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
  d[0] = bf16x2(w.x);
  d[1] = bf16x2(w.y);
  d[2] = bf16x2(w.z);
  d[3] = bf16x2(w.w);
}

// Activation chunk owned by a consumer thread: h[kt] holds act[kt*Kt + chunk*8 + 0..7]
// as four pairs.  QKV takes rmsnorm(x_res) * w_norm (layer 0: of the
// embedding row), gate/up rmsnorm(x_mid) * w_norm, the LM head
// rmsnorm(x_res) * w_final; O takes o, down takes a.  Tagged inputs are
// polled until they carry the version the task reads: the raw words land
// in h itself (one register set for the poll and the GEMV), stale chunks
// are reloaded until their tags match, then the tag bytes are cleared.
// Returns false when the CTA is aborting (h is then unspecified).
template <int NKT>
__device__ __forceinline__ bool load_activation(const StepParams& p, Smem& sm, const DevTask& t,
                                                const DevMat& M, int chunk, float2 (&h)[NKT][4],
                                                uint32_t task_idx, int64_t* tr) {
  const DevModel& m = p.m;
  const int tid = threadIdx.x;
  const bool norm = t.type == T_QKV || t.type == T_GATEUP || t.type == T_LMHEAD;
  const bool from_embed = t.type == T_QKV && t.layer == 0;
  const uint16_t* emb = m.embed + (int64_t)sm.token * m.hidden;
  const uint32_t* src = t.type == T_OPROJ ? m.o : t.type == T_DOWN ? m.a
                        : t.type == T_GATEUP ? m.xmid : m.xres;
  const int version = t.type == T_QKV ? t.layer : t.type == T_LMHEAD ? m.n_layers : t.layer + 1;
  const uint32_t tag = tag_of(p, version);
  auto load_raw = [&](const uint32_t* b, int kt) {
    const uint4 w0 = ld_relaxed_v4(b), w1 = ld_relaxed_v4(b + 4);
    h[kt][0] = make_float2(__uint_as_float(w0.x), __uint_as_float(w0.y));
    h[kt][1] = make_float2(__uint_as_float(w0.z), __uint_as_float(w0.w));
    h[kt][2] = make_float2(__uint_as_float(w1.x), __uint_as_float(w1.y));
    h[kt][3] = make_float2(__uint_as_float(w1.z), __uint_as_float(w1.w));
  };
  auto stale = [&](int kt) {
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      bad |= ((__float_as_uint(h[kt][i].x) & kTagMask) ^ tag) | ((__float_as_uint(h[kt][i].y) & kTagMask) ^ tag);
    return bad != 0;
  };
  uint32_t pending = 0;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt) {
    const int k = kt * M.Kt + chunk * 8;
    if (k < M.K) {  // K is a multiple of 8
      if (from_embed) load8_bf16(emb + k, h[kt]);
      else load_raw(src + k, kt);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[kt][i] = make_float2(0.f, 0.f);
    }
  }
  bool ok = true;
  if (!from_embed) {
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt)
      if (kt * M.Kt + chunk * 8 < M.K && stale(kt)) pending |= 1u << kt;
    uint64_t t0 = 0;
    while (pending) {
      if (sm.abort_flag) { ok = false; break; }
      const uint64_t now = global_timer();
      if (!t0) {
        t0 = now;
      } else if (now - t0 > p.timeout_ns) {
        set_status(m.status, ST_TIMEOUT, task_idx, SITE_DATA);
        sm.abort_flag = 1;
        ok = false;
        break;
      }
      // an opaque copy of the base keeps the compiler from holding NKT
      // precomputed addresses in registers across the retries
      const uint32_t* b = src + chunk * 8;
      asm volatile("" : "+l"(b));
#pragma unroll
      for (int kt = 0; kt < NKT; ++kt)
        if (pending & (1u << kt)) {
          load_raw(b + kt * M.Kt, kt);
          if (!stale(kt)) pending &= ~(1u << kt);
        }
    }
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[kt][i] = make_float2(tag_value(__float_as_uint(h[kt][i].x)), tag_value(__float_as_uint(h[kt][i].y)));
  }
  if (tr) tr[TR_C_WAITED] = (int64_t)global_timer();
  if (!norm) return ok;
  // threads tid < Kt/8 hold every chunk once: their squares sum to sum(x^2)
  float ss = 0.f;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(h[kt][i].x, h[kt][i].x, fmaf(h[kt][i].y, h[kt][i].y, ss));
  const int cpr = 1 << M.cpr_shift;
  ss = warp_sum(tid < cpr ? ss : 0.f);
  if ((tid & 31) == 0) sm.misc[tid >> 5] = ss;
  consumer_sync();
  // the eight warp sums in warp order (warps past cpr / 32 hold exact zeros)
  static_assert(kConsumerWarps == 8, "eight warp sums");
  const float4 m0 = *reinterpret_cast<const float4*>(sm.misc);
  const float4 m1 = *reinterpret_cast<const float4*>(sm.misc + 4);
  float tot = 0.f;
  tot += m0.x; tot += m0.y; tot += m0.z; tot += m0.w;
  tot += m1.x; tot += m1.y; tot += m1.z; tot += m1.w;
  const float r = rsqrtf(tot / (float)m.hidden + m.rms_eps);
  const uint16_t* nw = t.type == T_QKV ? m.attn_norm + (int64_t)t.layer * m.hidden
                       : t.type == T_GATEUP ? m.ffn_norm + (int64_t)t.layer * m.hidden
                                            : m.final_norm;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt) {
    const int k = kt * M.Kt + chunk * 8;
    if (k < M.K) {
      float2 w8[4];
      load8_bf16(nw + k, w8);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[kt][i] = make_float2(h[kt][i].x * r * w8[i].x, h[kt][i].y * r * w8[i].y);
    }
  }
  return ok;
}

// One chunk of one row against the thread's activations, accumulated as a
// pair of partial sums (packed FMA).  `a` is the chunk's shared address.
template <int FMT>
__device__ __forceinline__ float2 chunk_dot(uint32_t a, const float2 (&h)[4], float2 acc) {
  if constexpr (FMT == AMK_FORMAT_BF16) {
    const uint4 w = lds128(a);
    acc = __ffma2_rn(bf16x2(w.x), h[0], acc);
    acc = __ffma2_rn(bf16x2(w.y), h[1], acc);
    acc = __ffma2_rn(bf16x2(w.z), h[2], acc);
    acc = __ffma2_rn(bf16x2(w.w), h[3], acc);
    return acc;
  } else {
    static_assert(FMT == AMK_FORMAT_BF16, "int8 / int4 run on the tensor cores (act_fragments)");
    return acc;
  }
}

// int8 GEMV on the tensor cores (mma.sync m16n8k16, f16 in, fp32 accumulate).
// An int8 tile is 8 rows x 2048 codes; warp w owns k [256w, 256w + 256) of
// every tile, the same k its lanes hold as activation chunks (lane l:
// 256w + 8l .. + 8).  Per k block j (0..3) of the warp and row half hf
// (rows 4hf .. 4hf + 3) one mma computes D = A B with
//   A row m = 4r + s  (r: row of the half, s = 0..3: which 16-k segment),
//   A col kr          (position inside the segment),
//   B col n = s' + 4p (s': segment, p: 0 = hi, 1 = lo f16 part of the act),
// where segment s, position kr of lane-quad block j means
//   k = 256w + 16 (4s + ((kr & 7) >> 1)) + 4j + (kr & 1) + 2 (kr >> 3).
// Only D entries with s = s' are wanted; their sum over s and p is row r's
// dot over the warp's 64 k of block j.  So lane (g, t) = (lane >> 2,
// lane & 3) needs the 16 activations k = 256w + 16 (lane & 15) + 0..15 (as
// hi parts in lanes 0..15, lo parts in lanes 16..31) and the 8 codes
//   rows R = 4hf + (lane >> 4), R + 2;  k = 256w + 16 (lane & 15) + 4j + 0..3
// stored in the tile as 16 bytes per (w, j, lane): row half 0 then 1, each
// {W[R][k], W[R][k+1], W[R+2][k], W[R+2][k+1], W[R][k+2], W[R][k+3],
//  W[R+2][k+2], W[R+2][k+3]} offset-binary (q + 128).
// The activations are scaled by 2^-e (e from the warp's largest |act|, so
// that the hi part stays in f16 range and the lo part clear of f16
// underflow); hi + lo keep 22 significant bits.  Returns 2^e.
template <int NKT>
__device__ __forceinline__ float act_fragments(const float2 (&h)[NKT][4], uint32_t (&b)[NKT][4][2], float* stage,
                                              int lane) {
  float mx = 0.f;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(h[kt][i].x), fabsf(h[kt][i].y)));
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, msk));
  // max * 2^-e in [2^14, 2^15); finite inputs only (a NaN or inf propagates)
  int e = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 14 : 0;
  e = max(-126, min(126, e));
  const float down = __uint_as_float((uint32_t)(127 - e) << 23);
  const bool lo_part = lane >= 16;
  float4* st = reinterpret_cast<float4*>(stage);
  const float4* src = st + (lane & 15) * 4;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt) {
    st[2 * lane] = make_float4(h[kt][0].x, h[kt][0].y, h[kt][1].x, h[kt][1].y);
    st[2 * lane + 1] = make_float4(h[kt][2].x, h[kt][2].y, h[kt][3].x, h[kt][3].y);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = src[j];
      const float x[4] = {v.x * down, v.y * down, v.z * down, v.w * down};
      uint32_t r[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const __half2 hi = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);   // exact difference
        r[i] = lo_part ? *reinterpret_cast<const uint32_t*>(&lo) : *reinterpret_cast<const uint32_t*>(&hi);
      }
      b[kt][j][0] = r[0];
      b[kt][j][1] = r[1];
    }
    __syncwarp();
  }
  return __uint_as_float((uint32_t)(127 + e) << 23);
}


// Rotate the per-tile mma B fragments by one K tile (fragment kt + 1 moves
// to kt): with it, long int4 rows (NKT >= 4) run one copy of the ~8 KB tile
// code in a rolled loop instead of NKT unrolled copies, which keeps the
// loop inside the instruction cache (8 MOV per tile and K tile; 8B int4
// down projection 22.5 -> 17.3 us per layer).
template <int NKT>
__device__ __forceinline__ void rotate_fragments(uint32_t (&bq)[NKT][4][2]) {
  uint32_t t0[4][2];
#pragma unroll
  for (int j = 0; j < 4; ++j) { t0[j][0] = bq[0][j][0]; t0[j][1] = bq[0][j][1]; }
#pragma unroll
  for (int i = 0; i + 1 < NKT; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { bq[i][j][0] = bq[i + 1][j][0]; bq[i][j][1] = bq[i + 1][j][1]; }
#pragma unroll
  for (int j = 0; j < 4; ++j) { bq[NKT - 1][j][0] = t0[j][0]; bq[NKT - 1][j][1] = t0[j][1]; }
}

// GEMV task: rows [a0*Rt, a1*Rt) of one tiled matrix against the activation.
// `stage` counts the ring stages this CTA has consumed so far; returns the
// count after this task, or -1 when the CTA is aborting.
template <int FMT, int NKT>
__device__ __noinline__ int gemv_task(const StepParams& p, Smem& sm, const DevTask t, int stage,
                                      uint32_t task_idx, int64_t* tr) {
  constexpr int P = Fmt<FMT>::kPasses;
  constexpr int EB = Fmt<FMT>::kChunkBytes;
  const DevModel& m = p.m;
  const int kind = mat_kind(t.type);
  const DevMat M = m.mat[kind];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = M.cpr_shift;
  const int chunk = tid & ((1 << cs) - 1);
  const int rsub = tid >> cs;
  const int rpp = kConsumerThreads >> cs;
  const int wpg_shift = cs - 5;  // log2 warps per row group
  const int wg = warp & ((1 << wpg_shift) - 1);
  volatile int32_t* abort_flag = &sm.abort_flag;

  // constants the task reads after its input arrives go to L1 first (no
  // registers held): norm weights, and for the epilogue of this thread's
  // row (pair) its RoPE table entry or its int8 row scale(s)
  {
    const bool norm = t.type == T_QKV || t.type == T_GATEUP || t.type == T_LMHEAD;
    if (norm) {
      const uint16_t* nw = t.type == T_QKV ? m.attn_norm + (int64_t)t.layer * m.hidden
                           : t.type == T_GATEUP ? m.ffn_norm + (int64_t)t.layer * m.hidden
                                                : m.final_norm;
#pragma unroll
      for (int kt = 0; kt < NKT; ++kt) {
        const int k = kt * M.Kt + chunk * 8;
        if (k < M.K) asm volatile("prefetch.global.L1 [%0];" ::"l"(nw + k));
      }
    }
    const int rows = (t.a1 - t.a0) * M.Rt, r0 = t.a0 * M.Rt;
    const int my = (t.type == T_QKV || t.type == T_GATEUP) ? r0 + 2 * tid : r0 + tid;
    if (my < min(r0 + rows, M.rows)) {
      if (t.type == T_QKV) {
        const int hd = m.head_dim, gw = (m.group + 2) * hd;
        const int within = (my % gw) % hd, slot_h = (my % gw) / hd;
        if (slot_h <= m.group)
          asm volatile("prefetch.global.L1 [%0];" ::"l"(m.rope + (int64_t)p.pos * (hd >> 1) + (within >> 1)));
      }
      if (FMT == AMK_FORMAT_INT8)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(M.scales + (kind == M_LM ? 0 : (int64_t)t.layer * M.rows_padded) + my));
    }
  }
  float2 h[NKT][4];
  bool failed = !load_activation<NKT>(p, sm, t, M, chunk, h, task_idx, tr);
  // residual row of O / down (one row per thread): loaded now so that the
  // load overlaps the GEMV; its tag is checked (and the word re-polled if
  // stale) in the epilogue
  const int nrows = (t.a1 - t.a0) * M.Rt;
  const int row0 = t.a0 * M.Rt;
  const bool has_resid = (t.type == T_OPROJ || t.type == T_DOWN) && tid < nrows && row0 + tid < M.rows;
  const uint32_t* resid_src = t.type == T_OPROJ ? m.xres + row0 + tid : m.xmid + row0 + tid;
  const uint32_t resid_tag = tag_of(p, t.type == T_OPROJ ? t.layer : t.layer + 1);
  uint32_t resid_w = 0;
  if (has_resid) {
    if (t.type == T_OPROJ && t.layer == 0)   // layer 0: the embedding row, a constant
      resid_w = tag_word(__uint_as_float((uint32_t)__ldg(m.embed + (int64_t)sm.token * m.hidden + row0 + tid) << 16),
                         resid_tag);
    else
      resid_w = ld_relaxed(resid_src);
  }
  // int8 / int4: the activations as mma B fragments (staged through this
  // warp's slice of the scratch above the row partials), scaled by 1 / act_up
  constexpr bool kMma = FMT != AMK_FORMAT_BF16;
  uint32_t bq[kMma ? NKT : 1][4][2];
  float act_up = 1.f;
  if constexpr (kMma) act_up = act_fragments<NKT>(h, bq, sm.scratch + kActStageOffset + warp * 256, lane);

  const uint32_t ring0 = smem_addr(&sm.ring[0][0]);
  const uint32_t full0 = smem_addr(&sm.full[0]);
  const uint32_t empty0 = smem_addr(&sm.empty[0]);
  const uint32_t off0 = (uint32_t)(((rsub << cs) + chunk) * EB);   // pass 0 chunk
  const uint32_t pass_stride = (uint32_t)((rpp << cs) * EB);       // rows between passes
  constexpr uint32_t nslots = (uint32_t)kRingSlots;
  uint32_t slot = (uint32_t)stage % nslots, phase = ((uint32_t)stage / nslots) & 1u;
  int64_t starved = 0;

  float* red = sm.scratch;
  const int nrb = t.a1 - t.a0;
  if constexpr (FMT == AMK_FORMAT_INT8) {
    // D entries this lane keeps (see act_fragments): segment of row m = g is
    // g & 3; column 2t (+1 when that segment is odd) has the same segment
    // when t & 1 == (g & 3) >> 1
    const int sg = (lane >> 2) & 3;
    const bool keep = (lane & 1) == (sg >> 1);
    const bool odd = (sg & 1) != 0;
    const uint32_t unit0 = (uint32_t)(warp * 4 * 32 + lane) * 16;
    for (int rb = 0; rb < nrb; ++rb) {
      float d[2][2][4];   // [row half][k block parity][fragment]
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) d[a][c][e] = 0.f;
      // tiles in pairs: both waits first, then both tiles' loads and mma
      // (each accumulator still sums its k blocks in tile order)
#pragma unroll
      for (int kt = 0; kt < NKT; kt += 2) {
        const bool two = kt + 1 < NKT;
        const uint32_t slot2 = slot + 1 == nslots ? 0u : slot + 1;
        const uint32_t phase2 = slot + 1 == nslots ? phase ^ 1u : phase;
        if (!failed)
          failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
        if (two && !failed)
          failed = !wait_full(full0 + slot2 * 8, phase2, p, abort_flag, task_idx, tr ? &starved : nullptr);
        if (!failed) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u == 1 && !two) break;
            const int fk = u == 0 ? kt : (two ? kt + 1 : kt);
            const uint32_t tile = ring0 + (u == 0 ? slot : slot2) * kSlotBytes + unit0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 v = lds128(tile + (uint32_t)j * 512u);
              mma_f16_16816(d[0][j & 1], i8x2_lo(v.x), i8x2_hi(v.x), i8x2_lo(v.y), i8x2_hi(v.y), bq[fk][j][0],
                            bq[fk][j][1]);
              mma_f16_16816(d[1][j & 1], i8x2_lo(v.z), i8x2_hi(v.z), i8x2_lo(v.w), i8x2_hi(v.w), bq[fk][j][0],
                            bq[fk][j][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive32(empty0 + slot * 8);
          if (two) mbar_arrive32(empty0 + slot2 * 8);
        }
        slot = slot2;
        phase = phase2;
        if (two && ++slot == nslots) { slot = 0; phase ^= 1u; }
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float e0 = odd ? d[hf][0][1] + d[hf][1][1] : d[hf][0][0] + d[hf][1][0];
        const float e2 = odd ? d[hf][0][3] + d[hf][1][3] : d[hf][0][2] + d[hf][1][2];
        float v0 = keep ? e0 : 0.f;   // row 4 hf + (lane >> 4)
        float v1 = keep ? e2 : 0.f;   // row 4 hf + (lane >> 4) + 2
#pragma unroll
        for (int msk = 1; msk < 16; msk <<= 1) {
          v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, msk);
          v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, msk);
        }
        if ((lane & 15) == 0) {
          const int r = rb * 8 + 4 * hf + (lane >> 4);
          red[r * 8 + warp] = v0 * act_up;
          red[(r + 2) * 8 + warp] = v1 * act_up;
        }
      }
    }
  } else if constexpr (FMT == AMK_FORMAT_INT4) {
    // 16 rows x 2048 codes per tile: per k block j the lane's 16 bytes hold
    // one A word per row quarter q (rows 4q .. 4q + 3).  A lane's codes (and
    // the D entries it keeps) all lie in its segment sg, i.e. at k in
    // [256w + 64 sg, + 64) of every tile: quantisation group 2w + (sg >> 1)
    // of the tile, so one zero point and one scale per row serve all four
    // k blocks.  Side data: fp16 scales [16 groups][2 row parities][8],
    // then u8 zeros in the same order.
    const int sg = (lane >> 2) & 3;
    const bool keep = (lane & 1) == (sg >> 1);
    const bool odd = (sg & 1) != 0;
    const uint32_t unit0 = (uint32_t)(warp * 4 * 32 + lane) * 16;
    const int rl = lane >> 4;                 // row R = 4q + rl, and R + 2
    const int gq = 2 * warp + (sg >> 1);      // the lane's group in every tile
    for (int rb = 0; rb < nrb; ++rb) {
      float acc[4][2];   // [q][R, R + 2], scaled by the group scales
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = 0.f;
      // one 16-row tile against fragment set fk: the lane's 4 code words
      // per k block, its rows' scales and zero points from the side data
      auto tile_mma = [&](uint32_t tile, int fk) {
        const uint32_t side = tile + kStageBytes;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = lds128(tile + unit0 + (uint32_t)j * 512u);
        // the scales and zero points of the lane's 8 rows (R = 4q + rl and
        // R + 2 for q = 0..3: the rows of parity rl) in its group: 16 + 8
        // contiguous bytes of the side data (pack_kernel)
        const uint4 sc = lds128(side + (uint32_t)(gq * 2 + rl) * 16u);
        const uint2 zz = lds64(side + 512u + (uint32_t)(gq * 2 + rl) * 8u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // row R: entry 2q, row R + 2: entry 2q + 1
          const uint32_t zw = q < 2 ? zz.x : zz.y;
          const uint32_t zc0 = __byte_perm(zw, 0x64u, (q & 1) ? 0x4242u : 0x4040u);
          const uint32_t zc1 = __byte_perm(zw, 0x64u, (q & 1) ? 0x4343u : 0x4141u);
          const uint32_t sw = q == 0 ? sc.x : q == 1 ? sc.y : q == 2 ? sc.z : sc.w;
          const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sw));
          const uint32_t zf0 = u4_zf(zc0), zf1 = u4_zf(zc1);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t w = q == 0 ? v[j].x : q == 1 ? v[j].y : q == 2 ? v[j].z : v[j].w;
            uint32_t a[4];
            u4_fragment(w, zc0, zf0, zc1, zf1, a);
            mma_f16_16816(d, a[0], a[1], a[2], a[3], bq[fk][j][0], bq[fk][j][1]);
          }
          const float e0 = keep ? (odd ? d[1] : d[0]) : 0.f;
          const float e2 = keep ? (odd ? d[3] : d[2]) : 0.f;
          acc[q][0] = fmaf(s01.x, e0, acc[q][0]);
          acc[q][1] = fmaf(s01.y, e2, acc[q][1]);
        }
      };
      if constexpr (NKT >= 4) {
        // long rows: one rolled tile loop over rotated fragments (measured
        // faster for int4 than NKT unrolled copies)
#pragma unroll 1
        for (int kt = 0; kt < NKT; ++kt) {
          if (!failed)
            failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
          if (!failed) tile_mma(ring0 + slot * kSlotBytes, 0);
          __syncwarp();
          if (lane == 0) mbar_arrive32(empty0 + slot * 8);
          if (++slot == nslots) { slot = 0; phase ^= 1u; }
          rotate_fragments<NKT>(bq);
        }
      } else {
        // short rows: tiles in pairs, both waits first (each accumulator
        // still sums the tiles in order)
#pragma unroll
        for (int kt = 0; kt < NKT; kt += 2) {
          const bool two = kt + 1 < NKT;
          const uint32_t slot2 = slot + 1 == nslots ? 0u : slot + 1;
          const uint32_t phase2 = slot + 1 == nslots ? phase ^ 1u : phase;
          if (!failed)
            failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
          if (two && !failed)
            failed = !wait_full(full0 + slot2 * 8, phase2, p, abort_flag, task_idx, tr ? &starved : nullptr);
          if (!failed) {
            tile_mma(ring0 + slot * kSlotBytes, kt);
            if (two) tile_mma(ring0 + slot2 * kSlotBytes, two ? kt + 1 : kt);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive32(empty0 + slot * 8);
            if (two) mbar_arrive32(empty0 + slot2 * 8);
          }
          slot = slot2;
          phase = phase2;
          if (two && ++slot == nslots) { slot = 0; phase ^= 1u; }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v0 = acc[q][0], v1 = acc[q][1];
#pragma unroll
        for (int msk = 1; msk < 16; msk <<= 1) {
          v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, msk);
          v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, msk);
        }
        if ((lane & 15) == 0) {
          const int r = rb * 16 + 4 * q + rl;
          red[r * 8 + warp] = v0 * act_up;
          red[(r + 2) * 8 + warp] = v1 * act_up;
        }
      }
    }
  } else
  for (int rb = 0; rb < nrb; ++rb) {   // bf16: packed FMA
    float2 acc2[P];
#pragma unroll
    for (int i = 0; i < P; ++i) acc2[i] = make_float2(0.f, 0.f);
    // tiles in pairs: both waits first, so that the second tile's shared
    // loads issue with the first tile's FMAs in flight (the sums keep their
    // order: tile kt, then kt + 1)
#pragma unroll
    for (int kt = 0; kt < NKT; kt += 2) {
      const bool two = kt + 1 < NKT;
      const uint32_t slot2 = slot + 1 == nslots ? 0u : slot + 1;
      const uint32_t phase2 = slot + 1 == nslots ? phase ^ 1u : phase;
      if (!failed)
        failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
      if (two && !failed)
        failed = !wait_full(full0 + slot2 * 8, phase2, p, abort_flag, task_idx, tr ? &starved : nullptr);
      if (!failed) {
        const uint32_t tile = ring0 + slot * kSlotBytes;
#pragma unroll
        for (int ps = 0; ps < P; ++ps) acc2[ps] = chunk_dot<FMT>(tile + off0 + ps * pass_stride, h[kt], acc2[ps]);
        if (two) {
          const uint32_t tile2 = ring0 + slot2 * kSlotBytes;
#pragma unroll
          for (int ps = 0; ps < P; ++ps)
            acc2[ps] = chunk_dot<FMT>(tile2 + off0 + ps * pass_stride, h[two ? kt + 1 : kt], acc2[ps]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive32(empty0 + slot * 8);
        if (two) mbar_arrive32(empty0 + slot2 * 8);
      }
      slot = slot2;
      phase = phase2;
      if (two && ++slot == nslots) { slot = 0; phase ^= 1u; }
    }
    float v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] = acc2[i].x + acc2[i].y;
    const float tot = transpose_reduce<P>(v, lane);
    constexpr int kLaneStride = 32 / P;
    if ((lane & (kLaneStride - 1)) == 0) {
      const int ps = lane / kLaneStride;
      red[(rb * M.Rt + ps * rpp + rsub) * 8 + wg] = tot;
    }
  }

  if (tr) tr[TR_C_STARVED] = starved;
  if (consumer_sync_or(failed)) return -1;

  // epilogue: one row (or one row pair) per thread; tagged stores of version layer + 1
  const uint32_t tag = tag_of(p, t.layer + 1);
  const int nwg = 1 << wpg_shift;
  auto row_sum = [&](int r) {   // the first nwg of the row's 8 partials, in warp order
    const float4 a = *reinterpret_cast<const float4*>(red + r * 8);
    const float4 b = *reinterpret_cast<const float4*>(red + r * 8 + 4);
    float y = 0.f;
    y += a.x;
    y += nwg > 1 ? a.y : 0.f;
    y += nwg > 2 ? a.z : 0.f;
    y += nwg > 2 ? a.w : 0.f;
    y += nwg > 4 ? b.x : 0.f;
    y += nwg > 4 ? b.y : 0.f;
    y += nwg > 4 ? b.z : 0.f;
    y += nwg > 4 ? b.w : 0.f;
    return y;
  };
  if (t.type == T_QKV || t.type == T_GATEUP) {
    const int hd = m.head_dim, half = hd >> 1, G = m.group, gw = (G + 2) * hd;
    const int hd_shift = hd == 128 ? 7 : 6;   // head_dim is 64 or 128
    for (int pr = tid; pr < nrows / 2; pr += kConsumerThreads) {
      const int R = row0 + 2 * pr;
      if (R >= M.rows) continue;
      float y0 = row_sum(2 * pr), y1 = row_sum(2 * pr + 1);
      if (FMT == AMK_FORMAT_INT8) {
        const uint16_t* sc = M.scales + (int64_t)t.layer * M.rows_padded;
        y0 *= fp16_bits_to_float(sc[R]);
        y1 *= fp16_bits_to_float(sc[R + 1]);
      }
      if (t.type == T_GATEUP) {
        st_relaxed(m.a + (R >> 1), tag_word(silu(y0) * y1, tag));
        continue;
      }
      // packed QKV rows per KV head: G query heads, k, v (RoPE pairs adjacent)
      const int grp = R / gw, r = R - grp * gw, slot_h = r >> hd_shift, within = r & (hd - 1);
      uint32_t* dst = m.qkv + (int64_t)grp * gw + slot_h * hd;
      if (slot_h <= G) {
        // rotate-half RoPE pair (i, i + hd/2) at position pos
        const int i = within >> 1;
        const float2 cs2 = m.rope[(int64_t)p.pos * half + i];
        float a = y0 * cs2.x - y1 * cs2.y;
        float b = y1 * cs2.x + y0 * cs2.y;
        if (slot_h == G) {  // k: the cache holds bf16, attention uses the same values
          const __nv_bfloat16 ka = __float2bfloat16_rn(a), kb = __float2bfloat16_rn(b);
          uint16_t* kr = const_cast<uint16_t*>(kv_row(m, t.layer, 0, grp, p.pos));
          kr[i] = __bfloat16_as_ushort(ka);
          kr[half + i] = __bfloat16_as_ushort(kb);
          a = __bfloat162float(ka);
          b = __bfloat162float(kb);
        }
        st_relaxed(dst + i, tag_word(a, tag));
        st_relaxed(dst + half + i, tag_word(b, tag));
      } else {
        const __nv_bfloat16 v0 = __float2bfloat16_rn(y0), v1 = __float2bfloat16_rn(y1);
        uint16_t* vrow = const_cast<uint16_t*>(kv_row(m, t.layer, 1, grp, p.pos));
        vrow[within] = __bfloat16_as_ushort(v0);
        vrow[within + 1] = __bfloat16_as_ushort(v1);
        st_relaxed(dst + within, tag_word(__bfloat162float(v0), tag));
        st_relaxed(dst + within + 1, tag_word(__bfloat162float(v1), tag));
      }
    }
  } else {
    float best_v = -INFINITY;   // LM head: this thread's (max logit, row)
    int best_i = 0x7FFFFFFF;
    for (int r = tid; r < nrows; r += kConsumerThreads) {
      const int R = row0 + r;
      if (R >= M.rows) continue;
      float y = row_sum(r);
      if (FMT == AMK_FORMAT_INT8) {
        const uint16_t* sc = M.scales + (kind == M_LM ? 0 : (int64_t)t.layer * M.rows_padded);
        y *= fp16_bits_to_float(sc[R]);
      }
      if (t.type == T_LMHEAD) {
        p.logits[R] = y;
        amax_merge(best_v, best_i, y, R);
      } else {  // O / down: residual add on the owned row (r == tid)
        float resid = tag_value(resid_w);
        if ((resid_w & kTagMask) != resid_tag &&
            !poll_word(resid_src, resid_tag, &resid, m.status, abort_flag, p.timeout_ns, task_idx))
          continue;   // aborting: the step's status word already says why
        st_relaxed((t.type == T_OPROJ ? m.xmid : m.xres) + R, tag_word(resid + y, tag));
      }
    }
    // greedy decoding on the device: this task's (max logit, row) pair
    if (t.type == T_LMHEAD && p.amax) {
      block_amax(best_v, best_i, sm.misc);
      if (tid == 0) {
        p.amax[2 * t.a2] = __float_as_uint(best_v);
        p.amax[2 * t.a2 + 1] = (uint32_t)best_i;
      }
    }
  }
  return stage + nrb * NKT;
}

template <int FMT>
__device__ __forceinline__ int gemv_dispatch(const StepParams& p, Smem& sm, const DevTask& t,
                                             int stage, uint32_t i, int64_t* tr) {
  switch (p.m.mat[mat_kind(t.type)].nkt) {
    case 1: return gemv_task<FMT, 1>(p, sm, t, stage, i, tr);
    case 2: return gemv_task<FMT, 2>(p, sm, t, stage, i, tr);
    case 3: return gemv_task<FMT, 3>(p, sm, t, stage, i, tr);
    case 4: return gemv_task<FMT, 4>(p, sm, t, stage, i, tr);
    case 5: return gemv_task<FMT, 5>(p, sm, t, stage, i, tr);
    case 6: return gemv_task<FMT, 6>(p, sm, t, stage, i, tr);
    case 7: return gemv_task<FMT, 7>(p, sm, t, stage, i, tr);
    default: return gemv_task<FMT, 8>(p, sm, t, stage, i, tr);
  }
}


// Split-K GQA attention of one KV head over one context split (positions
// [t0, t1) of the cache, plus the step's own position for the last split),
// on the tensor cores.  The K,V history arrives through the ring in
// 128-byte-swizzled boxes; a chunk of up to kKvChunkStages resident stages is
// split into runs of 16 (hd 128) or 32 (hd 64) positions, one per warp.
// Per 16 positions a warp computes
//   S^T [16 positions x 8 heads] = K [16 x hd] . Q^T [hd x 8]    (hd/16 mma pairs)
//   O^T [hd x 8]              += V^T [hd x 16] . P^T [16 x 8]    (hd/16 mma pairs)
// with ldmatrix fragments of K and (transposed) V, G <= 8 real heads in the
// 8 columns, and q and P split into bf16 hi + lo so that the products keep
// fp32-level accuracy (K, V are bf16 already).  The softmax is one maximum
// and one sum per head and chunk over the run, folded into the warp's
// running (m, l, O); the eight warp states are merged (LSE) through shared
// memory and stored as the split's partial (acc, m, l).
template <int HD, int G>
__device__ __noinline__ int attn_task(const StepParams& p, Smem& sm, const DevTask t, int stage,
                                      uint32_t task_idx, int64_t* tr) {
  constexpr int PPS = (kStageBytes / 2) / (HD * 2);   // cached positions per KV stage
  constexpr int CP = kKvChunkStages * PPS;            // positions per chunk at most
  constexpr int RUN = CP / kConsumerWarps;            // positions of a warp's run at most
  constexpr int MT = RUN / 16;                        // 16-position tiles per run
  constexpr int KS = HD / 16;                         // k-steps (QK) and dim tiles (PV)
  static_assert(G <= 8 && RUN % 16 == 0 && HD % 64 == 0 && RUN <= PPS, "attention tile shapes");
  // scratch (floats): q staging, the step's own k / v as bf16 rows, then
  // at the end the warp states [warp][G][HD + 2]
  constexpr int WS = G * (HD + 2);
  constexpr int QS_OFF = 0, CUR_OFF = kScratchFloats - HD, MG_OFF = 0;
  static_assert(QS_OFF + G * HD <= CUR_OFF && MG_OFF + kConsumerWarps * WS <= CUR_OFF,
                "attention scratch");
  const DevModel& m = p.m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq4 = lane >> 2, tq4 = lane & 3;   // mma fragment coordinates
  const int g = t.a0, j = t.a1;
  volatile int32_t* abort_flag = &sm.abort_flag;
  float* qs = sm.scratch + QS_OFF;
  float* mg = sm.scratch + MG_OFF;
  uint16_t* cur = reinterpret_cast<uint16_t*>(sm.scratch + CUR_OFF);   // [2][HD] bf16: k, v

  const uint32_t tag = tag_of(p, t.layer + 1);
  const uint32_t* gqp = m.qkv + (int64_t)g * (G + 2) * HD;   // q heads, k, v of this KV head
  constexpr int QV = G * HD / 4, KVV = HD / 2;
  static_assert(QV + KVV <= kConsumerThreads, "one vector per thread");
  const bool last = j == m.splits - 1;
  bool failed = false;
  // inputs: q of the group (fp32) and, last split, the step's k and v (as
  // the bf16 they are) by 16-byte vectors into shared memory
  if (tid < QV || (last && tid < QV + KVV)) {
    const uint32_t* src = tid < QV ? gqp + tid * 4 : gqp + G * HD + (tid - QV) * 4;
    uint4 v[1];
    failed = !poll_tagged<1>([&](int) { return src; }, v, 1u, tag, m.status, abort_flag,
                             p.timeout_ns, task_idx);
    if (tid < QV) {
      float* dst = qs + tid * 4;
      dst[0] = tag_value(v[0].x);
      dst[1] = tag_value(v[0].y);
      dst[2] = tag_value(v[0].z);
      dst[3] = tag_value(v[0].w);
    } else {
      // k dims then v dims; the words carry bf16 values, whose bits are the
      // upper half of the fp32 (the tag sits in the low nibble)
      uint16_t* dst = cur + (tid - QV) * 4;
      dst[0] = (uint16_t)(v[0].x >> 16);
      dst[1] = (uint16_t)(v[0].y >> 16);
      dst[2] = (uint16_t)(v[0].z >> 16);
      dst[3] = (uint16_t)(v[0].w >> 16);
    }
  }
  if (tr) tr[TR_C_WAITED] = (int64_t)global_timer();
  failed = consumer_sync_or(failed);
  if (tr) tr[TR_A_INPUTS] = (int64_t)global_timer();
  // Q^T fragments (hi, lo) of every k-step, pre-scaled into log2 units;
  // columns (heads) >= G are zero
  const float qscale = 1.4426950408889634f * rsqrtf((float)HD);
  uint32_t qb[KS][2][2];   // [k-step][b0 / b1][hi / lo]
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d = ks * 16 + half * 8 + 2 * tq4;
      float x0 = 0.f, x1 = 0.f;
      if (gq4 < G) {
        x0 = qs[gq4 * HD + d] * qscale;
        x1 = qs[gq4 * HD + d + 1] * qscale;
      }
      split_bf16x2(x0, x1, qb[ks][half][0], qb[ks][half][1]);
    }
  // warp state: running max / sum of heads 2*tq4 and 2*tq4 + 1, O^T fragments
  float mx0 = -INFINITY, mx1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[KS][4];
#pragma unroll
  for (int k2 = 0; k2 < KS; ++k2)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[k2][e] = 0.f;

  constexpr uint32_t kvs = (uint32_t)kRingSlots;   // the ring's slots (>= kKvChunkStages)
  const uint32_t cur0 = smem_addr(cur);
  const uint32_t kfull0 = smem_addr(&sm.full[0]);
  const uint32_t kempty0 = smem_addr(&sm.empty[0]);
  int64_t starved = 0;
  int t0, t1;
  attn_range(p.pos, m.splits, j, &t0, &t1);
  const int ncached = t1 - t0;
  const int ntotal = ncached + (last ? 1 : 0);
  const int nst = (ncached + PPS - 1) / PPS;
  uint32_t kslot = (uint32_t)stage % kvs, kphase = ((uint32_t)stage / kvs) & 1u;

  for (int c0 = 0; c0 < ntotal; c0 += CP) {
    const int len = min(CP, ntotal - c0);
    const int s_begin = c0 / PPS;
    const int s_end = min(c0 + len, ncached) > c0 ? (min(c0 + len, ncached) + PPS - 1) / PPS : s_begin;
    const uint32_t slot0 = kslot;
    // this warp's run [c0 + w0, c0 + w0 + n)
    const int per = (len + kConsumerWarps - 1) / kConsumerWarps;
    const int w0 = min(len, warp * per);
    const int n = min(len, w0 + per) - w0;
    // a warp waits only for the stages that hold its run's cached positions
    // (an mbarrier wait costs ~300 cycles even on a completed phase); every
    // stage is some warp's, and a stage's slot is refilled only after all
    // eight warps released it, so no slot is released before its data
    // landed and was read
    const int cfirst = c0 + w0, clast = min(c0 + w0 + n, ncached) - 1;
    for (int s2 = s_begin; s2 < s_end; ++s2) {
      const bool mine = s2 * PPS <= clast && (s2 + 1) * PPS > cfirst;
      if (!failed && mine)
        failed = !wait_full(kfull0 + kslot * 8, kphase, p, abort_flag, task_idx, tr ? &starved : nullptr);
      if (++kslot == kvs) { kslot = 0; kphase ^= 1u; }
    }
    // shared address of 16-byte chunk c (8 dims) of K (kv = 0) or V (kv = 1)
    // of task position pi: a swizzled ring row, or the step's own k / v
    // The warp's run (at most RUN <= PPS positions) lies in stages stA and
    // stA + 1 at most: their slot addresses are computed once per chunk.
    const int stA = (c0 + w0) / PPS;
    auto slot_base = [&](int st) -> uint32_t {
      uint32_t slot = slot0 + (uint32_t)(st - s_begin);
      if (slot >= kvs) slot -= kvs;
      return smem_addr(&sm.ring[slot][0]);
    };
    const uint32_t baseA = slot_base(stA), baseB = slot_base(stA + 1);
    auto addr_of = [&](int pi, int c, int kv) -> uint32_t {
      if (pi >= ncached) return cur0 + (uint32_t)(kv * HD * 2 + c * 16);
      const int r = pi % PPS;
      return (pi / PPS == stA ? baseA : baseB) +
             (uint32_t)(kv * (kStageBytes / 2) + (c >> 3) * (PPS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    };
    if (!failed && n > 0) {
      const int base = c0 + w0;
      const int plast = base + n - 1;   // padding rows read this position (masked)
      // scores S^T: rows (positions) gq4 and gq4 + 8 of each tile, columns
      // (heads) 2*tq4 and 2*tq4 + 1
      float sc[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[mt][e] = 0.f;
        if (mt * 16 < n) {
          const int mi = lane >> 3, rr = lane & 7;
          const int pi = min(base + mt * 16 + rr + 8 * (mi & 1), plast);
          // four independent accumulation chains (k-step parity x hi / lo
          // part of q), summed once: a single chain serialises 2 KS mma
          float acc4[4][4];
#pragma unroll
          for (int c = 0; c < 4; ++c) acc4[c][0] = acc4[c][1] = acc4[c][2] = acc4[c][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(addr_of(pi, 2 * ks + (mi >> 1), 0), a);
            mma_bf16_16816(acc4[2 * (ks & 1)], a, qb[ks][0][0], qb[ks][1][0]);
            mma_bf16_16816(acc4[2 * (ks & 1) + 1], a, qb[ks][0][1], qb[ks][1][1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[mt][e] = (acc4[0][e] + acc4[2][e]) + (acc4[1][e] + acc4[3][e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (mt * 16 + gq4 + 8 * (e >> 1) >= n) sc[mt][e] = -INFINITY;
      }
      // softmax of the run for heads 2*tq4, 2*tq4 + 1: lanes of a head
      // differ in gq4 (lane bits 2..4)
      float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        cm0 = fmaxf(cm0, fmaxf(sc[mt][0], sc[mt][2]));
        cm1 = fmaxf(cm1, fmaxf(sc[mt][1], sc[mt][3]));
      }
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        cm0 = fmaxf(cm0, __shfl_xor_sync(0xFFFFFFFFu, cm0, msk));
        cm1 = fmaxf(cm1, __shfl_xor_sync(0xFFFFFFFFu, cm1, msk));
      }
      const float mn0 = fmaxf(mx0, cm0), mn1 = fmaxf(mx1, cm1);
      const float al0 = exp2f(mx0 - mn0), al1 = exp2f(mx1 - mn1);   // 0 on the first chunk
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        sc[mt][0] = exp2f(sc[mt][0] - mn0);
        sc[mt][1] = exp2f(sc[mt][1] - mn1);
        sc[mt][2] = exp2f(sc[mt][2] - mn0);
        sc[mt][3] = exp2f(sc[mt][3] - mn1);
        ls0 += sc[mt][0] + sc[mt][2];
        ls1 += sc[mt][1] + sc[mt][3];
      }
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        ls0 += __shfl_xor_sync(0xFFFFFFFFu, ls0, msk);
        ls1 += __shfl_xor_sync(0xFFFFFFFFu, ls1, msk);
      }
      l0 = fmaf(l0, al0, ls0);
      l1 = fmaf(l1, al1, ls1);
      mx0 = mn0;
      mx1 = mn1;
#pragma unroll
      for (int k2 = 0; k2 < KS; ++k2) {
        o[k2][0] *= al0;
        o[k2][1] *= al1;
        o[k2][2] *= al0;
        o[k2][3] *= al1;
      }
      // values: P^T fragments (positions 2*tq4 (+1), (+8) of head gq4)
      // gathered from the lanes holding them, then O^T += V^T . P^T
      const int sa = (2 * tq4) * 4 + (gq4 >> 1), sb = (2 * tq4 + 1) * 4 + (gq4 >> 1);
      const bool odd = (gq4 & 1) != 0;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        if (mt * 16 >= n) continue;
        const float a0 = __shfl_sync(0xFFFFFFFFu, sc[mt][0], sa), a1 = __shfl_sync(0xFFFFFFFFu, sc[mt][1], sa);
        const float a2 = __shfl_sync(0xFFFFFFFFu, sc[mt][2], sa), a3 = __shfl_sync(0xFFFFFFFFu, sc[mt][3], sa);
        const float b0 = __shfl_sync(0xFFFFFFFFu, sc[mt][0], sb), b1 = __shfl_sync(0xFFFFFFFFu, sc[mt][1], sb);
        const float b2 = __shfl_sync(0xFFFFFFFFu, sc[mt][2], sb), b3 = __shfl_sync(0xFFFFFFFFu, sc[mt][3], sb);
        uint32_t pb0h, pb0l, pb1h, pb1l;
        split_bf16x2(odd ? a1 : a0, odd ? b1 : b0, pb0h, pb0l);   // positions 2*tq4, 2*tq4 + 1
        split_bf16x2(odd ? a3 : a2, odd ? b3 : b2, pb1h, pb1l);   // positions 2*tq4 + 8, + 9
        const int mi = lane >> 3, rr = lane & 7;
        const int pi = min(base + mt * 16 + rr + 8 * (mi >> 1), plast);
#pragma unroll
        for (int k2 = 0; k2 < KS; ++k2) {
          uint32_t a[4];
          ldsm_x4_trans(addr_of(pi, 2 * k2 + (mi & 1), 1), a);
          mma_bf16_16816(o[k2], a, pb0h, pb1h);
          mma_bf16_16816(o[k2], a, pb0l, pb1l);
        }
      }
    }
    // release the chunk's stages
    __syncwarp();
    if (lane == 0) {
      uint32_t sl = slot0;
      for (int s2 = s_begin; s2 < s_end; ++s2) {
        mbar_arrive32(kempty0 + sl * 8);
        if (++sl == kvs) sl = 0;
      }
    }
  }
  if (tr) {
    tr[TR_C_STARVED] = starved;
    tr[TR_A_STAGES] = (int64_t)global_timer();
  }
  // merge the eight warps' states (mg overlaps the q staging: wait for all)
  consumer_sync();
  {
    const int h0 = 2 * tq4, h1 = 2 * tq4 + 1;
#pragma unroll
    for (int k2 = 0; k2 < KS; ++k2) {
      const int d = k2 * 16 + gq4;
      if (h0 < G) {
        mg[warp * WS + h0 * (HD + 2) + d] = o[k2][0];
        mg[warp * WS + h0 * (HD + 2) + d + 8] = o[k2][2];
      }
      if (h1 < G) {
        mg[warp * WS + h1 * (HD + 2) + d] = o[k2][1];
        mg[warp * WS + h1 * (HD + 2) + d + 8] = o[k2][3];
      }
    }
    if (gq4 == 0) {
      if (h0 < G) {
        mg[warp * WS + h0 * (HD + 2) + HD] = mx0;
        mg[warp * WS + h0 * (HD + 2) + HD + 1] = l0;
      }
      if (h1 < G) {
        mg[warp * WS + h1 * (HD + 2) + HD] = mx1;
        mg[warp * WS + h1 * (HD + 2) + HD + 1] = l1;
      }
    }
  }
  if (consumer_sync_or(failed)) return -1;
  // partial of this split: acc [G][HD], then (m, l) per head, then padding,
  // as tagged words.  m is rounded to the tagged grid before it scales acc
  // and l, so the stored (m, acc, l) stay consistent; an empty split stores
  // m = -1e30 (weight 0 in the merge) instead of -inf, which has no room for
  // a tag.
  uint32_t* part = m.part + (int64_t)(g * m.splits + j) * m.part_stride;
  for (int idx = tid; idx < G * HD; idx += kConsumerThreads) {
    const int h = idx / HD, d = idx % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mg[w * WS + h * (HD + 2) + HD]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      M = tag_round(M);
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mg[w * WS + h * (HD + 2) + HD];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L = fmaf(mg[w * WS + h * (HD + 2) + HD + 1], sc, L);
        A = fmaf(mg[w * WS + h * (HD + 2) + d], sc, A);
      }
    } else {
      M = -1e30f;
    }
    st_relaxed(part + idx, tag_word(A, tag));
    if (d == 0) {
      st_relaxed(part + G * HD + 2 * h, tag_word(M, tag));
      st_relaxed(part + G * HD + 2 * h + 1, tag_word(L, tag));
    }
  }
  for (int idx = G * HD + 2 * G + tid; idx < m.part_stride; idx += kConsumerThreads)
    st_relaxed(part + idx, tag_word(0.f, tag));
  if (tr) tr[TR_A_MERGED] = (int64_t)global_timer();
  return stage + nst;
}

// LSE merge of one query head's S attention splits into o (AMK's split-K
// attention followed by its combine step): o = sum_s w_s acc_s / sum_s w_s l_s
// with w_s = 2^(m_s - max_s m_s).  Per chunk of up to NH * SC splits, a
// thread polls SC acc vectors (4 consecutive dims of the head, splits
// hf, hf + NH, ...) while the first threads poll the chunk's (m, l) pairs
// into shared memory; the chunk maximum then gives every weight directly,
// a running (M, L, A) per thread folds the chunks, and the NH subsets are
// merged through shared memory.
// Head size and group are runtime values here (one instance serves every
// model): HD in {64, 128}, so NE in {16, 32} quads and NH in {16, 8} subsets.
__device__ __noinline__ int combine_task(const StepParams& p, Smem& sm, const DevTask t, int stage,
                                         uint32_t task_idx, int64_t* tr) {
  constexpr int SC = 4;                          // acc vectors polled at once per thread
  constexpr int kMaxNH = kConsumerThreads / 16;  // subsets at head size 64
  constexpr int kMaxCH = kMaxNH * SC;            // and splits per chunk
  static_assert((kConsumerThreads / 16) * SC <= kConsumerThreads, "one (m, l) vector per thread");
  static_assert((kConsumerThreads / 16) * SC * 2 + kConsumerThreads * 6 <= kScratchFloats,
                "combine exceeds the scratch");
  const DevModel& m = p.m;
  const int HD = m.head_dim, G = m.group;
  const int NE = HD / 4;                         // dim quads of the head
  const int NH = kConsumerThreads / NE;          // split subsets
  const int CH = NH * SC;                        // splits per chunk
  const int tid = threadIdx.x;
  const int g = t.a0, hh = t.a1, S = m.splits, ps = m.part_stride;
  const int e = tid % NE, hf = tid / NE;
  const uint32_t tag = tag_of(p, t.layer + 1);
  volatile int32_t* abort_flag = &sm.abort_flag;
  const uint32_t* pg = m.part + (int64_t)g * S * ps;
  float* mls = sm.scratch;                  // [CH][2] (m, l) of the head, per split of the chunk
  float* sub = sm.scratch + CH * 2;         // [NH][NE][6] subset states
  float M = -INFINITY, L = 0.f, A[4] = {0.f, 0.f, 0.f, 0.f};
  bool failed = false;
  for (int c0 = 0; c0 < S; c0 += CH) {
    const int nc = min(CH, S - c0);
    uint4 v[SC];
    uint32_t act = 0;
#pragma unroll
    for (int i = 0; i < SC; ++i)
      if (hf + i * NH < nc) act |= 1u << i;
    const uint32_t* base = pg + (int64_t)(c0 + hf) * ps + hh * HD + e * 4;
    const int64_t step = (int64_t)NH * ps;
    if (!failed)
      failed = !poll_tagged<SC>([&](int i) { return base + i * step; }, v, act, tag, m.status,
                                abort_flag, p.timeout_ns, task_idx);
    if (tid < nc && !failed) {
      // (m, l) of heads 2k and 2k + 1 share a vector (G == 1: m, l, pad, pad)
      const uint32_t* mlp = pg + (int64_t)(c0 + tid) * ps + G * HD + (hh >> 1) * 4;
      uint4 mv[1];
      failed = !poll_tagged<1>([&](int) { return mlp; }, mv, 1u, tag, m.status, abort_flag,
                               p.timeout_ns, task_idx);
      mls[tid * 2] = tag_value((hh & 1) ? mv[0].z : mv[0].x);
      mls[tid * 2 + 1] = tag_value((hh & 1) ? mv[0].w : mv[0].y);
    }
    if (consumer_sync_or(failed)) return -1;
    // the chunk maximum (exact in any order): (m, l) pairs two at a time,
    // the loop bound the largest chunk (head size 64)
    float Mc = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxCH; s += 2) {
      if (s >= nc) break;
      const float4 q = *reinterpret_cast<const float4*>(mls + s * 2);
      Mc = fmaxf(Mc, q.x);
      if (s + 1 < nc) Mc = fmaxf(Mc, q.z);
    }
    const float Mn = fmaxf(M, Mc);
    const float a = exp2f(M - Mn);
    L *= a;
#pragma unroll
    for (int c = 0; c < 4; ++c) A[c] *= a;
#pragma unroll
    for (int i = 0; i < SC; ++i) {
      if (!(act & (1u << i))) continue;
      const int s = hf + i * NH;
      const float w = exp2f(mls[s * 2] - Mn);
      L = fmaf(mls[s * 2 + 1], w, L);
      A[0] = fmaf(tag_value(v[i].x), w, A[0]);
      A[1] = fmaf(tag_value(v[i].y), w, A[1]);
      A[2] = fmaf(tag_value(v[i].z), w, A[2]);
      A[3] = fmaf(tag_value(v[i].w), w, A[3]);
    }
    M = Mn;
    consumer_sync();   // mls is refilled by the next chunk
  }
  if (tr) tr[TR_C_WAITED] = (int64_t)global_timer();
  float* mine = sub + (hf * NE + e) * 6;
  mine[0] = M; mine[1] = L; mine[2] = A[0]; mine[3] = A[1]; mine[4] = A[2]; mine[5] = A[3];
  consumer_sync();
  if (hf == 0) {
    float Mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxNH; ++k) {
      if (k >= NH) break;
      Mt = fmaxf(Mt, sub[(k * NE + e) * 6]);
    }
    float Lt = 0.f, At[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kMaxNH; ++k) {
      if (k >= NH) break;
      const float* o = sub + (k * NE + e) * 6;
      const float w = exp2f(o[0] - Mt);   // a subset without splits has M = -inf: weight 0
      Lt = fmaf(o[1], w, Lt);
#pragma unroll
      for (int c = 0; c < 4; ++c) At[c] = fmaf(o[2 + c], w, At[c]);
    }
    const float inv = 1.0f / Lt;
    st_relaxed_v4(m.o + (int64_t)(g * G + hh) * HD + e * 4,
                  make_uint4(tag_word(At[0] * inv, tag), tag_word(At[1] * inv, tag),
                             tag_word(At[2] * inv, tag), tag_word(At[3] * inv, tag)));
  }
  return stage;
}

template <int HD>
__device__ __forceinline__ int attn_dispatch(const StepParams& p, Smem& sm, const DevTask& t,
                                             int stage, uint32_t i, int64_t* tr) {
  switch (p.m.group) {
    case 1: return attn_task<HD, 1>(p, sm, t, stage, i, tr);
    case 2: return attn_task<HD, 2>(p, sm, t, stage, i, tr);
    case 4: return attn_task<HD, 4>(p, sm, t, stage, i, tr);
    default:
      if constexpr (HD == 64) return attn_task<HD, 8>(p, sm, t, stage, i, tr);
      return -1;
  }
}

// Runs the CTA's queue in order.  There is no wait or signal around a task:
// each task polls its own tagged inputs and its stores are the signal.
template <int QKV_FMT, int LM_FMT>
__device__ void consumer_loop(const StepParams& p, Smem& sm, const DevTask* q, int n) {
  const DevModel& m = p.m;
  const int tid = threadIdx.x;
  int stage = 0;   // ring tiles consumed so far
  volatile int32_t* abort_flag = &sm.abort_flag;
  for (int i = 0; i < n; ++i) {
    if (*abort_flag) return;
    const DevTask t = q[i];
    int64_t* tr = p.trace ? trace_row(p, i) : nullptr;
    if (tid == 0) *(volatile int32_t*)&sm.cur_task = i;
    if (tr && tid == 0) {
      tr[TR_C_BEGIN] = (int64_t)global_timer();
      tr[TR_TAG] = t.type | (t.layer << 8);
    }
    int64_t* tr0 = tid == 0 ? tr : nullptr;
    if (t.type == T_ATTN)
      stage = m.head_dim == 128 ? attn_dispatch<128>(p, sm, t, stage, (uint32_t)i, tr0)
                                : attn_dispatch<64>(p, sm, t, stage, (uint32_t)i, tr0);
    else if (t.type == T_COMBINE)
      stage = combine_task(p, sm, t, stage, (uint32_t)i, tr0);
    else if (t.type == T_LMHEAD) stage = gemv_dispatch<LM_FMT>(p, sm, t, stage, (uint32_t)i, tr0);
    else stage = gemv_dispatch<QKV_FMT>(p, sm, t, stage, (uint32_t)i, tr0);
    if (stage < 0) {
      *abort_flag = 1;
      return;
    }
    if (tr && tid == 0) tr[TR_C_DONE] = (int64_t)global_timer();
    consumer_sync();  // every thread's stores issued; scratch free for the next task
    if (tr && tid == 0) tr[TR_C_SIGNALLED] = (int64_t)global_timer();
  }
}

template <int FMT, int LM_FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    // the swizzled KV boxes need 1 KB alignment (slots are 17 KB apart):
    // refuse to run without it
    static_assert(kSlotBytes % 1024 == 0 && kStageBytes % 1024 == 0, "KV slot alignment");
    sm.abort_flag = (smem_addr(&sm.ring[0][0]) & 1023u) ? 1 : 0;
    // the in-flight cap must lie within the ring
    if (p.m.ring_slots < 1 || p.m.ring_slots > kRingSlots) sm.abort_flag = 1;
    if (sm.abort_flag) set_status(p.m.status, ST_CHECK, 0xFFFFFFFFu, SITE_SMEM);
    sm.cur_task = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const int c = blockIdx.x;
  const int q0 = p.m.queue_off[c];
  const int n = p.skip_lm ? p.m.queue_body[c] : p.m.queue_off[c + 1] - q0;
  const DevTask* q = p.m.tasks + q0;
  int64_t* hdr = p.trace ? p.trace + (int64_t)c * (1 + p.trace_stride) * kTraceWords : nullptr;
  if (hdr && tid == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    hdr[0] = (int64_t)global_timer();
    hdr[1] = clock64();
    hdr[4] = n;
    hdr[5] = smid;
  }
  if (tid >= kConsumerThreads) {
    if (tid == kConsumerThreads) producer_loop(p, sm, q, n);
  } else {
    // the step's token: given, or (greedy decoding on the device) the
    // argmax of the previous step's LM-task pairs
    if (p.token_src) {
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int k = tid; k < p.n_lm; k += kConsumerThreads)
        amax_merge(v, i, __uint_as_float(__ldcg(p.token_src + 2 * k)), (int)__ldcg(p.token_src + 2 * k + 1));
      block_amax(v, i, sm.misc);
      if (tid == 0) {
        if (i < 0 || i >= p.m.vocab) {   // no finite logit: report, read a valid row
          set_status(p.m.status, ST_CHECK, 0xFFFFFFFFu, SITE_TOKEN);
          i = 0;
        }
        sm.token = i;
        if (p.token_out && c == 0) *p.token_out = i;
      }
    } else if (tid == 0) {
      sm.token = p.token;
    }
    consumer_sync();
    consumer_loop<FMT, LM_FMT>(p, sm, q, n);
  }
  if (hdr && tid == 0) {
    hdr[2] = (int64_t)global_timer();
    hdr[3] = clock64();
  }
}

// ------------------------------------------------------------- dispatch

using KernelFn = void (*)(StepParams);

static KernelFn pick_kernel(int fmt, int lm_fmt) {
#define AMK_K(a, b) \
  if (fmt == a && lm_fmt == b) return decode_kernel<a, b>;
  AMK_K(AMK_FORMAT_BF16, AMK_FORMAT_BF16)
  AMK_K(AMK_FORMAT_INT8, AMK_FORMAT_INT8)
  AMK_K(AMK_FORMAT_INT8, AMK_FORMAT_BF16)
  AMK_K(AMK_FORMAT_INT4, AMK_FORMAT_INT4)
  AMK_K(AMK_FORMAT_INT4, AMK_FORMAT_BF16)
#undef AMK_K
  return nullptr;
}

const void* decode_kernel_for(int fmt, int lm_fmt) {
  return reinterpret_cast<const void*>(pick_kernel(fmt, lm_fmt));
}

int decode_smem_bytes() { return (int)sizeof(Smem); }

// --------------------------------------------------------- weight packing

struct PackArgs {
  DevMat dst;                 // base already at the layer
  uint16_t* scales_dst;       // int8 row scales of the layer, or null
  const void* w[3];
  const void* s[3];
  const void* z[3];
  int kind, fmt, n_heads, n_kv_heads, head_dim;
};

// packed row -> (source index, source row) or -1.  QKV rows are packed per
// KV head g: its query heads g*G .. g*G+G-1, then k head g, then v head g
// (G = n_heads / n_kv_heads); within a q or k head, row 2i holds dim i and
// row 2i+1 dim i + hd/2, so that each rotate-half RoPE pair sits in one
// thread's pair of rows.  Gate/up rows interleave (gate r, up r).
__device__ int pack_source(const PackArgs& a, int pr, int* row) {
  const DevMat& M = a.dst;
  if (pr >= M.rows) return -1;
  if (a.kind == M_QKV) {
    const int hd = a.head_dim, G = a.n_heads / a.n_kv_heads, gw = (G + 2) * hd;
    const int grp = pr / gw, r = pr % gw, slot = r / hd, i = r % hd;
    const int paired = (i >> 1) + (i & 1) * (hd / 2);
    if (slot < G) {
      *row = (grp * G + slot) * hd + paired;
      return 0;
    }
    *row = grp * hd + (slot == G ? paired : i);
    return slot == G ? 1 : 2;
  }
  if (a.kind == M_GU) {
    *row = pr >> 1;
    return pr & 1;
  }
  *row = pr;
  return 0;
}

// int8 code of physical row pr at k, offset-binary (q + 128); padding is q = 0
__device__ __forceinline__ uint32_t pack_i8_code(const PackArgs& a, int pr, int k) {
  int row = 0;
  const int src = pack_source(a, pr, &row);
  const int8_t q = (src >= 0 && k < a.dst.K) ? static_cast<const int8_t*>(a.w[src])[(int64_t)row * a.dst.K + k] : 0;
  return (uint32_t)(uint8_t)q ^ 0x80u;
}

__global__ void pack_kernel(const PackArgs a) {
  const DevMat& M = a.dst;
  const int chunks = M.Kp / 8;
  const int64_t total = (int64_t)M.rows_padded * chunks;
  if (a.fmt == AMK_FORMAT_INT8) {
    // tensor-core fragment order (act_fragments): 8-byte units
    // ((w * 4 + j) * 32 + lane) * 2 + hf of each 8 x 2048 tile
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
      if (idx < M.rows_padded) {
        int row = 0;
        const int src = pack_source(a, (int)idx, &row);
        a.scales_dst[idx] = src >= 0 ? static_cast<const uint16_t*>(a.s[src])[row] : (uint16_t)0;
      }
      const int64_t per_rb = (int64_t)M.nkt * 2048;
      const int rb = (int)(idx / per_rb);
      const int rem = (int)(idx % per_rb);
      const int kt = rem / 2048, u = rem % 2048;
      const int hf = u & 1, lane = (u >> 1) & 31, j = (u >> 6) & 3, w = u >> 8;
      const int pr0 = rb * 8 + 4 * hf + (lane >> 4), pr1 = pr0 + 2;
      const int k0 = kt * 2048 + 256 * w + 16 * (lane & 15) + 4 * j;
      const uint32_t lo = pack_i8_code(a, pr0, k0) | pack_i8_code(a, pr0, k0 + 1) << 8 |
                          pack_i8_code(a, pr1, k0) << 16 | pack_i8_code(a, pr1, k0 + 1) << 24;
      const uint32_t hi = pack_i8_code(a, pr0, k0 + 2) | pack_i8_code(a, pr0, k0 + 3) << 8 |
                          pack_i8_code(a, pr1, k0 + 2) << 16 | pack_i8_code(a, pr1, k0 + 3) << 24;
      uint8_t* tile = const_cast<uint8_t*>(M.base) + ((int64_t)rb * M.nkt + kt) * M.stage_bytes;
      *reinterpret_cast<uint2*>(tile + (int64_t)u * 8) = make_uint2(lo, hi);
    }
    return;
  }
  if (a.fmt == AMK_FORMAT_INT4) {
    // tensor-core fragment order (gemv_task, u4_fragment): 32-bit words
    // ((w * 4 + j) * 32 + lane) * 4 + rq of each 16 x 2048 tile, then the
    // side data: fp16 scales [16 groups][2][8], u8 zeros [16][2][8] per tile
    const int ng_pad = M.Kp / 128;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
      if (idx < (int64_t)M.rows_padded * ng_pad) {
        const int pr = (int)(idx / ng_pad), gg = (int)(idx % ng_pad);
        int row = 0;
        const int src = pack_source(a, pr, &row);
        uint16_t sc = 0;
        uint8_t zz = 0;
        if (src >= 0 && gg * 128 < M.K) {
          const int ng = M.K / 128, zb = (ng + 1) / 2;
          sc = static_cast<const uint16_t*>(a.s[src])[(int64_t)row * ng + gg];
          const uint8_t zbyte = static_cast<const uint8_t*>(a.z[src])[(int64_t)row * zb + gg / 2];
          zz = (gg & 1) ? (zbyte >> 4) : (zbyte & 15);
        }
        // side data of the tile: scales, then zero points, each ordered
        // [group][row parity][row / 2], so that the 8 rows of one parity in
        // one group (a lane's rows in gemv_task) are contiguous
        uint8_t* side = const_cast<uint8_t*>(M.base) + ((int64_t)(pr / 16) * M.nkt + gg / 16) * M.stage_bytes + kStageBytes;
        const int r16 = pr % 16, si = ((gg % 16) * 2 + (r16 & 1)) * 8 + (r16 >> 1);
        reinterpret_cast<uint16_t*>(side)[si] = sc;
        side[512 + si] = zz;
      }
      const int64_t per_rb = (int64_t)M.nkt * 4096;
      const int rb = (int)(idx / per_rb);
      const int rem = (int)(idx % per_rb);
      const int kt = rem / 4096, u = rem % 4096;
      const int rq = u & 3, lane = (u >> 2) & 31, j = (u >> 7) & 3, w = u >> 9;
      const int pr0 = rb * 16 + 4 * rq + (lane >> 4), pr1 = pr0 + 2;
      const int k0 = kt * 2048 + 256 * w + 16 * (lane & 15) + 4 * j;
      auto nib = [&](int pr, int k) -> uint32_t {
        int row = 0;
        const int src = pack_source(a, pr, &row);
        if (src < 0 || k >= M.K) return 0u;
        const uint8_t b = static_cast<const uint8_t*>(a.w[src])[(int64_t)row * (M.K / 2) + k / 2];
        return (k & 1) ? (uint32_t)(b >> 4) : (uint32_t)(b & 15);
      };
      const uint32_t word = nib(pr0, k0) | nib(pr0, k0 + 2) << 4 | nib(pr1, k0) << 8 | nib(pr1, k0 + 2) << 12 |
                            nib(pr0, k0 + 1) << 16 | nib(pr0, k0 + 3) << 20 | nib(pr1, k0 + 1) << 24 |
                            nib(pr1, k0 + 3) << 28;
      uint8_t* tile = const_cast<uint8_t*>(M.base) + ((int64_t)rb * M.nkt + kt) * M.stage_bytes;
      *reinterpret_cast<uint32_t*>(tile + (int64_t)u * 4) = word;
    }
    return;
  }
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int pr = (int)(idx / chunks);
    const int c = (int)(idx % chunks);
    const int k = c * 8;
    int row = 0;
    const int src = pack_source(a, pr, &row);
    const int rb = pr / M.Rt, r = pr % M.Rt, kt = k / M.Kt, kk = k % M.Kt;
    uint8_t* tile = const_cast<uint8_t*>(M.base) + ((int64_t)rb * M.nkt + kt) * M.stage_bytes;
    const bool live = src >= 0 && k < M.K;
    if (a.fmt == AMK_FORMAT_BF16) {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (live) v = *reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(a.w[src]) + (int64_t)row * M.K + k);
      *reinterpret_cast<uint4*>(tile + ((int64_t)r * M.Kt + kk) * 2) = v;
    }
  }
}

void launch_pack_matrix(int kind, int fmt, const DevMat& dst, int layer, const void* w0,
                        const void* s0, const void* z0, const void* w1, const void* s1,
                        const void* z1, const void* w2, const void* s2, const void* z2,
                        int n_heads, int n_kv_heads, int head_dim, void* stream) {
  PackArgs a;
  a.dst = dst;
  a.dst.base = dst.base + (kind == M_LM ? 0 : (int64_t)layer * dst.layer_bytes);
  a.scales_dst = dst.scales ? const_cast<uint16_t*>(dst.scales) +
                                  (kind == M_LM ? 0 : (int64_t)layer * dst.rows_padded)
                            : nullptr;
  a.w[0] = w0; a.w[1] = w1; a.w[2] = w2;
  a.s[0] = s0; a.s[1] = s1; a.s[2] = s2;
  a.z[0] = z0; a.z[1] = z1; a.z[2] = z2;
  a.kind = kind;
  a.fmt = fmt;
  a.n_heads = n_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  const int64_t total = (int64_t)dst.rows_padded * (dst.Kp / 8);
  int blocks = (int)std::min<int64_t>((total + 255) / 256, 65536);
  pack_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(a);
}

// ---------------------------------------------------------- test aids

// A poll on tagged words nothing writes: must end with ST_TIMEOUT, not hang.
__global__ void watchdog_probe_kernel(uint32_t* scratch, uint64_t timeout_ns) {
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    // scratch[0..4) stay 0 (tag 0 is never written), scratch[16..20) status words
    uint4 v[1];
    poll_tagged<1>([&](int) { return (const uint32_t*)scratch; }, v, 1u, 1u, scratch + 16,
                   &abort_flag, timeout_ns, blockIdx.x);
  }
}

// argmax over n (value bits, index) pairs, one block of 256 threads
__global__ void argmax_pairs_kernel(const uint32_t* pairs, int n, int32_t* out) {
  __shared__ float misc[32];
  float v = -INFINITY;
  int i = 0x7FFFFFFF;
  for (int k = threadIdx.x; k < n; k += kConsumerThreads)
    amax_merge(v, i, __uint_as_float(pairs[2 * k]), (int)pairs[2 * k + 1]);
  block_amax(v, i, misc);
  if (threadIdx.x == 0) *out = i == 0x7FFFFFFF ? -1 : i;
}

void launch_argmax_pairs(const uint32_t* pairs, int n, int32_t* out, void* stream) {
  argmax_pairs_kernel<<<1, kConsumerThreads, 0, (cudaStream_t)stream>>>(pairs, n, out);
}

void launch_watchdog_probe(uint32_t* scratch, uint64_t timeout_ns, void* stream) {
  watchdog_probe_kernel<<<4, 32, 0, (cudaStream_t)stream>>>(scratch, timeout_ns);
}

// element (r, k) of a HF-layout matrix through the kernel's chunk decoders
__global__ void dequant_kernel(int fmt, const void* w, const void* scales, const void* zeros,
                               int rows, int K, float* out) {
  const int64_t total = (int64_t)rows * (K / 8);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / (K / 8)), k = (int)(idx % (K / 8)) * 8;
    float* o = out + (int64_t)r * K + k;
    if (fmt == AMK_FORMAT_BF16) {
      const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(w) + (int64_t)r * K + k);
      o[0] = bf16_lo(v.x); o[1] = bf16_hi(v.x); o[2] = bf16_lo(v.y); o[3] = bf16_hi(v.y);
      o[4] = bf16_lo(v.z); o[5] = bf16_hi(v.z); o[6] = bf16_lo(v.w); o[7] = bf16_hi(v.w);
    } else if (fmt == AMK_FORMAT_INT8) {
      const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const int8_t*>(w) + (int64_t)r * K + k);
      const float s = fp16_bits_to_float(static_cast<const uint16_t*>(scales)[r]);
      const uint32_t a = v.x ^ 0x80808080u, b = v.y ^ 0x80808080u;   // offset-binary, as packed
      const float2 q[4] = {f16x2_to_float2(i8x2_lo(a)), f16x2_to_float2(i8x2_hi(a)),
                           f16x2_to_float2(i8x2_lo(b)), f16x2_to_float2(i8x2_hi(b))};
      for (int i = 0; i < 4; ++i) {
        o[2 * i] = q[i].x * s;
        o[2 * i + 1] = q[i].y * s;
      }
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(w) + (int64_t)r * (K / 2) + k / 2);
      const int ng = K / 128, zb = (ng + 1) / 2, g = k / 128;
      const float s = fp16_bits_to_float(static_cast<const uint16_t*>(scales)[(int64_t)r * ng + g]);
      const uint8_t zbyte = static_cast<const uint8_t*>(zeros)[(int64_t)r * zb + g / 2];
      const uint32_t zc = u4_zc((g & 1) ? (zbyte >> 4) : (zbyte & 15u)), zf = u4_zf(zc);
      // codes k .. k+7 (low nibble = even k) rearranged into one fragment
      // word: its "row R" takes k .. k+3, its "row R + 2" k+4 .. k+7
      auto nb = [&](int i) { return (v >> (4 * i)) & 15u; };
      const uint32_t word = nb(0) | nb(2) << 4 | nb(4) << 8 | nb(6) << 12 | nb(1) << 16 | nb(3) << 20 |
                            nb(5) << 24 | nb(7) << 28;
      uint32_t q[4];
      u4_fragment(word, zc, zf, zc, zf, q);
      const float2 f0 = f16x2_to_float2(q[0]), f2 = f16x2_to_float2(q[2]);   // k, k+1 / k+2, k+3
      const float2 f1 = f16x2_to_float2(q[1]), f3 = f16x2_to_float2(q[3]);   // k+4, k+5 / k+6, k+7
      o[0] = f0.x * s; o[1] = f0.y * s; o[2] = f2.x * s; o[3] = f2.y * s;
      o[4] = f1.x * s; o[5] = f1.y * s; o[6] = f3.x * s; o[7] = f3.y * s;
    }
  }
}

void launch_debug_dequant(int fmt, const void* w, const void* scales, const void* zeros,
                          int rows, int K, float* out, void* stream) {
  const int64_t total = (int64_t)rows * (K / 8);
  int blocks = (int)std::min<int64_t>((total + 255) / 256, 65536);
  if (blocks < 1) blocks = 1;
  dequant_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(fmt, w, scales, zeros, rows, K, out);
}

}  // namespace amk
