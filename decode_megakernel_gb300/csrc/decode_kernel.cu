// Persistent batch-1 decode kernel for sm_103a.
//
// One cooperative CTA per SM walks its static task queue (wait -> dispatch
// -> signal on monotonic counters, the execution model of the
// AutoMegaKernel "Layer 0" VM).  Unlike the pages' design, a CTA is split
// into a producer warp and eight consumer warps:
//   * the producer streams every weight tile (and the KV-cache history) of
//     the CTA's whole queue through a shared-memory ring of kStageBytes
//     stages (128 KB in flight by default) with 1-D TMA bulk copies
//     completing on mbarriers.  Weights never depend on
//     activations, so the producer runs ahead across the counter waits;
//     this hides the per-tile cross-SM synchronisation cost the pages name
//     as the bottleneck on high-bandwidth GPUs (AMK "Experimental results":
//     training-class GPUs).
//   * the consumers wait on counters, keep the activation vector in
//     registers, reduce with warp shuffles, apply the fused epilogues
//     (RoPE + KV append, residual adds, SwiGLU, logits) and signal.
// Every wait is bounded by %globaltimer: on expiry the kernel records a
// status word, lets its own copies land and returns.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_model.hpp"

namespace amk {

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

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

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
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
  uint8_t ring[kStages][kSlotBytes];
  float scratch[kScratchFloats];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float misc[32];
  int32_t abort_flag;
  int32_t flag;
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

// Bounded wait on a counter: true once counter >= target (wrap-safe).
__device__ bool wait_counter(const uint32_t* ctr, uint32_t target, uint32_t* status,
                             volatile int32_t* abort_flag, uint64_t timeout_ns, uint32_t task) {
  const uint64_t t0 = global_timer();
  for (uint32_t spin = 1;; ++spin) {
    if ((int32_t)(ld_acquire(ctr) - target) >= 0) return true;
    if ((spin & 31u) == 0u) {
      if (*abort_flag || ld_relaxed(status) != 0u) return false;
      if (global_timer() - t0 > timeout_ns) {
        set_status(status, ST_TIMEOUT, task, SITE_COUNTER);
        return false;
      }
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
    tt.k = reinterpret_cast<const uint8_t*>(kv_row(m, t.layer, 0, t.a0, 0));
    tt.v = reinterpret_cast<const uint8_t*>(kv_row(m, t.layer, 1, t.a0, 0));
    tt.nst = (tt.t1 - tt.t0 + tt.pps - 1) / tt.pps;
    tt.attn = true;
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

// Producer: one thread streams every tile of the CTA's queue into the ring.
// Whenever no slot is free it prefetches later tiles into L2 (up to
// m.prefetch_tiles ahead of the last copy), so HBM keeps streaming while the
// consumers wait on a counter; the ring copies then hit L2.
__device__ void producer_loop(const StepParams& p, Smem& sm, const DevTask* q, int n) {
  const DevModel& m = p.m;
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_kv = policy_evict_normal();
  volatile int32_t* abort_flag = &sm.abort_flag;
  const uint32_t nslots = (uint32_t)m.ring_slots;
  uint32_t slot = 0, phase = 0;
  uint32_t issued = 0;     // slots that have held a copy
  uint32_t parity = 0;     // parity of each slot's last issued phase
  bool ok = true;
  const int64_t ahead = m.prefetch_tiles;

  int ct = 0, cs = 0;                // copy cursor: task, tile
  TaskTiles ctt;
  bool cvalid = false;
  int pt = 0, ps = 0;                // prefetch cursor
  TaskTiles ptt;
  bool pvalid = false;
  int64_t copied = 0, prefetched = 0;
  int64_t blocked = 0;

  while (ct < n && ok) {
    if (!cvalid) {
      ctt = task_tiles(p, q[ct]);
      cs = 0;
      cvalid = true;
      blocked = 0;
      if (p.trace) trace_row(p, ct)[TR_P_FIRST] = (int64_t)global_timer();
    }
    if (cs == ctt.nst) {
      if (p.trace) {
        int64_t* tr = trace_row(p, ct);
        tr[TR_P_LAST] = (int64_t)global_timer();
        tr[TR_P_BLOCKED] = blocked;
      }
      ++ct;
      cvalid = false;
      continue;
    }
    if (mbar_test_wait(&sm.empty[slot], phase ^ 1u)) {
      if (*abort_flag) { ok = false; break; }
      if (ctt.attn) {
        const int p0 = ctt.t0 + cs * ctt.pps;
        const uint32_t bytes = (uint32_t)(min(ctt.pps, ctt.t1 - p0) * ctt.row);
        mbar_arrive_expect_tx(&sm.full[slot], 2 * bytes);
        bulk_copy_g2s(sm.ring[slot], ctt.k + (int64_t)p0 * ctt.row, bytes, &sm.full[slot], pol_kv);
        bulk_copy_g2s(sm.ring[slot] + kStageBytes / 2, ctt.v + (int64_t)p0 * ctt.row, bytes,
                      &sm.full[slot], pol_kv);
      } else {
        mbar_arrive_expect_tx(&sm.full[slot], ctt.bytes);
        bulk_copy_g2s(sm.ring[slot], ctt.k + (int64_t)cs * ctt.stride, ctt.bytes, &sm.full[slot], pol_w);
      }
      issued |= 1u << slot;
      parity = (parity & ~(1u << slot)) | (phase << slot);
      if (++slot == nslots) { slot = 0; phase ^= 1u; }
      ++cs;
      ++copied;
      continue;
    }
    // no free slot: prefetch a later tile into L2 while there is one in reach
    if (prefetched < copied) {  // the copies overtook the prefetches
      pt = ct;
      ps = cs;
      ptt = ctt;
      pvalid = true;
      prefetched = copied;
    }
    if (pt < n && prefetched < copied + ahead) {
      if (!pvalid) {
        ptt = task_tiles(p, q[pt]);
        ps = 0;
        pvalid = true;
      }
      if (ps >= ptt.nst) {
        ++pt;
        pvalid = false;
        continue;
      }
      if (ptt.attn) {
        const int p0 = ptt.t0 + ps * ptt.pps;
        const uint32_t bytes = (uint32_t)(min(ptt.pps, ptt.t1 - p0) * ptt.row);
        prefetch_l2(ptt.k + (int64_t)p0 * ptt.row, bytes);
        prefetch_l2(ptt.v + (int64_t)p0 * ptt.row, bytes);
      } else {
        prefetch_l2(ptt.k + (int64_t)ps * ptt.stride, ptt.bytes);
      }
      ++ps;
      ++prefetched;
      continue;
    }
    // nothing to issue: wait for the oldest slot to be released
    const int64_t c0 = p.trace ? clock64() : 0;
    ok = wait_phase(&sm.empty[slot], phase ^ 1u, m.status, abort_flag, p.timeout_ns, ct,
                    SITE_EMPTY) && !*abort_flag;
    if (p.trace) blocked += clock64() - c0;
  }
  // Every copy this CTA issued must land before its shared memory goes away.
  // Consumers normally wait for all of them already; when they stop early
  // (a failed wait anywhere) this is what keeps the CTA from exiting with
  // a copy in flight.
  for (int s = 0; s < kStages; ++s) {
    if (!(issued & (1u << s))) continue;
    const uint32_t par = (parity >> s) & 1u;
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(&sm.full[s], par)) {
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

// int8 byte i of (w ^ 0x80808080) placed under the exponent of 2^23: 2^23 + q + 128
__device__ __forceinline__ float i8_biased(uint32_t w_xor80, int i) {
  return __uint_as_float(__byte_perm(w_xor80, 0x4B000000u, 0x7440u | (uint32_t)i));
}
__device__ __forceinline__ float i8_at(uint32_t w_xor80, int i) {
  return i8_biased(w_xor80, i) - 8388736.0f;
}

// int4 nibble i of w as float (exact)
__device__ __forceinline__ float u4_at(uint32_t w, int i) {
  return __uint_as_float(0x4B000000u | ((w >> (4 * i)) & 0xFu)) - 8388608.0f;
}

// int4 nibble i of w, left where it sits, under the exponent of 2^23:
// 2^23 + q * 2^s with s = u4_shift(i); (value - 2^23) is exact.
__device__ __forceinline__ constexpr int u4_shift(int i) { return i < 5 ? 4 * i : 4 * i - 12; }
__device__ __forceinline__ float u4_biased(uint32_t w, uint32_t w_hi, int i) {
  return i < 5 ? __uint_as_float(0x4B000000u | (w & (0xFu << (4 * i))))
               : __uint_as_float(0x4B000000u | (w_hi & (0xFu << (4 * i - 12))));
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
__device__ __forceinline__ bool mbar_try_wait32(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
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
// as four pairs.  QKV, gate/up and LM head take rmsnorm(x) * w_norm; O takes
// o; down takes a.
template <int NKT>
__device__ __forceinline__ void load_activation(const StepParams& p, Smem& sm, const DevTask& t,
                                                const DevMat& M, int chunk, float2 (&h)[NKT][4]) {
  const DevModel& m = p.m;
  const int tid = threadIdx.x;
  const bool norm = t.type == T_QKV || t.type == T_GATEUP || t.type == T_LMHEAD;
  const bool from_embed = t.type == T_QKV && t.layer == 0;
  const float* src = t.type == T_OPROJ ? m.o : t.type == T_DOWN ? m.a : m.x;
  const uint16_t* emb = m.embed + (int64_t)p.token * m.hidden;
  float ss = 0.f;
#pragma unroll
  for (int kt = 0; kt < NKT; ++kt) {
    const int k = kt * M.Kt + chunk * 8;
    if (k < M.K) {  // K is a multiple of 8
      if (from_embed) load8_bf16(emb + k, h[kt]);
      else load8_f32(src + k, h[kt]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) h[kt][i] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(h[kt][i].x, h[kt][i].x, fmaf(h[kt][i].y, h[kt][i].y, ss));
  }
  if (!norm) return;
  // threads tid < Kt/8 hold every chunk once: their squares sum to sum(x^2)
  const int cpr = 1 << M.cpr_shift;
  ss = warp_sum(tid < cpr ? ss : 0.f);
  if ((tid & 31) == 0) sm.misc[tid >> 5] = ss;
  consumer_sync();
  float tot = 0.f;
  for (int w = 0; w < (cpr >> 5); ++w) tot += sm.misc[w];
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
    const uint2 w = lds64(a);
    const uint32_t x = w.x ^ 0x80808080u, y = w.y ^ 0x80808080u;
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
    acc = __ffma2_rn(__fadd2_rn(make_float2(i8_biased(x, 0), i8_biased(x, 1)), bias), h[0], acc);
    acc = __ffma2_rn(__fadd2_rn(make_float2(i8_biased(x, 2), i8_biased(x, 3)), bias), h[1], acc);
    acc = __ffma2_rn(__fadd2_rn(make_float2(i8_biased(y, 0), i8_biased(y, 1)), bias), h[2], acc);
    acc = __ffma2_rn(__fadd2_rn(make_float2(i8_biased(y, 2), i8_biased(y, 3)), bias), h[3], acc);
    return acc;
  }
}

// int4 chunk: h holds act * 2^-s per element position (see u4_shift), hs the
// chunk's plain sum; returns acc + s_g * (sum(q * act) - z_g * sum(act)).
__device__ __forceinline__ float chunk_dot_u4(uint32_t a, uint32_t side_s, uint32_t side_z,
                                              const float2 (&h)[4], float hs, float acc) {
  const uint32_t w = lds32(a);
  const float s = fp16_bits_to_float((uint16_t)lds16(side_s));
  const float z = (float)lds8(side_z);
  const uint32_t w_hi = w >> 12;
  const float2 bias = make_float2(-8388608.0f, -8388608.0f);
  float2 d = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __fadd2_rn(make_float2(u4_biased(w, w_hi, 2 * i), u4_biased(w, w_hi, 2 * i + 1)), bias);
    d = __ffma2_rn(q, h[i], d);
  }
  return fmaf(s, fmaf(-z, hs, d.x + d.y), acc);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

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

  float2 h[NKT][4];
  load_activation<NKT>(p, sm, t, M, chunk, h);
  float hs[NKT];  // int4: per-chunk activation sums, then activations pre-scaled by 2^-s
  if constexpr (FMT == AMK_FORMAT_INT4) {
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt) {
      hs[kt] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hs[kt] += h[kt][i].x + h[kt][i].y;
        h[kt][i].x *= 1.0f / (float)(1 << u4_shift(2 * i));        // exact: power of two
        h[kt][i].y *= 1.0f / (float)(1 << u4_shift(2 * i + 1));
      }
    }
  }

  // layer-0 QKV tasks also initialise their slice of the residual stream
  if (t.type == T_QKV && t.layer == 0) {
    const uint16_t* emb = m.embed + (int64_t)p.token * m.hidden;
    for (int e = t.a2 + tid; e < t.a3; e += kConsumerThreads)
      m.x[e] = __uint_as_float((uint32_t)emb[e] << 16);
  }

  const uint32_t ring0 = smem_addr(&sm.ring[0][0]);
  const uint32_t full0 = smem_addr(&sm.full[0]);
  const uint32_t empty0 = smem_addr(&sm.empty[0]);
  const uint32_t off0 = (uint32_t)(((rsub << cs) + chunk) * EB);   // pass 0 chunk
  const uint32_t pass_stride = (uint32_t)((rpp << cs) * EB);       // rows between passes
  // int4 side data: fp16 scales [Rt][Kt/128] then u8 zeros [Rt][Kt/128]
  const int ngt = M.Kt >> 7;
  const uint32_t side_s0 = kStageBytes + (uint32_t)((rsub * ngt + (chunk >> 4)) * 2);
  const uint32_t side_z0 = kStageBytes + (uint32_t)(M.Rt * ngt * 2 + rsub * ngt + (chunk >> 4));
  const uint32_t nslots = (uint32_t)m.ring_slots;
  uint32_t slot = (uint32_t)stage % nslots, phase = ((uint32_t)stage / nslots) & 1u;
  bool failed = false;
  int64_t starved = 0;

  float* red = sm.scratch;
  const int nrb = t.a1 - t.a0;
  for (int rb = 0; rb < nrb; ++rb) {
    float2 acc2[FMT == AMK_FORMAT_INT4 ? 1 : P];
    float acc1[FMT == AMK_FORMAT_INT4 ? P : 1];
#pragma unroll
    for (int i = 0; i < (FMT == AMK_FORMAT_INT4 ? 1 : P); ++i) acc2[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < (FMT == AMK_FORMAT_INT4 ? P : 1); ++i) acc1[i] = 0.f;
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt) {
      if (!failed)
        failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
      if (!failed) {
        const uint32_t tile = ring0 + slot * kSlotBytes;
#pragma unroll
        for (int ps = 0; ps < P; ++ps) {
          if constexpr (FMT == AMK_FORMAT_INT4)
            acc1[ps] = chunk_dot_u4(tile + off0 + ps * pass_stride,
                                    tile + side_s0 + (uint32_t)(ps * rpp * ngt * 2),
                                    tile + side_z0 + (uint32_t)(ps * rpp * ngt), h[kt], hs[kt],
                                    acc1[ps]);
          else
            acc2[ps] = chunk_dot<FMT>(tile + off0 + ps * pass_stride, h[kt], acc2[ps]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive32(empty0 + slot * 8);
      if (++slot == nslots) { slot = 0; phase ^= 1u; }
    }
    float v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      if constexpr (FMT == AMK_FORMAT_INT4) v[i] = acc1[i];
      else v[i] = acc2[i].x + acc2[i].y;
    }
    const float tot = transpose_reduce<P>(v, lane);
    constexpr int kLaneStride = 32 / P;
    if ((lane & (kLaneStride - 1)) == 0) {
      const int ps = lane / kLaneStride;
      red[(rb * M.Rt + ps * rpp + rsub) * 8 + wg] = tot;
    }
  }

  if (tr) tr[TR_C_STARVED] = starved;
  if (consumer_sync_or(failed)) return -1;

  // epilogue: one row (or one row pair) per thread
  const int nrows = nrb * M.Rt;
  const int row0 = t.a0 * M.Rt;
  const int nwg = 1 << wpg_shift;
  auto row_sum = [&](int r) {
    float y = 0.f;
    for (int w = 0; w < nwg; ++w) y += red[r * 8 + w];
    return y;
  };
  if (t.type == T_QKV || t.type == T_GATEUP) {
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
        m.a[R >> 1] = silu(y0) * y1;
        continue;
      }
      const int hd = m.head_dim, half = hd >> 1;
      const int qd = m.n_heads * hd, kvd = m.n_kv_heads * hd;
      if (R < qd + kvd) {
        // rotate-half RoPE pair (i, i + hd/2) at position pos
        const bool is_q = R < qd;
        const int rr = is_q ? R : R - qd;
        const int head = rr / hd, i = (rr % hd) >> 1;
        const float2 cs2 = m.rope[(int64_t)p.pos * half + i];
        const float a = y0 * cs2.x - y1 * cs2.y;
        const float b = y1 * cs2.x + y0 * cs2.y;
        if (is_q) {
          m.q[head * hd + i] = a;
          m.q[head * hd + half + i] = b;
        } else {
          uint16_t* kr = const_cast<uint16_t*>(kv_row(m, t.layer, 0, head, p.pos));
          kr[i] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
          kr[half + i] = __bfloat16_as_ushort(__float2bfloat16_rn(b));
        }
      } else {
        const int vr = R - qd - kvd;
        uint16_t* vrow = const_cast<uint16_t*>(kv_row(m, t.layer, 1, vr / hd, p.pos));
        vrow[vr % hd] = __bfloat16_as_ushort(__float2bfloat16_rn(y0));
        vrow[vr % hd + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(y1));
      }
    }
  } else {
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
      } else {  // O projection / down projection: residual add on owned rows
        m.x[R] = __ldcg(m.x + R) + y;
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

// Split-K GQA attention of one KV head over one context split.  Per ring
// stage a warp takes NPW cached positions; scores for R positions x G heads
// are reduced in one transposed warp reduction, then the warp's running
// softmax state is rescaled once per block of R positions.  The last split
// of a KV head to finish merges all splits (LSE combine) into o.
// HD: head_dim (a lane owns HD/32 dims of every head), G: query heads per KV head.
template <int HD, int G>
__device__ __noinline__ int attn_task(const StepParams& p, Smem& sm, const DevTask t, int stage,
                                      uint32_t task_idx, int64_t* tr) {
  constexpr int DPL = HD / 32;
  constexpr int PPS = (kStageBytes / 2) / (HD * 2);   // positions per stage
  constexpr int NPW = PPS / kConsumerWarps;           // positions per warp per stage
  constexpr int R = (32 / G) < NPW ? (32 / G) : NPW;  // positions per block
  constexpr int V = R * G;                            // scores per block
  constexpr int LS = 32 / V;                          // lanes per score after the reduction
  const DevModel& m = p.m;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = t.a0, j = t.a1;
  volatile int32_t* abort_flag = &sm.abort_flag;

  // queries of the group, pre-scaled so that scores are in log2 units
  const float qscale = 1.4426950408889634f * rsqrtf((float)HD);
  float qr[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int d = 0; d < DPL; ++d)
      qr[h][d] = __ldcg(m.q + (int64_t)(g * G + h) * HD + lane * DPL + d) * qscale;
  float mx[G], l[G], acc[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mx[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[h][d] = 0.f;
  }

  // one block of `np` (<= R) positions whose K and V rows this lane holds
  auto block = [&](const float (&kf)[R][DPL], const float (&vf)[R][DPL], int np) {
    float sc[V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float s = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) s = fmaf(qr[h][d], kf[r][d], s);
        sc[r * G + h] = s;
      }
    float s = transpose_reduce<V>(sc, lane);   // score of (r, h) = lane / LS
    const int idx = lane / LS;
    const int my_r = idx / G, my_h = idx % G;
    if (my_r >= np) s = -INFINITY;               // positions past the end of the split
    // block maximum per head: reduce over the lanes holding other positions
    float bm = s;
#pragma unroll
    for (int msk = LS * G; msk < 32; msk <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, msk));
    float alpha[G], mnew[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float b = __shfl_sync(0xFFFFFFFFu, bm, h * LS);
      mnew[h] = fmaxf(mx[h], b);
      alpha[h] = exp2f(mx[h] - mnew[h]);
    }
    float mine = mnew[0];
#pragma unroll
    for (int h = 1; h < G; ++h) mine = my_h == h ? mnew[h] : mine;
    const float pe = exp2f(s - mine);            // 0 for the padding positions
    float bs = pe;
#pragma unroll
    for (int msk = LS * G; msk < 32; msk <<= 1) bs += __shfl_xor_sync(0xFFFFFFFFu, bs, msk);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l[h] = fmaf(l[h], alpha[h], __shfl_sync(0xFFFFFFFFu, bs, h * LS));
      mx[h] = mnew[h];
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[h][d] *= alpha[h];
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = __shfl_sync(0xFFFFFFFFu, pe, (r * G + h) * LS);
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[h][d] = fmaf(pr, vf[r][d], acc[h][d]);
      }
  };
  auto unpack = [&](uint32_t lo, uint32_t hi, float* f) {
    if constexpr (DPL == 4) {
      f[0] = bf16_lo(lo); f[1] = bf16_hi(lo); f[2] = bf16_lo(hi); f[3] = bf16_hi(hi);
    } else {
      f[0] = bf16_lo(lo); f[1] = bf16_hi(lo);
    }
  };

  const uint32_t ring0 = smem_addr(&sm.ring[0][0]);
  const uint32_t full0 = smem_addr(&sm.full[0]);
  const uint32_t empty0 = smem_addr(&sm.empty[0]);
  const uint32_t nslots = (uint32_t)m.ring_slots;
  uint32_t slot = (uint32_t)stage % nslots, phase = ((uint32_t)stage / nslots) & 1u;
  bool failed = false;
  int64_t starved = 0;
  int t0, t1;
  attn_range(p.pos, m.splits, j, &t0, &t1);
  int nst = 0;
  for (int s0 = t0; s0 < t1; s0 += PPS) {
    const int np = min(PPS, t1 - s0);
    ++nst;
    if (!failed)
      failed = !wait_full(full0 + slot * 8, phase, p, abort_flag, task_idx, tr ? &starved : nullptr);
    if (!failed) {
      const uint32_t kt = ring0 + slot * kSlotBytes;
      const uint32_t vt = kt + kStageBytes / 2;
      // warp w takes positions [w*NPW, (w+1)*NPW) of the stage
#pragma unroll
      for (int b0 = 0; b0 < NPW; b0 += R) {
        const int first = warp * NPW + b0;
        const int nb = min(R, np - first);
        if (nb > 0) {
          float kf[R][DPL], vf[R][DPL];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int pi = min(first + r, np - 1);
            const uint32_t ko = kt + (uint32_t)((pi * HD + lane * DPL) * 2);
            const uint32_t vo = vt + (uint32_t)((pi * HD + lane * DPL) * 2);
            if constexpr (DPL == 4) {
              const uint2 kw = lds64(ko), vw = lds64(vo);
              unpack(kw.x, kw.y, kf[r]);
              unpack(vw.x, vw.y, vf[r]);
            } else {
              unpack(lds32(ko), 0u, kf[r]);
              unpack(lds32(vo), 0u, vf[r]);
            }
          }
          block(kf, vf, nb);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive32(empty0 + slot * 8);
    if (++slot == nslots) { slot = 0; phase ^= 1u; }
  }
  // the current position, written this step by the QKV tasks
  if (!failed && j == m.splits - 1 && warp == 0) {
    float kf[R][DPL], vf[R][DPL];
    const uint16_t* kr = kv_row(m, t.layer, 0, g, p.pos) + lane * DPL;
    const uint16_t* vr = kv_row(m, t.layer, 1, g, p.pos) + lane * DPL;
    if constexpr (DPL == 4) {
      const uint2 kw = __ldcg(reinterpret_cast<const uint2*>(kr));
      const uint2 vw = __ldcg(reinterpret_cast<const uint2*>(vr));
      unpack(kw.x, kw.y, kf[0]);
      unpack(vw.x, vw.y, vf[0]);
    } else {
      unpack(__ldcg(reinterpret_cast<const unsigned int*>(kr)), 0u, kf[0]);
      unpack(__ldcg(reinterpret_cast<const unsigned int*>(vr)), 0u, vf[0]);
    }
#pragma unroll
    for (int r = 1; r < R; ++r)
#pragma unroll
      for (int d = 0; d < DPL; ++d) { kf[r][d] = kf[0][d]; vf[r][d] = vf[0][d]; }
    block(kf, vf, 1);
  }

  if (tr) {
    tr[TR_C_STARVED] = starved;
    tr[TR_A_STAGES] = (int64_t)global_timer();
  }
  // merge the eight warps' partial softmax states
  float* mg = sm.scratch;  // [warp][G][HD + 2]
  constexpr int WS = G * (HD + 2);
  static_assert(kConsumerWarps * WS <= kScratchFloats, "warp merge exceeds the scratch");
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int d = 0; d < DPL; ++d) mg[warp * WS + h * (HD + 2) + lane * DPL + d] = acc[h][d];
    if (lane == 0) {
      mg[warp * WS + h * (HD + 2) + HD] = mx[h];
      mg[warp * WS + h * (HD + 2) + HD + 1] = l[h];
    }
  }
  if (consumer_sync_or(failed)) return -1;
  float* part = m.part + (int64_t)(g * m.splits + j) * m.part_stride;
  for (int idx = tid; idx < G * HD; idx += kConsumerThreads) {
    const int h = idx / HD, d = idx % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mg[w * WS + h * (HD + 2) + HD]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mg[w * WS + h * (HD + 2) + HD];
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L = fmaf(mg[w * WS + h * (HD + 2) + HD + 1], sc, L);
        A = fmaf(mg[w * WS + h * (HD + 2) + d], sc, A);
      }
    }
    part[h * (HD + 2) + d] = A;
    if (d == 0) {
      part[h * (HD + 2) + HD] = M;
      part[h * (HD + 2) + HD + 1] = L;
    }
  }
  consumer_sync();
  if (tr) tr[TR_A_MERGED] = (int64_t)global_timer();

  // ticket: the last split of this KV head to arrive merges all splits
  if (tid == 0) {
    const uint32_t old = atom_add_acq_rel(m.counters + t.signal, 1u);
    sm.flag = (old + 1u == p.epoch * (uint32_t)m.splits) ? 1 : 0;
  }
  consumer_sync();
  if (tr) tr[TR_A_TICKET] = (int64_t)global_timer();
  if (sm.flag) {
    // LSE merge of the S splits of this KV head, in chunks of up to SC splits.
    // Per chunk every load is issued at once (the (m, l) pairs by one thread
    // each, every output element's SC partial sums by its thread), so a
    // chunk costs one L2 round trip; a running (M, L, A) per element folds
    // the chunks together.  Shared memory: 2 * SC * G floats.
    constexpr int SC = 24;
    constexpr int EPT = (G * HD + kConsumerThreads - 1) / kConsumerThreads;  // elements per thread
    static_assert(SC * G <= kConsumerThreads, "one (m, l) pair per thread");
    const int S = m.splits;
    const float* pg = m.part + (int64_t)g * S * m.part_stride;
    float* ml = sm.scratch;  // [SC][G] maxima, then [SC][G] normalisers
    float runM[EPT], runL[EPT], runA[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) { runM[e] = -INFINITY; runL[e] = 0.f; runA[e] = 0.f; }
    for (int c0 = 0; c0 < S; c0 += SC) {
      const int sc = min(SC, S - c0);
      float mv = 0.f, lv = 0.f;
      if (tid < sc * G) {
        const float* pp = pg + (int64_t)(c0 + tid / G) * m.part_stride + (tid % G) * (HD + 2) + HD;
        mv = __ldcg(pp);
        lv = __ldcg(pp + 1);
      }
      float av[EPT][SC];
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int idx = tid + e * kConsumerThreads;
        const int h = idx / HD, d = idx % HD;
#pragma unroll
        for (int s2 = 0; s2 < SC; ++s2)
          av[e][s2] = (idx < G * HD && s2 < sc)
                          ? __ldcg(pg + (int64_t)(c0 + s2) * m.part_stride + h * (HD + 2) + d) : 0.f;
      }
      if (tid < sc * G) {
        ml[tid] = mv;
        ml[SC * G + tid] = lv;
      }
      consumer_sync();
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int idx = tid + e * kConsumerThreads;
        if (idx >= G * HD) continue;
        const int h = idx / HD;
        float Mc = -INFINITY;
        for (int s2 = 0; s2 < sc; ++s2) Mc = fmaxf(Mc, ml[s2 * G + h]);
        if (Mc == -INFINITY) continue;
        float Lc = 0.f, Ac = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < SC; ++s2) {
          if (s2 < sc) {
            const float ms = ml[s2 * G + h];
            const float w = ms == -INFINITY ? 0.f : exp2f(ms - Mc);
            Lc = fmaf(ml[SC * G + s2 * G + h], w, Lc);
            Ac = fmaf(av[e][s2], w, Ac);
          }
        }
        const float Mn = fmaxf(runM[e], Mc);
        const float wr = runM[e] == -INFINITY ? 0.f : exp2f(runM[e] - Mn);
        const float wc = exp2f(Mc - Mn);
        runL[e] = runL[e] * wr + Lc * wc;
        runA[e] = runA[e] * wr + Ac * wc;
        runM[e] = Mn;
      }
      consumer_sync();  // the next chunk reuses ml
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int idx = tid + e * kConsumerThreads;
      if (idx < G * HD) m.o[(int64_t)(g * G + idx / HD) * HD + idx % HD] = runA[e] / runL[e];
    }
    consumer_sync();
    if (tid == 0) red_release_add(m.counters + t.a2, 1u);
    if (tr) tr[TR_A_COMBINED] = (int64_t)global_timer();
  }
  return stage + nst;
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

template <int QKV_FMT, int LM_FMT>
__device__ void consumer_loop(const StepParams& p, Smem& sm, const DevTask* q, int n) {
  const DevModel& m = p.m;
  const int tid = threadIdx.x;
  int stage = 0;
  volatile int32_t* abort_flag = &sm.abort_flag;
  for (int i = 0; i < n; ++i) {
    const DevTask t = q[i];
    bool failed = false;
    int64_t* tr = p.trace ? trace_row(p, i) : nullptr;
    if (tr && tid == 0) {
      tr[TR_C_BEGIN] = (int64_t)global_timer();
      tr[TR_TAG] = t.type | (t.layer << 8);
    }
    if (t.wait_counter >= 0 && tid == 0)
      failed = !wait_counter(m.counters + t.wait_counter, p.epoch * t.wait_count, m.status,
                             abort_flag, p.timeout_ns, (uint32_t)i);
    if (consumer_sync_or(failed)) {
      *abort_flag = 1;
      return;
    }
    if (tr && tid == 0) tr[TR_C_WAITED] = (int64_t)global_timer();
    int64_t* tr0 = tid == 0 ? tr : nullptr;
    if (t.type == T_ATTN)
      stage = m.head_dim == 128 ? attn_dispatch<128>(p, sm, t, stage, (uint32_t)i, tr0)
                                : attn_dispatch<64>(p, sm, t, stage, (uint32_t)i, tr0);
    else if (t.type == T_LMHEAD) stage = gemv_dispatch<LM_FMT>(p, sm, t, stage, (uint32_t)i, tr0);
    else stage = gemv_dispatch<QKV_FMT>(p, sm, t, stage, (uint32_t)i, tr0);
    if (stage < 0) {
      *abort_flag = 1;
      return;
    }
    if (tr && tid == 0) tr[TR_C_DONE] = (int64_t)global_timer();
    if (t.type != T_ATTN) {
      consumer_sync();  // epilogue stores done; scratch free for the next task
      if (tid == 0 && t.signal >= 0) red_release_add(m.counters + t.signal, 1u);
    }
    if (tr && tid == 0) tr[TR_C_SIGNALLED] = (int64_t)global_timer();
  }
}

template <int FMT, int LM_FMT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort_flag = 0;
    sm.flag = 0;
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

// packed row -> (source index, source row) or -1
__device__ int pack_source(const PackArgs& a, int pr, int* row) {
  const DevMat& M = a.dst;
  if (pr >= M.rows) return -1;
  if (a.kind == M_QKV) {
    const int hd = a.head_dim, qd = a.n_heads * hd, kvd = a.n_kv_heads * hd;
    if (pr < qd + kvd) {
      const int rr = pr < qd ? pr : pr - qd;
      const int i = rr % hd;
      *row = rr / hd * hd + (i >> 1) + (i & 1) * (hd / 2);
      return pr < qd ? 0 : 1;
    }
    *row = pr - qd - kvd;
    return 2;
  }
  if (a.kind == M_GU) {
    *row = pr >> 1;
    return pr & 1;
  }
  *row = pr;
  return 0;
}

__global__ void pack_kernel(const PackArgs a) {
  const DevMat& M = a.dst;
  const int chunks = M.Kp / 8;
  const int64_t total = (int64_t)M.rows_padded * chunks;
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
    } else if (a.fmt == AMK_FORMAT_INT8) {
      uint2 v = make_uint2(0, 0);
      if (live) v = *reinterpret_cast<const uint2*>(
                    static_cast<const int8_t*>(a.w[src]) + (int64_t)row * M.K + k);
      *reinterpret_cast<uint2*>(tile + (int64_t)r * M.Kt + kk) = v;
      if (c == 0)
        a.scales_dst[pr] = src >= 0 ? static_cast<const uint16_t*>(a.s[src])[row] : (uint16_t)0;
    } else {
      uint32_t v = 0;
      if (live) v = *reinterpret_cast<const uint32_t*>(
                    static_cast<const uint8_t*>(a.w[src]) + (int64_t)row * (M.K / 2) + k / 2);
      *reinterpret_cast<uint32_t*>(tile + ((int64_t)r * M.Kt + kk) / 2) = v;
      if ((kk & 127) == 0) {
        const int ngt = M.Kt >> 7, gl = kk >> 7, gg = k >> 7;
        uint16_t sc = 0;
        uint8_t zz = 0;
        if (live) {
          const int ng = M.K / 128, zb = (ng + 1) / 2;
          sc = static_cast<const uint16_t*>(a.s[src])[(int64_t)row * ng + gg];
          const uint8_t zbyte = static_cast<const uint8_t*>(a.z[src])[(int64_t)row * zb + gg / 2];
          zz = (gg & 1) ? (zbyte >> 4) : (zbyte & 15);
        }
        uint8_t* side = tile + kStageBytes;
        reinterpret_cast<uint16_t*>(side)[r * ngt + gl] = sc;
        side[M.Rt * ngt * 2 + r * ngt + gl] = zz;
      }
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

// A wait on a counter nothing signals: must end with ST_TIMEOUT, not hang.
__global__ void watchdog_probe_kernel(uint32_t* scratch, uint64_t timeout_ns) {
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    // scratch[0] counter (stays 0), scratch[16..20) status words
    wait_counter(scratch, 1u, scratch + 16, &abort_flag, timeout_ns, blockIdx.x);
  }
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
      const uint32_t a = v.x ^ 0x80808080u, b = v.y ^ 0x80808080u;
      for (int i = 0; i < 4; ++i) o[i] = i8_at(a, i) * s;
      for (int i = 0; i < 4; ++i) o[4 + i] = i8_at(b, i) * s;
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(w) + (int64_t)r * (K / 2) + k / 2);
      const int ng = K / 128, zb = (ng + 1) / 2, g = k / 128;
      const float s = fp16_bits_to_float(static_cast<const uint16_t*>(scales)[(int64_t)r * ng + g]);
      const uint8_t zbyte = static_cast<const uint8_t*>(zeros)[(int64_t)r * zb + g / 2];
      const float z = (float)((g & 1) ? (zbyte >> 4) : (zbyte & 15));
      for (int i = 0; i < 8; ++i) o[i] = (u4_at(v, i) - z) * s;
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
