// Tensor-core prefill kernels (see prefill.hpp for the algorithm).
//
// GEMM: 128-token x BN-row output tiles (BN = 256, or 224 where that fills
// the SMs better: prefill_gemm_bn), a persistent CTA per SM taking every
// gridDim-th tile.  Warp 0 (one thread)
// streams k blocks of the activation parts and the weight slice through a
// kPfStages-deep ring with TMA; warp 1 (one thread) issues tcgen05.mma
// (kind::f16, bf16 x bf16 -> fp32, M 128, N 256, K 16) into one of two
// 256-column TMEM accumulators, a fresh one every kPfSegKB k blocks, and
// releases each stage with tcgen05.commit; eight epilogue warps (two per
// TMEM lane quarter, 128 columns each) read each finished segment back
// (tcgen05.ld, one token row per thread), add it into fp32 registers, hand
// the buffer back, and at the end run the fused epilogue.  Every wait is bounded by the context's watchdog
// limit; a timeout records ST_TIMEOUT in the status words.
//
// Attention: flash-attention over the KV cache with mma.sync (bf16 in,
// fp32 accumulate), one CTA per (16 x attn_groups(G) query tokens, KV head),
// launched longest first, two CTAs per SM; one warp per (query head of the
// group, 16 tokens), all warps sharing the CTA's K,V tiles; q and P split into bf16 hi + lo as in the decode
// kernel's attention (softmax weights and pre-scaled scores need no more:
// the attention's K,V are bf16 already).
#include "device_model.hpp"
#include "prefill.hpp"
#include "ptx.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace amk {

namespace {

constexpr uint32_t kPfATile = kPfBM * kPfBK * 2;   // 16 KB: 128 tokens x 64 k, bf16
constexpr int kPfTmemCols = 2 * kPfBN;             // two accumulator buffers kPfBN columns apart

// one stage: the activation parts (128 x 64 bf16 each) and the weight
// slice (BN x 64 bf16); as many stages as fit in 200 KB of shared memory
template <int PARTS, int BN>
struct GemmShape {
  static constexpr uint32_t kBTile = (uint32_t)BN * kPfBK * 2;   // BN rows x 64 k, bf16
  static constexpr int kStages = (200 * 1024) / (PARTS * (int)kPfATile + (int)kBTile);
  static constexpr int kEpiCols = BN / (kPfEpiWarps / 4);       // accumulator columns per epilogue warp
};

template <int PARTS, int BN>
struct __align__(1024) GemmSmem {
  static constexpr int S = GemmShape<PARTS, BN>::kStages;
  uint8_t a[S][PARTS][kPfATile];
  uint8_t w[S][GemmShape<PARTS, BN>::kBTile];
  uint64_t full[S], empty[S];
  uint64_t acc_full[2], acc_empty[2];   // TMEM accumulator buffers: segment done / drained
  uint32_t tmem;
  uint32_t failed;
};




// bounded wait for a phase of an mbarrier: false after limit_ns
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait32(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (!mbar_try_wait32(bar, parity))
    if (global_timer() - t0 > limit_ns) return false;
  return true;
}

// Programmatic dependent launch: every prefill kernel is launched with
// programmatic stream serialisation, so it may start (and run its prologue:
// barrier setup, tensor-memory allocation) while the kernel before it on the
// stream drains.  pdl_wait blocks until that kernel has completed and its
// writes are visible; each kernel calls it before its first access to
// global memory that another kernel writes or reads.  pdl_launch_dependents
// lets the next kernel start launching once every CTA of this one has
// called it (or exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ void pf_timeout(uint32_t* status, uint32_t site) {
  if (atomicCAS(&status[0], 0u, (uint32_t)ST_TIMEOUT) == 0u) {
    status[1] = blockIdx.x;
    status[2] = blockIdx.y;
    status[3] = site;
    __threadfence();
  }
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* m, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(m), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* m, int x, int y, int z, int w,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];"
      ::"r"(dst), "l"(m), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes (64 bf16 of k), 8-row swizzle
// atoms 1024 bytes apart.  The k-th 16-element slice starts k * 32 bytes in.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address / 16
  d |= (uint64_t)1 << 16;                              // leading offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;                    // stride offset: next 8-row atom
  d |= (uint64_t)1 << 46;                              // descriptor version
  d |= (uint64_t)2 << 61;                              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = kPfBM x N = BN (a multiple of 16 up to 256).
template <int BN>
__host__ __device__ constexpr uint32_t idesc_bf16() {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kPfBM >> 4) << 24);
}

template <int BN>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc_bf16<BN>()), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 or 64 consecutive TMEM columns of the warp's lane quarter, one
// register each, waited for in the same statement
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// x = p[0] + p[1] + p[2] to 2^-27 relative (the first two: 2^-18): each
// part is the bf16 rounding of what the previous parts left (the remainders
// are exact in fp32)
__device__ __forceinline__ void split_parts(float x, uint16_t (&p)[kPfParts]) {
#pragma unroll
  for (int i = 0; i < kPfParts; ++i) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    p[i] = __bfloat16_as_ushort(h);
    x -= __bfloat162float(h);
  }
}



// Epilogue of 16 consecutive packed rows [n, n + 16) of token t (t < T).
template <int EPI>
__device__ __forceinline__ void gemm_epilogue(const PrefillGemm& g, int t, int n, const uint32_t (&v)[16]) {
  if constexpr (EPI == PE_RESID) {
    float* xr = g.x + (int64_t)t * g.ldx + n;
    if (n + 16 <= g.N) {
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        float4 a = *reinterpret_cast<float4*>(xr + j);
        a.x += __uint_as_float(v[j]);
        a.y += __uint_as_float(v[j + 1]);
        a.z += __uint_as_float(v[j + 2]);
        a.w += __uint_as_float(v[j + 3]);
        *reinterpret_cast<float4*>(xr + j) = a;
      }
    } else {
      for (int j = 0; j < 16 && n + j < g.N; ++j) xr[j] += __uint_as_float(v[j]);
    }
  } else if constexpr (EPI == PE_SWIGLU) {
    // packed rows interleave gate (even) and up (odd) of unit n / 2 + i
    const int j0 = n >> 1;
    uint16_t part[kPfParts][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint16_t p[kPfParts];
      split_parts(silu(__uint_as_float(v[2 * i])) * __uint_as_float(v[2 * i + 1]), p);
#pragma unroll
      for (int k = 0; k < kPfParts; ++k) part[k][i] = p[k];
    }
#pragma unroll
    for (int k = 0; k < kPfParts; ++k) {
      if (k >= g.parts) break;
      uint16_t* d = g.out[k] + (int64_t)t * g.ldo + j0;
      if (n + 16 <= g.N)
        *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(part[k]);
      else
        for (int i = 0; i < 8 && n + 2 * i + 1 < g.N; ++i) d[i] = part[k][i];
    }
  } else {
    // packed QKV rows per KV head grp: G query heads, k, v (hd rows each);
    // in a q or k head, rows 2i, 2i + 1 hold dims i, i + hd/2 (a rotate-half
    // RoPE pair).  A 16-row chunk never straddles a head (hd % 16 == 0).
    const int hd = g.hd, half = hd >> 1, G = g.group, gw = (G + 2) * hd;
    const int grp = n / gw, slot = (n % gw) / hd, within = (n % gw) % hd;
    const int pos = g.s0 + t;
    if (n >= g.N) return;
    if (slot <= G) {
      // dims i0 .. i0 + 7 and half + i0 .. + 7: two 8-wide runs of the row,
      // stored with 16-byte vectors (i0 is a multiple of 8)
      const int i0 = within >> 1;
      const float4* cs = reinterpret_cast<const float4*>(g.rope + (int64_t)pos * half + i0);
      float a[8], b[8];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float4 c = cs[pp];   // (cos, sin) of dims i0 + 2 pp and i0 + 2 pp + 1
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pr = 2 * pp + e;
          const float y0 = __uint_as_float(v[2 * pr]), y1 = __uint_as_float(v[2 * pr + 1]);
          const float cx = e ? c.z : c.x, sy = e ? c.w : c.y;
          a[pr] = y0 * cx - y1 * sy;
          b[pr] = y1 * cx + y0 * sy;
        }
      }
      if (slot < G) {
        float* qrow = g.q + (int64_t)t * g.ldq + (int64_t)(grp * G + slot) * hd;
        float4* qa = reinterpret_cast<float4*>(qrow + i0);
        float4* qb = reinterpret_cast<float4*>(qrow + half + i0);
        qa[0] = make_float4(a[0], a[1], a[2], a[3]);
        qa[1] = make_float4(a[4], a[5], a[6], a[7]);
        qb[0] = make_float4(b[0], b[1], b[2], b[3]);
        qb[1] = make_float4(b[4], b[5], b[6], b[7]);
      } else {
        uint16_t* krow = g.kv + ((((int64_t)g.layer * 2 + 0) * g.n_kv + grp) * g.max_seq + pos) * hd;
        uint16_t ka[8], kb[8];
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          ka[pr] = bf16_bits(a[pr]);
          kb[pr] = bf16_bits(b[pr]);
        }
        *reinterpret_cast<uint4*>(krow + i0) = *reinterpret_cast<const uint4*>(ka);
        *reinterpret_cast<uint4*>(krow + half + i0) = *reinterpret_cast<const uint4*>(kb);
      }
    } else {
      uint16_t* vrow = g.kv + ((((int64_t)g.layer * 2 + 1) * g.n_kv + grp) * g.max_seq + pos) * hd + within;
      uint16_t o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = bf16_bits(__uint_as_float(v[j]));
      *reinterpret_cast<uint4*>(vrow) = *reinterpret_cast<const uint4*>(o);
      *reinterpret_cast<uint4*>(vrow + 8) = *reinterpret_cast<const uint4*>(o + 8);
    }
  }
}

// the activation parts' maps and the weight slice's map of one GEMM
struct GemmMaps {
  CUtensorMap a[kPfParts];
  CUtensorMap w;
};

template <int EPI, int PARTS, int BN>
__global__ void __launch_bounds__(kPfGemmThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ PrefillGemm g) {
  using Shape = GemmShape<PARTS, BN>;
  constexpr int kPfStages = Shape::kStages, kPfEpiCols = Shape::kEpiCols;
  extern __shared__ uint8_t pf_smem_raw[];
  GemmSmem<PARTS, BN>& sm = *reinterpret_cast<GemmSmem<PARTS, BN>*>(
      (reinterpret_cast<uintptr_t>(pf_smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // persistent: CTA c takes tiles c, c + gridDim.x, ... (token tile fastest,
  // so the CTAs working at one time share weight slices through L2); each
  // role keeps its ring stage and accumulator segment counters across tiles,
  // so the next tile's loads and first MMAs overlap this tile's epilogue
  const int mt = (g.T + kPfBM - 1) / kPfBM;
  const int n_tiles = mt * ((g.N + BN - 1) / BN);
  const int nseg = (g.nk + kPfSegKB - 1) / kPfSegKB;
  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.full[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.empty[s])));
    }
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.acc_full[b])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.acc_empty[b])), "r"(kPfEpiWarps));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.failed = 0;
  }
  if (warp == 1) {   // the MMA warp owns the accumulators' TMEM columns
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem)),
                 "r"(kPfTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = sm.tmem;
  pdl_wait();   // the activation parts, the residual rows and the KV cache are the previous kernels'

  if (warp == 0) {
    if (lane == 0) {   // TMA producer
      int it = 0;      // ring stages used so far
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        const int m0 = (tile % mt) * kPfBM, n0 = (tile / mt) * BN;
        for (int kb = 0; kb < g.nk; ++kb, ++it) {
          const int s = it % kPfStages;
          const uint32_t ph = (uint32_t)(it / kPfStages) & 1u;
          if (!bar_wait(smem_addr(&sm.empty[s]), ph ^ 1u, g.timeout_ns)) {
            pf_timeout(g.status, SITE_PF_TMA);
            sm.failed = 1;
            ok = false;
            break;
          }
          const uint32_t fb = smem_addr(&sm.full[s]);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                       "r"(PARTS * kPfATile + Shape::kBTile)
                       : "memory");
          const int k = kb * kPfBK;
#pragma unroll
          for (int part = 0; part < PARTS; ++part) tma_2d(smem_addr(sm.a[s][part]), &maps.a[part], k, m0, fb);
          tma_4d(smem_addr(sm.w[s]), &maps.w, k % g.Kt, 0, k / g.Kt, n0 / g.Rt, fb);
        }
      }
      // copies the MMA warp never waited for (it stopped early) land before
      // the CTA's shared memory goes away
      if (!ok)
        for (int j = max(0, it - kPfStages); j < it; ++j)
          bar_wait(smem_addr(&sm.full[j % kPfStages]), (uint32_t)(j / kPfStages) & 1u, g.timeout_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {   // MMA issuer: the parts of A against the same W slice
      int it = 0, gseg = 0;   // ring stages and accumulator segments used so far
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < g.nk; ++kb, ++it) {
          const int seg = gseg + kb / kPfSegKB, b = seg & 1;
          const uint32_t dt = tmem + (uint32_t)(b * kPfBN);
          const bool first = kb % kPfSegKB == 0;
          if (first) {   // this buffer's previous segment must have been drained
            if (!bar_wait(smem_addr(&sm.acc_empty[b]), ((uint32_t)(seg >> 1) & 1u) ^ 1u, g.timeout_ns)) {
              pf_timeout(g.status, SITE_PF_MMA);
              sm.failed = 1;
              ok = false;
              break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;");
          }
          const int s = it % kPfStages;
          const uint32_t ph = (uint32_t)(it / kPfStages) & 1u;
          if (!bar_wait(smem_addr(&sm.full[s]), ph, g.timeout_ns)) {
            pf_timeout(g.status, SITE_PF_MMA);
            sm.failed = 1;
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint32_t bw = smem_addr(sm.w[s]);
#pragma unroll
          for (int k = 0; k < kPfBK / 16; ++k) {
            const uint64_t bd = kmajor_sw128_desc(bw + k * 32);
#pragma unroll
            for (int part = 0; part < PARTS; ++part)
              umma_bf16<BN>(dt, kmajor_sw128_desc(smem_addr(sm.a[s][part]) + k * 32), bd,
                            (!first || k != 0 || part != 0) ? 1u : 0u);
          }
          umma_commit(smem_addr(&sm.empty[s]));
          // the segment is complete once every MMA issued into it has finished
          if (kb % kPfSegKB == kPfSegKB - 1 || kb == g.nk - 1) umma_commit(smem_addr(&sm.acc_full[b]));
        }
        gseg += nseg;
      }
    }
  } else {
    const int quarter = warp & 3;   // TMEM lanes this warp may read: 32 * quarter ..
    const int col0 = ((warp - 2) >> 2) * kPfEpiCols;   // this warp's accumulator columns
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0;
    int gseg = 0;   // accumulator segments drained so far
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
      const int m0 = (tile % mt) * kPfBM, n0 = (tile / mt) * BN;
      const int t = m0 + quarter * 32 + lane;
      float acc[kPfEpiCols];
#pragma unroll
      for (int i = 0; i < kPfEpiCols; ++i) acc[i] = 0.f;
      for (int sg = 0; sg < nseg; ++sg, ++gseg) {
        const int b = gseg & 1;
        ok = __all_sync(0xFFFFFFFFu,
                        bar_wait(smem_addr(&sm.acc_full[b]), (uint32_t)(gseg >> 1) & 1u, g.timeout_ns));
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
#pragma unroll
        for (int c = 0; c < kPfEpiCols; c += 16) {
          uint32_t v[16];
          tmem_ld16(lane_base + (uint32_t)(b * kPfBN + c), v);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[c + j] += __uint_as_float(v[j]);
        }
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm.acc_empty[b])) : "memory");
      }
      if (!ok) {
        if (lane == 0) pf_timeout(g.status, SITE_PF_EPI);
      } else if (!sm.failed && t < g.T) {
#pragma unroll
        for (int c = 0; c < kPfEpiCols; c += 16) {
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(acc[c + j]);
          if (n0 + col0 + c < g.N) gemm_epilogue<EPI>(g, t, n0 + col0 + c, v);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPfTmemCols));
  }
}

// ------------------------------------------------------------ elementwise

__global__ void prefill_embed_kernel(const int32_t* tokens, int T, const uint16_t* embed, int hidden, float* x) {
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= T) return;
  pdl_wait();
  const uint16_t* e = embed + (int64_t)tokens[t] * hidden;
  float* xr = x + (int64_t)t * hidden;
  for (int k = threadIdx.x; k < hidden; k += blockDim.x) xr[k] = __uint_as_float((uint32_t)e[k] << 16);
}

// one CTA (256 threads) per token row
struct Parts {
  uint16_t* p[kPfParts];
};

// float4 groups of a row each thread holds in registers (hidden <= 4 *
// kNormVec * 1024)
constexpr int kNormVec = 8;

// One CTA per token row: the row is loaded once into registers (all loads
// in flight together), reduced, scaled by the norm weight and stored as
// bf16 parts, four elements (8 bytes per part) at a time.
__global__ void __launch_bounds__(1024) prefill_norm_kernel(const float* x, int T, int hidden, const uint16_t* w,
                                                            float eps, const Parts out, int parts) {
  __shared__ float part[32];
  pdl_launch_dependents();
  const int t = blockIdx.x;
  if (t >= T) return;
  pdl_wait();
  const int n4 = hidden >> 2, tid = threadIdx.x, nt = blockDim.x;
  const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)t * hidden);
  float4 v[kNormVec];
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int k4 = tid + i * nt;
    v[i] = k4 < n4 ? xr[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i)
    ss += fmaf(v[i].x, v[i].x, v[i].y * v[i].y) + fmaf(v[i].z, v[i].z, v[i].w * v[i].w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((tid & 31) == 0) part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (nt >> 5); ++i) tot += part[i];
  const float r = rsqrtf(tot / (float)hidden + eps);
  const uint2* w4 = reinterpret_cast<const uint2*>(w);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int k4 = tid + i * nt;
    if (k4 >= n4) break;
    const uint2 wb = w4[k4];
    const float y[4] = {v[i].x * r * __uint_as_float(wb.x << 16), v[i].y * r * __uint_as_float(wb.x & 0xFFFF0000u),
                        v[i].z * r * __uint_as_float(wb.y << 16), v[i].w * r * __uint_as_float(wb.y & 0xFFFF0000u)};
    uint16_t pp[4][kPfParts];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_parts(y[e], pp[e]);
#pragma unroll
    for (int j = 0; j < kPfParts; ++j)
      if (j < parts)
        *reinterpret_cast<uint2*>(out.p[j] + (int64_t)t * hidden + 4 * k4) =
            make_uint2((uint32_t)pp[0][j] | ((uint32_t)pp[1][j] << 16), (uint32_t)pp[2][j] | ((uint32_t)pp[3][j] << 16));
  }
}

// -------------------------------------------------------------- attention


__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// 16-token groups per attention CTA: up to eight warps (G of them per group)
__host__ __device__ constexpr int attn_groups(int group) {
  return group >= 8 ? 1 : group >= 4 ? 2 : 4;
}

template <int HD>
struct AttnShape {
  static constexpr int RP = HD + 8;   // bf16 row pitch: rows 16 bytes apart in the banks
  static constexpr int KV_ELEMS = 2 * kPfKB * RP;   // one K or V buffer pair (double buffered)
  static int bytes(int group) { return (2 * KV_ELEMS + group * attn_groups(group) * 2 * kPfQT * RP) * 2; }
};

// Shared memory (bf16 elements): K [2][64][RP], V [2][64][RP], then per
// warp (query head x token group) q hi [16][RP] and q lo [16][RP].
template <int HD>
__global__ void __launch_bounds__(256, 2) prefill_attn_kernel(const PrefillAttn a) {
  using S = AttnShape<HD>;
  constexpr int RP = S::RP, KS = HD / 16, DN = HD / 8, NT = kPfKB / 8;
  extern __shared__ __align__(16) uint16_t at_smem[];
  uint16_t* ks = at_smem;
  uint16_t* vs = at_smem + S::KV_ELEMS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  pdl_launch_dependents();
  pdl_wait();   // q and the K,V rows of this chunk come from the QKV GEMM
  const int gq = lane >> 2, tq = lane & 3;
  // CTA i: KV head i mod n_kv, token block nb - 1 - i / n_kv.  The causal
  // work of a token block grows with its position, so the CTAs launch
  // longest first and the short ones fill the SMs at the end.
  const int nb = (int)gridDim.x / a.n_kv;
  const int g = (int)blockIdx.x % a.n_kv, G = a.group;
  const int cta_tokens = kPfQT * attn_groups(G);
  const int tb0 = (nb - 1 - (int)blockIdx.x / a.n_kv) * cta_tokens;   // the CTA's first token
  const int tb = tb0 + (warp / G) * kPfQT;           // this warp's first token
  const int head = g * G + warp % G;
  uint16_t* qh = at_smem + 2 * S::KV_ELEMS + warp * 2 * kPfQT * RP;
  uint16_t* ql = qh + kPfQT * RP;

  // this block's queries, pre-scaled into log2 units, as bf16 hi + lo
  const float qscale = 1.4426950408889634f * rsqrtf((float)HD);
  for (int i = lane; i < kPfQT * HD / 4; i += 32) {
    const int r = i / (HD / 4), d = (i % (HD / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tb + r < a.T) x = *reinterpret_cast<const float4*>(a.q + (int64_t)(tb + r) * a.ldq + (int64_t)head * HD + d);
    uint32_t h0, l0, h1, l1;
    split_bf16x2(x.x * qscale, x.y * qscale, h0, l0);
    split_bf16x2(x.z * qscale, x.w * qscale, h1, l1);
    *reinterpret_cast<uint2*>(qh + r * RP + d) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(ql + r * RP + d) = make_uint2(l0, l1);
  }

  // positions [0, kv_end) are needed by the CTA's last valid token
  const int t_last = min(a.T, tb0 + cta_tokens) - 1;
  const int kv_end = a.s0 + t_last + 1;
  const int nblk = (kv_end + kPfKB - 1) / kPfKB;
  const uint16_t* kbase = a.kv + (((int64_t)a.layer * 2 + 0) * a.n_kv + g) * a.max_seq * HD;
  const uint16_t* vbase = a.kv + (((int64_t)a.layer * 2 + 1) * a.n_kv + g) * a.max_seq * HD;
  auto load_block = [&](int blk, int buf) {
    constexpr int CH = HD / 8;   // 16-byte chunks per row
    for (int i = tid; i < 2 * kPfKB * CH; i += nthr) {
      const int which = i / (kPfKB * CH), r = (i / CH) % kPfKB, c = i % CH;
      const int p = blk * kPfKB + r;
      uint16_t* dst = (which ? vs : ks) + buf * kPfKB * RP + r * RP + c * 8;
      if (p < kv_end)
        cp_async16(smem_addr(dst), (which ? vbase : kbase) + (int64_t)p * HD + c * 8);
      else   // past the filled cache: zeros (masked scores must meet finite values)
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float o[DN][4];
#pragma unroll
  for (int i = 0; i < DN; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int lim0 = a.s0 + tb + gq, lim1 = lim0 + 8;   // last visible position of rows gq, gq + 8

  load_block(0, 0);
  for (int blk = 0; blk < nblk; ++blk) {
    const int buf = blk & 1;
    if (blk + 1 < nblk) {
      load_block(blk + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const uint32_t kb_s = smem_addr(ks + buf * kPfKB * RP), vb_s = smem_addr(vs + buf * kPfKB * RP);

    // S = Q K^T: 16 tokens x kPfKB positions, NT tiles of 8 positions; per
    // k step the hi parts of q go into every tile before the lo parts, so
    // that no mma waits on the one just issued
    float s[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      uint32_t qa_h[4], qa_l[4];
      const uint32_t qoff = (uint32_t)(((lane & 15) * RP + k * 16 + (lane >> 4) * 8) * 2);
      ldsm_x4(smem_addr(qh) + qoff, qa_h);
      ldsm_x4(smem_addr(ql) + qoff, qa_l);
      uint32_t kf[NT / 2][4];
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int mi = lane >> 3;
        const int key = (2 * np + (mi >> 1)) * 8 + (lane & 7);
        ldsm_x4(kb_s + (uint32_t)((key * RP + k * 16 + (mi & 1) * 8) * 2), kf[np]);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        mma_bf16_16816(s[2 * np], qa_h, kf[np][0], kf[np][1]);
        mma_bf16_16816(s[2 * np + 1], qa_h, kf[np][2], kf[np][3]);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        mma_bf16_16816(s[2 * np], qa_l, kf[np][0], kf[np][1]);
        mma_bf16_16816(s[2 * np + 1], qa_l, kf[np][2], kf[np][3]);
      }
    }
    // causal mask, online softmax (rows gq and gq + 8 of the warp's tile)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int p = blk * kPfKB + nt * 8 + 2 * tq + e;
        if (p > lim0) s[nt][e] = -INFINITY;
        if (p > lim1) s[nt][2 + e] = -INFINITY;
        mx[0] = fmaxf(mx[0], s[nt][e]);
        mx[1] = fmaxf(mx[1], s[nt][2 + e]);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 2));
      const float mn = fmaxf(mrow[r], mx[r]);
      mu[r] = mn == -INFINITY ? 0.f : mn;
      alpha[r] = exp2f(mrow[r] - mu[r]);
      mrow[r] = mn;
      lrow[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[nt][e] = exp2f(s[nt][e] - mu[e >> 1]);
        lrow[e >> 1] += s[nt][e];
      }
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      o[dn][0] *= alpha[0];
      o[dn][1] *= alpha[0];
      o[dn][2] *= alpha[1];
      o[dn][3] *= alpha[1];
    }
    // O += P V: kPfKB / 16 k-steps of 16 positions, P as bf16 hi + lo A
    // fragments
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      uint32_t pa_h[4], pa_l[4];
      split_bf16x2(s[2 * kk][0], s[2 * kk][1], pa_h[0], pa_l[0]);
      split_bf16x2(s[2 * kk][2], s[2 * kk][3], pa_h[1], pa_l[1]);
      split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], pa_h[2], pa_l[2]);
      split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], pa_h[3], pa_l[3]);
#pragma unroll
      for (int dp = 0; dp < DN / 2; ++dp) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
        uint32_t vf[4];
        ldsm_x4_trans(vb_s + (uint32_t)((key * RP + (2 * dp + (mi >> 1)) * 8) * 2), vf);
        mma_bf16_16816(o[2 * dp], pa_h, vf[0], vf[1]);
        mma_bf16_16816(o[2 * dp + 1], pa_h, vf[2], vf[3]);
        mma_bf16_16816(o[2 * dp], pa_l, vf[0], vf[1]);
        mma_bf16_16816(o[2 * dp + 1], pa_l, vf[2], vf[3]);
      }
    }
    __syncthreads();   // the buffer is reloaded two blocks on
  }
  // normalise and store rows gq, gq + 8 of the tile
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xFFFFFFFFu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xFFFFFFFFu, lrow[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = tb + gq + 8 * r;
    if (t >= a.T) continue;
    const float inv = 1.0f / lrow[r];
    const int64_t row = (int64_t)t * a.ldo + (int64_t)head * HD;
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) {
      uint16_t p0[kPfParts], p1[kPfParts];
      split_parts(o[dn][2 * r] * inv, p0);
      split_parts(o[dn][2 * r + 1] * inv, p1);
      const int d = dn * 8 + 2 * tq;
#pragma unroll
      for (int i = 0; i < kPfParts; ++i)
        if (i < a.parts) *reinterpret_cast<uint32_t*>(a.o[i] + row + d) = (uint32_t)p0[i] | ((uint32_t)p1[i] << 16);
    }
  }
}


// ------------------------------------------------ attention on tcgen05
//
// One CTA: kTcRows query rows (TPC = 128 / G tokens x the G query heads
// of KV head g, head-major: row = h * TPC + t) against the cache's keys
// [0, kv_end) in blocks of kTcKeys.  Per block:
//   S  = Q K^T           tcgen05.mma M 128, N 64: q as bf16 hi + lo (two
//                        MMAs per 16-dim step) into one of two TMEM buffers
//   softmax              eight math warps, a row's 64 scores split over two
//                        warps (tcgen05.ld of 32 columns each); running max
//                        and sum in registers, block maxima exchanged through
//                        shared memory; P as bf16 hi + lo into shared memory
//   O += P V             tcgen05.mma M 128, N head_dim, K 16 keys (P hi and
//                        lo), V read in place from its TMA layout as an
//                        MN-major operand; the block's product lands in one
//                        of two TMEM buffers and is added into fp32
//                        registers (O scaled by the max correction), as the
//                        GEMM promotes its segments, one block late: the
//                        math warps compute block i's softmax while the
//                        tensor cores run block i - 1's P.V
// Warp 0 streams K blocks (each stage freed once its S is computed) and V
// blocks (freed after P.V) with TMA, warp 1 issues the S MMAs and warp 10
// the P.V MMAs, warps 2..9 compute.  Every wait is bounded.
constexpr int kTcKStages = 2;
constexpr int kTcVStages = 2;
constexpr uint32_t kTcTmemCols = 512;   // S buffers [0, 128), P.V buffers [128, 384)
constexpr int kTcMathWarps = 8;
// warps: 0 TMA, 1 S issue, 2..9 math, 10 P.V issue
constexpr int kTcThreads = 96 + 32 * kTcMathWarps;
constexpr int kTcPvWarp = 2 + kTcMathWarps;

template <int HD>
struct __align__(1024) TcAttnSmem {
  static constexpr int A = HD / 64;                 // 128-byte atoms along the head dim
  uint8_t q[2][A][kTcRows * 128];                   // q hi / lo: [part][atom][row][128 B], swizzled
  uint8_t k[kTcKStages][A][kTcKeys * 128];          // K block: [atom][key][128 B] (TMA, swizzled)
  uint8_t v[kTcVStages][A][kTcKeys * 128];          // V block, the same layout
  uint8_t p[2][2][kTcRows * 128];                   // P [block parity][hi / lo]: [row][64 keys], swizzled
  float mx[2][2][kTcRows];                          // block maxima [block parity][row half][row]
  float ls[2][kTcRows];                             // row sums [row half][row]
  uint64_t k_full[kTcKStages], k_empty[kTcKStages], v_full[kTcVStages], v_empty[kTcVStages];
  uint64_t q_full, s_full[2], s_free[2], p_full[2], pv_full[2], x_bar[2], l_bar;
  uint32_t tmem;
};

struct TcAttnArgs {
  CUtensorMap kv;   // KV cache rows, boxes of 64 dims x kTcKeys rows
  PrefillAttn a;
};

// MN-major operand with 128-byte swizzle: rows of 128 bytes (64 elements
// along M / N) for consecutive k, 8-row groups 1024 bytes apart, the next
// 64 elements along M / N lbo bytes on.
__device__ __forceinline__ uint64_t mnmajor_sw128_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// 2^x by the SFU's approximate exp2 (ex2.approx), subnormal results
// flushed to zero: softmax weights that small do not count
__device__ __forceinline__ float exp2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// a non-blocking test of an mbarrier phase (acquire on success)
__device__ __forceinline__ bool mbar_test32(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_attn_tc_kernel(const __grid_constant__ TcAttnArgs args) {
  using Sm = TcAttnSmem<HD>;
  constexpr int A = Sm::A, DH = HD / 2;   // atoms; head dims per math warp (row half)
  constexpr uint32_t kColPV = 128;        // TMEM columns: S buffers at 0 and 64, P.V buffers at 128 and 256
  constexpr uint32_t kIdS = idesc_bf16<kTcKeys>();
  constexpr uint32_t kIdPV = idesc_bf16<HD>() | (1u << 16);   // B (V) MN-major
  const PrefillAttn& a = args.a;
  extern __shared__ uint8_t tc_smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group, TPC = kTcRows / G;
  const int nb = (a.T + TPC - 1) / TPC;
  const int g = (int)blockIdx.x % a.n_kv;
  const int tb0 = (nb - 1 - (int)blockIdx.x / a.n_kv) * TPC;   // longest first
  const int kv_end = a.s0 + min(a.T, tb0 + TPC);               // keys [0, kv_end) are needed
  const int nblk = (kv_end + kTcKeys - 1) / kTcKeys;
  const int limit = a.s0 + a.T;                                 // keys [0, limit) are written
  // first key of block i's window: the block itself, or for a block that
  // would run past the written keys, the last kTcKeys written keys (the
  // keys it repeats are masked)
  auto win = [&](int i) { return min(i * kTcKeys, limit - kTcKeys); };
  const int row_k = ((a.layer * 2 + 0) * a.n_kv + g) * a.max_seq;
  const int row_v = ((a.layer * 2 + 1) * a.n_kv + g) * a.max_seq;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int st = 0; st < kTcKStages; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.k_full[st])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.k_empty[st])));
    }
    for (int st = 0; st < kTcVStages; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.v_full[st])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.v_empty[st])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.q_full)), "r"(kTcMathWarps));
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.s_full[b])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.x_bar[b])), "r"(kTcMathWarps));
    }
    for (int b = 0; b < 2; ++b) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.s_free[b])), "r"(kTcMathWarps));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.p_full[b])), "r"(kTcMathWarps));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.pv_full[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.pv_full[1])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&sm.l_bar)), "r"(kTcMathWarps));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sm.tmem)),
                 "r"(kTcTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = sm.tmem;
  pdl_wait();   // q and this chunk's K,V come from the QKV GEMM

  if (warp == 0) {
    if (lane == 0) {   // TMA producer: K blocks run ahead of V blocks, each in its own ring
      int kc = 0, vc = 0;   // next block to load, per ring
      uint64_t t0 = global_timer();
      bool ok = true;
      while (kc < nblk || vc < nblk) {
        bool moved = false;
        if (kc < nblk &&
            mbar_test32(smem_addr(&sm.k_empty[kc % kTcKStages]), ((uint32_t)(kc / kTcKStages) & 1u) ^ 1u)) {
          const uint32_t fb = smem_addr(&sm.k_full[kc % kTcKStages]);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(A * kTcKeys * 128)
                       : "memory");
#pragma unroll
          for (int at = 0; at < A; ++at)
            tma_2d(smem_addr(sm.k[kc % kTcKStages][at]), &args.kv, 64 * at, row_k + win(kc), fb);
          ++kc;
          moved = true;
        }
        if (vc < kc &&
            mbar_test32(smem_addr(&sm.v_empty[vc % kTcVStages]), ((uint32_t)(vc / kTcVStages) & 1u) ^ 1u)) {
          const uint32_t fb = smem_addr(&sm.v_full[vc % kTcVStages]);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(A * kTcKeys * 128)
                       : "memory");
#pragma unroll
          for (int at = 0; at < A; ++at)
            tma_2d(smem_addr(sm.v[vc % kTcVStages][at]), &args.kv, 64 * at, row_v + win(vc), fb);
          ++vc;
          moved = true;
        }
        if (moved) {
          t0 = global_timer();
        } else if (global_timer() - t0 > a.timeout_ns) {
          pf_timeout(a.status, SITE_PF_TMA);
          ok = false;
          break;
        } else {
          __nanosleep(128);   // leave the issue slots to the math warps
        }
      }
      // copies the consumers never waited for (they stopped early) land
      // before the CTA's shared memory goes away
      if (!ok) {
        for (int blk = max(0, kc - kTcKStages); blk < kc; ++blk)
          bar_wait(smem_addr(&sm.k_full[blk % kTcKStages]), (uint32_t)(blk / kTcKStages) & 1u, a.timeout_ns);
        for (int blk = max(0, vc - kTcVStages); blk < vc; ++blk)
          bar_wait(smem_addr(&sm.v_full[blk % kTcVStages]), (uint32_t)(blk / kTcVStages) & 1u, a.timeout_ns);
      }
    }
  } else if (warp == 1 || warp == kTcPvWarp) {
    // MMA issue, split over two threads (issuing one of these small MMAs
    // takes about as long as running it): warp 1 issues S = Q K^T, warp 10
    // P.V.  Operand descriptors are computed once; a 16-element k step is
    // 32 bytes further in the 128-byte rows, +2 in the descriptor's address
    // field (which no step carries out of).
    constexpr uint64_t kAtomQ = (kTcRows * 128) >> 4, kAtomK = (kTcKeys * 128) >> 4;   // atom strides
    constexpr uint64_t kStageK = (uint64_t)(A * kTcKeys * 128) >> 4, kPart = (kTcRows * 128) >> 4;
    if (lane == 0 && warp == 1) {
      bool ok = bar_wait(smem_addr(&sm.q_full), 0u, a.timeout_ns);
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint64_t dq0 = kmajor_sw128_desc(smem_addr(sm.q[0][0])), dq1 = kmajor_sw128_desc(smem_addr(sm.q[1][0]));
      const uint64_t dk0 = kmajor_sw128_desc(smem_addr(sm.k[0][0]));
      for (int blk = 0; ok && blk < nblk; ++blk) {
        // the S buffer this block reuses was read by the math warps
        if (blk >= 2 && !(ok = bar_wait(smem_addr(&sm.s_free[blk & 1]), (uint32_t)((blk - 2) >> 1) & 1u, a.timeout_ns)))
          break;
        const int st = blk % kTcKStages;
        if (!(ok = bar_wait(smem_addr(&sm.k_full[st]), (uint32_t)(blk / kTcKStages) & 1u, a.timeout_ns))) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t d = tmem + (uint32_t)((blk & 1) * kTcKeys);
        const uint64_t dk = dk0 + (uint64_t)st * kStageK;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint64_t step = (uint64_t)((ks & 3) * 2);
          const uint64_t bd = dk + (uint64_t)(ks >> 2) * kAtomK + step;
          umma_f16(d, dq0 + (uint64_t)(ks >> 2) * kAtomQ + step, bd, kIdS, ks != 0 ? 1u : 0u);
          umma_f16(d, dq1 + (uint64_t)(ks >> 2) * kAtomQ + step, bd, kIdS, 1u);
        }
        umma_commit(smem_addr(&sm.s_full[blk & 1]));
        umma_commit(smem_addr(&sm.k_empty[st]));
      }
      if (!ok) pf_timeout(a.status, SITE_PF_MMA);
    } else if (lane == 0) {
      bool ok = true;
      const uint64_t dp0 = kmajor_sw128_desc(smem_addr(sm.p[0][0]));
      const uint64_t dv0 = mnmajor_sw128_desc(smem_addr(sm.v[0][0]), (uint32_t)(kTcKeys * 128));
      for (int blk = 0; ok && blk < nblk; ++blk) {
        // P of this block written (and block blk - 2's P.V drained from the
        // TMEM buffer and P buffer this block reuses)
        if (!(ok = bar_wait(smem_addr(&sm.p_full[blk & 1]), (uint32_t)(blk >> 1) & 1u, a.timeout_ns))) break;
        const int st = blk % kTcVStages;
        if (!(ok = bar_wait(smem_addr(&sm.v_full[st]), (uint32_t)(blk / kTcVStages) & 1u, a.timeout_ns))) break;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const uint32_t dpv = tmem + kColPV + (uint32_t)((blk & 1) * 128);
        const uint64_t dv = dv0 + (uint64_t)st * kStageK;
        const uint64_t dp = dp0 + (uint64_t)(blk & 1) * 2 * kPart;
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk) {
          const uint64_t bd = dv + (uint64_t)(kk * 16 * 128 / 16);   // 16 keys = 16 rows of 128 bytes
          umma_f16(dpv, dp + (uint64_t)(kk * 2), bd, kIdPV, kk != 0 ? 1u : 0u);
          umma_f16(dpv, dp + kPart + (uint64_t)(kk * 2), bd, kIdPV, 1u);
        }
        umma_commit(smem_addr(&sm.v_empty[st]));
        umma_commit(smem_addr(&sm.pv_full[blk & 1]));
      }
      if (!ok) pf_timeout(a.status, SITE_PF_MMA);
    }
  } else {
    // math warps: row r = TMEM lane, columns / dims of half hf
    const int quarter = warp & 3, hf = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int h_local = r / TPC, t = tb0 + r % TPC;
    const bool row_ok = t < a.T;
    const int pos = a.s0 + t;
    const int head = g * G + h_local;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    // q row, this half's dims, pre-scaled into log2 units, as bf16 hi + lo
    const float qscale = 1.4426950408889634f * rsqrtf((float)HD);
#pragma unroll
    for (int c = 0; c < DH / 8; ++c) {
      const int d0 = hf * DH + c * 8;
      float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
      if (row_ok) {
        const float4* src = reinterpret_cast<const float4*>(a.q + (int64_t)t * a.ldq + (int64_t)head * HD + d0);
        x0 = src[0];
        x1 = src[1];
      }
      uint32_t hi[4], lo[4];
      split_bf16x2(x0.x * qscale, x0.y * qscale, hi[0], lo[0]);
      split_bf16x2(x0.z * qscale, x0.w * qscale, hi[1], lo[1]);
      split_bf16x2(x1.x * qscale, x1.y * qscale, hi[2], lo[2]);
      split_bf16x2(x1.z * qscale, x1.w * qscale, hi[3], lo[3]);
      const int cc = (d0 & 63) >> 3;
      const uint32_t off = (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
      *reinterpret_cast<uint4*>(sm.q[0][d0 >> 6] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sm.q[1][d0 >> 6] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive_cta(smem_addr(&sm.q_full));

    float o[DH];
#pragma unroll
    for (int i = 0; i < DH; ++i) o[i] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, alpha_prev = 0.f;
    // o = o * alpha + the P.V of block i (waits for it)
    auto accumulate = [&](int i, float alpha) -> bool {
      if (!__all_sync(0xFFFFFFFFu, bar_wait(smem_addr(&sm.pv_full[i & 1]), (uint32_t)(i >> 1) & 1u, a.timeout_ns)))
        return false;
      asm volatile("tcgen05.fence::after_thread_sync;");
      uint32_t v[DH];
      if constexpr (DH == 64)
        tmem_ld_x64(lane_base + kColPV + (uint32_t)((i & 1) * 128 + hf * DH), v);
      else
        tmem_ld_x32(lane_base + kColPV + (uint32_t)((i & 1) * 128 + hf * DH), v);
#pragma unroll
      for (int j = 0; j < DH; ++j) o[j] = fmaf(o[j], alpha, __uint_as_float(v[j]));
      asm volatile("tcgen05.fence::before_thread_sync;");
      return true;
    };
    bool ok = true;
    for (int blk = 0; blk < nblk; ++blk) {
      const int b = blk & 1;
      ok = __all_sync(0xFFFFFFFFu, bar_wait(smem_addr(&sm.s_full[b]), (uint32_t)(blk >> 1) & 1u, a.timeout_ns));
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      uint32_t sv[32];
      tmem_ld_x32(lane_base + (uint32_t)(b * kTcKeys + hf * 32), sv);
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.s_free[b]));   // S may be overwritten two blocks on
      // keys of the window; valid: not taken by an earlier block, causal.
      // A block whose keys are all valid for every row of the CTA (all but
      // the last one or two) needs no mask.
      const int w0 = win(blk), k0 = w0 + hf * 32, k_lo = blk * kTcKeys;
      float sc[32];
      float mh = -INFINITY;
      if (w0 == k_lo && k_lo + kTcKeys - 1 <= a.s0 + tb0) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sc[c] = __uint_as_float(sv[c]);
          mh = fmaxf(mh, sc[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int key = k0 + c;
          sc[c] = (row_ok && key >= k_lo && key <= pos) ? __uint_as_float(sv[c]) : -INFINITY;
          mh = fmaxf(mh, sc[c]);
        }
      }
      sm.mx[b][hf][r] = mh;
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.x_bar[b]));
      ok = __all_sync(0xFFFFFFFFu, bar_wait(smem_addr(&sm.x_bar[b]), (uint32_t)(blk >> 1) & 1u, a.timeout_ns));
      if (!ok) break;
      const float m_new = fmaxf(m_run, fmaxf(sm.mx[b][0][r], sm.mx[b][1][r]));
      const float mu = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2_sfu(m_run - mu);   // 0 while nothing was seen
      m_run = m_new;
      float lsum = 0.f;
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = exp2_sfu(sc[2 * i] - mu), p1 = exp2_sfu(sc[2 * i + 1] - mu);
        lsum += p0 + p1;
        split_bf16x2(p0, p1, ph[i], pl[i]);
      }
      l_run = fmaf(l_run, alpha, lsum);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int cc = 4 * hf + j;
        const uint32_t off = (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
        *reinterpret_cast<uint4*>(sm.p[b][0] + off) = make_uint4(ph[4 * j], ph[4 * j + 1], ph[4 * j + 2], ph[4 * j + 3]);
        *reinterpret_cast<uint4*>(sm.p[b][1] + off) = make_uint4(pl[4 * j], pl[4 * j + 1], pl[4 * j + 2], pl[4 * j + 3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.p_full[b]));
      // the previous block's P.V ran on the tensor cores meanwhile
      if (blk > 0 && !(ok = accumulate(blk - 1, alpha_prev))) break;
      alpha_prev = alpha;
    }
    if (ok) ok = accumulate(nblk - 1, alpha_prev);
    if (ok) {
      sm.ls[hf][r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(smem_addr(&sm.l_bar));
      ok = __all_sync(0xFFFFFFFFu, bar_wait(smem_addr(&sm.l_bar), 0u, a.timeout_ns));
    }
    if (!ok) {
      if (lane == 0) pf_timeout(a.status, SITE_PF_EPI);
    } else if (row_ok) {
      const float inv = 1.0f / (sm.ls[0][r] + sm.ls[1][r]);
      const int64_t base = (int64_t)t * a.ldo + (int64_t)head * HD + hf * DH;
#pragma unroll
      for (int c = 0; c < DH; c += 8) {
        uint16_t pp[8][kPfParts];
#pragma unroll
        for (int j = 0; j < 8; ++j) split_parts(o[c + j] * inv, pp[j]);
#pragma unroll
        for (int i = 0; i < kPfParts; ++i) {
          if (i >= a.parts) break;
          *reinterpret_cast<uint4*>(a.o[i] + base + c) =
              make_uint4((uint32_t)pp[0][i] | ((uint32_t)pp[1][i] << 16), (uint32_t)pp[2][i] | ((uint32_t)pp[3][i] << 16),
                         (uint32_t)pp[4][i] | ((uint32_t)pp[5][i] << 16), (uint32_t)pp[6][i] | ((uint32_t)pp[7][i] << 16));
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols));
  }
}

}  // namespace

// Launch with programmatic stream serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int prefill_gemm_smem_bytes(int parts, int bn) {
  const int b = bn == kPfBNNarrow ? (parts == 2 ? (int)sizeof(GemmSmem<2, kPfBNNarrow>)
                                                : (int)sizeof(GemmSmem<3, kPfBNNarrow>))
                                  : (parts == 2 ? (int)sizeof(GemmSmem<2, kPfBN>) : (int)sizeof(GemmSmem<3, kPfBN>));
  return b + 1024;
}

int prefill_gemm_bn(int n_rows, int T, int sms) {
  if (sms <= 0 || T <= 0 || n_rows <= 0) return kPfBN;
  const int64_t mt = (T + kPfBM - 1) / kPfBM;
  auto cost = [&](int bn) {
    const int64_t tiles = mt * ((n_rows + bn - 1) / bn);
    return (tiles + sms - 1) / sms * bn;
  };
  return cost(kPfBNNarrow) < cost(kPfBN) ? kPfBNNarrow : kPfBN;
}

int prefill_attn_smem_bytes(int head_dim, int group) {
  return head_dim == 64 ? AttnShape<64>::bytes(group) : AttnShape<128>::bytes(group);
}

cudaError_t launch_prefill_embed(const int32_t* tokens, int T, const uint16_t* embed, int hidden, float* x,
                                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  return launch_pdl(prefill_embed_kernel, dim3(T), dim3(256), 0, s, tokens, T, embed, hidden, x);
}

cudaError_t launch_prefill_norm(const float* x, int T, int hidden, const uint16_t* w, float eps,
                                uint16_t* const* out, int parts, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  Parts p;
  for (int i = 0; i < kPfParts; ++i) p.p[i] = out[i];
  // threads: enough for kNormVec float4 each, whole warps, at least 128
  const int n4 = hidden / 4;
  int threads = ((n4 + kNormVec - 1) / kNormVec + 31) / 32 * 32;
  threads = std::max(threads, 128);
  if (hidden % 4 || threads > 1024) return cudaErrorInvalidValue;
  return launch_pdl(prefill_norm_kernel, dim3(T), dim3(threads), 0, s, x, T, hidden, w, eps, p, parts);
}

template <int EPI, int PARTS, int BN>
cudaError_t launch_gemm_instance(const GemmMaps& maps, const PrefillGemm& g, cudaStream_t s) {
  const int smem = prefill_gemm_smem_bytes(PARTS, BN);
  cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<EPI, PARTS, BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = ((g.T + kPfBM - 1) / kPfBM) * ((g.N + BN - 1) / BN);
  const dim3 grid((unsigned)std::max(1, std::min(tiles, g.ctas)));
  return launch_pdl(prefill_gemm_kernel<EPI, PARTS, BN>, grid, dim3(kPfGemmThreads), smem, s, maps, g);
}

template <int PARTS, int BN>
cudaError_t launch_gemm_epi(int epi, const GemmMaps& maps, const PrefillGemm& g, cudaStream_t s) {
  if (epi == PE_QKV) return launch_gemm_instance<PE_QKV, PARTS, BN>(maps, g, s);
  if (epi == PE_RESID) return launch_gemm_instance<PE_RESID, PARTS, BN>(maps, g, s);
  return launch_gemm_instance<PE_SWIGLU, PARTS, BN>(maps, g, s);
}

cudaError_t launch_prefill_gemm(int epi, const CUtensorMap* a, const CUtensorMap* w, int bn, const PrefillGemm& g,
                                cudaStream_t s) {
  if (g.T <= 0) return cudaSuccess;
  if (g.parts != 2 && g.parts != 3) return cudaErrorInvalidValue;
  if (bn != kPfBN && bn != kPfBNNarrow) return cudaErrorInvalidValue;
  GemmMaps maps;
  for (int i = 0; i < kPfParts; ++i) maps.a[i] = a[i];
  maps.w = *w;
  if (g.parts == 2)
    return bn == kPfBN ? launch_gemm_epi<2, kPfBN>(epi, maps, g, s) : launch_gemm_epi<2, kPfBNNarrow>(epi, maps, g, s);
  return bn == kPfBN ? launch_gemm_epi<3, kPfBN>(epi, maps, g, s) : launch_gemm_epi<3, kPfBNNarrow>(epi, maps, g, s);
}

bool prefill_attn_uses_tc(int head_dim, int group, int s0, int T) {
  return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= kTcRows && kTcRows % group == 0 &&
         s0 + T >= kTcKeys;
}

template <int HD>
cudaError_t launch_attn_tc(const PrefillAttn& a, const CUtensorMap* kv_map, cudaStream_t s) {
  const int smem = (int)sizeof(TcAttnSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  TcAttnArgs args;
  args.kv = *kv_map;
  args.a = a;
  const int tpc = kTcRows / a.group;
  const dim3 grid((unsigned)(((a.T + tpc - 1) / tpc) * a.n_kv));
  return launch_pdl(prefill_attn_tc_kernel<HD>, grid, dim3(kTcThreads), (size_t)smem, s, args);
}

cudaError_t launch_prefill_attn(const PrefillAttn& a, const CUtensorMap* kv_map, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (kv_map && prefill_attn_uses_tc(a.hd, a.group, a.s0, a.T))
    return a.hd == 64 ? launch_attn_tc<64>(a, kv_map, s) : launch_attn_tc<128>(a, kv_map, s);
  const int smem = prefill_attn_smem_bytes(a.hd, a.group);
  const int groups = attn_groups(a.group), cta_tokens = kPfQT * groups;
  const dim3 grid((unsigned)(((a.T + cta_tokens - 1) / cta_tokens) * a.n_kv));
  const int threads = 32 * a.group * groups;
  const void* fn = a.hd == 64 ? (const void*)prefill_attn_kernel<64> : (const void*)prefill_attn_kernel<128>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (a.hd == 64) return launch_pdl(prefill_attn_kernel<64>, grid, dim3(threads), smem, s, a);
  return launch_pdl(prefill_attn_kernel<128>, grid, dim3(threads), smem, s, a);
}

}  // namespace amk
