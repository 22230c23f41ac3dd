// Read-only HBM stream probe: the rate at which this GPU can stream a
// buffer it only reads, the denominator the decode kernel's weight stream
// actually competes against (a copy moves the same bytes twice).
//
// Two ways of reading, timed by the caller on the launch stream:
//   mode 0  one CTA per SM, one thread keeping a ring of eight 16 KB
//           cp.async.bulk copies in flight into shared memory (the decode
//           kernel's producer pattern without its consumers);
//   mode 1  a grid of 128-bit non-caching global loads, grid-stride.
// Each CTA folds a few words of what it read into a checksum so that no
// load can be dropped.  Every mbarrier wait is bounded by %globaltimer.
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace amk {

namespace {

constexpr int kProbeSlots = 8;
constexpr uint32_t kProbeTile = 16384;

__device__ __forceinline__ void probe_bar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void probe_bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// bounded wait for the phase of `bar` with the given parity
__device__ __forceinline__ bool probe_wait(uint64_t* bar, uint32_t parity, uint64_t t0, uint64_t timeout_ns) {
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try_wait32(smem_addr(bar), parity)) return true;
    if ((spin & 15u) == 15u && global_timer() - t0 > timeout_ns) return false;
  }
}

__global__ void __launch_bounds__(32, 1)
    hbm_probe_bulk_kernel(const uint8_t* buf, uint64_t bytes, uint32_t* out, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kProbeSlots];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kProbeSlots; ++s) probe_bar_init(&full[s]);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  // this CTA's share: whole tiles, contiguous
  const uint64_t tiles = bytes / kProbeTile;
  const uint64_t per = (tiles + gridDim.x - 1) / gridDim.x;
  const uint64_t t_begin = (uint64_t)blockIdx.x * per;
  const uint64_t t_end = t_begin + per < tiles ? t_begin + per : tiles;
  uint32_t sum = 0;
  uint32_t issued = 0;               // slots holding a copy that has not been waited for
  uint32_t last_use[kProbeSlots];    // use index of each slot's latest copy
  for (int s = 0; s < kProbeSlots; ++s) last_use[s] = 0;
  const uint64_t t0 = global_timer();
  bool ok = true;
  for (uint64_t t = t_begin; t < t_end && ok; ++t) {
    const uint32_t slot = (uint32_t)((t - t_begin) % kProbeSlots);
    const uint32_t use = (uint32_t)((t - t_begin) / kProbeSlots);   // uses of this slot so far
    if (use > 0) {
      ok = probe_wait(&full[slot], (use - 1) & 1u, t0, timeout_ns);
      if (!ok) break;
      sum ^= *reinterpret_cast<const uint32_t*>(ring + slot * kProbeTile + (t & 63u) * 4u);
      issued &= ~(1u << slot);
    }
    probe_bulk(ring + slot * kProbeTile, buf + t * kProbeTile, kProbeTile, &full[slot]);
    issued |= 1u << slot;
    last_use[slot] = use;
  }
  // wait for the copies still in flight (their shared memory must not go away)
  for (uint32_t slot = 0; slot < kProbeSlots; ++slot) {
    if (!(issued & (1u << slot))) continue;
    if (!probe_wait(&full[slot], last_use[slot] & 1u, global_timer(), timeout_ns)) ok = false;
    else sum ^= *reinterpret_cast<const uint32_t*>(ring + slot * kProbeTile);
  }
  out[2 * blockIdx.x] = sum;
  out[2 * blockIdx.x + 1] = ok ? 0u : 1u;
}

__global__ void __launch_bounds__(512)
    hbm_probe_ld_kernel(const uint4* buf, uint64_t n_vec, uint32_t* out) {
  uint32_t sum = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint64_t j = i + u * stride;
      if (j < n_vec) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                     : "l"(buf + j));
      } else {
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) sum ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  sum = __reduce_xor_sync(0xFFFFFFFFu, sum);
  if ((threadIdx.x & 31) == 0) atomicXor(&out[2 * blockIdx.x], sum);
}

}  // namespace

int hbm_probe_smem_bytes() { return kProbeSlots * (int)kProbeTile; }

// out: 2 words per CTA (checksum, failure flag), >= 2 * grid words, zeroed by
// the caller for mode 1.  Returns the CUDA launch error.
cudaError_t launch_hbm_probe(int mode, const void* buf, uint64_t bytes, uint32_t* out, int sms,
                             uint64_t timeout_ns, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mode == 0) {
    const int smem = hbm_probe_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(hbm_probe_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    hbm_probe_bulk_kernel<<<sms, 32, smem, s>>>(static_cast<const uint8_t*>(buf), bytes, out, timeout_ns);
  } else {
    hbm_probe_ld_kernel<<<sms * 4, 512, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16, out);
  }
  return cudaGetLastError();
}

}  // namespace amk
