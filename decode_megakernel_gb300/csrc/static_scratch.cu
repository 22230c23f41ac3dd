// Decode step whose per-step scratch lives in a fixed array inside this
// library instead of the context's workspace.
//
// A decode step needs, besides its inputs (the loaded weights, the KV cache,
// token and position) and its output (the logits), some scratch: the tagged
// activation words (x_res, x_mid, qkv, o, a, attention partials) and a
// status word.  amk_decode_step keeps them in the workspace
// the caller handed to amk_load_weights.  amk_decode_step_static_scratch
// takes them from g_step_scratch below, a file-scope device array that
// every GPU loading this library holds until the process exits.  It calls
// no allocating routine (no cudaMalloc / cudaFree / cudaMallocAsync, no
// allocating library call).
#include <cuda_runtime.h>

#include <cstdio>

#include "../../include/amk.h"
#include "device_model.hpp"

namespace amk {

amk_status internal_begin_step(amk_ctx* ctx, int32_t token, int32_t pos, const float* logits,
                               DevModel* dm, StepScratchPlan* plan);
amk_status internal_launch_fresh(amk_ctx* ctx, const DevModel& dm, int32_t token, int32_t pos,
                                 float* logits);
amk_status internal_end_step(amk_ctx* ctx, int32_t pos, const uint32_t status[4]);
amk_status internal_fail(amk_ctx* ctx, amk_status st, const char* msg);
amk_status internal_poison(amk_ctx* ctx, cudaError_t e, const char* what);

// 1 MiB: an 8B-shape model with 19 attention splits per KV head needs ~450 KB.
constexpr size_t kStaticScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

namespace {

// Device address of g_step_scratch in the current device's context.  Host
// code may only name the array through this address: the symbol itself is a
// host-side stand-in.  Looked up on every call (the lookup allocates
// nothing), so that an address never outlives the context it belongs to
// (after a cudaDeviceReset the library's device code is loaded anew, at a
// new address).
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace amk

using namespace amk;

extern "C" amk_status amk_decode_step_static_scratch(amk_ctx* ctx, int32_t token, int32_t pos,
                                                     float* logits_dev) {
  DevModel dm;
  StepScratchPlan plan;
  amk_status st = internal_begin_step(ctx, token, pos, logits_dev, &dm, &plan);
  if (st != AMK_OK) return st;
  if (plan.total > kStaticScratchBytes) {
    char msg[192];
    snprintf(msg, sizeof msg,
             "this model needs %zu bytes of per-step scratch; the static scratch holds at most %zu",
             plan.total, kStaticScratchBytes);
    return internal_fail(ctx, AMK_ERR_OOM, msg);
  }
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    return internal_fail(ctx, AMK_ERR_CUDA, msg);
  }
  uint8_t* b = static_cast<uint8_t*>(base);
  dm.xres = reinterpret_cast<uint32_t*>(b + plan.xres);
  dm.xmid = reinterpret_cast<uint32_t*>(b + plan.xmid);
  dm.qkv = reinterpret_cast<uint32_t*>(b + plan.qkv);
  dm.o = reinterpret_cast<uint32_t*>(b + plan.o);
  dm.a = reinterpret_cast<uint32_t*>(b + plan.a);
  dm.part = reinterpret_cast<uint32_t*>(b + plan.part);
  dm.status = reinterpret_cast<uint32_t*>(b + plan.status);
  cudaStream_t s = static_cast<cudaStream_t>(plan.stream);

  // The array keeps whatever the previous call left.  Every call runs as
  // launch 1, so a previous call's words carry exactly the version tags
  // this one waits for: the whole plan (tagged words and status) is zeroed
  // first, and tag 0 is never a version's tag.
  e = cudaMemsetAsync(b, 0, plan.total, s);
  if (e != cudaSuccess) return internal_fail(ctx, AMK_ERR_CUDA, "clearing the static scratch failed");
  st = internal_launch_fresh(ctx, dm, token, pos, logits_dev);
  if (st != AMK_OK) return st;
  uint32_t status[4] = {0, 0, 0, 0};
  e = cudaMemcpyAsync(status, dm.status, sizeof status, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return internal_poison(ctx, e, "reading the step status");
  return internal_end_step(ctx, pos, status);
}
