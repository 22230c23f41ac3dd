// Tensor-core prefill: the K,V rows of a prompt for every layer, computed
// over a chunk of tokens at once with GEMMs on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA)
// instead of one decode step per token.  Same math as the decode step,
// batched and causal (the AMK pages leave prefill open; their decode task
// graph is the batch-1 special case of this one).
//
// Per chunk of T <= chunk tokens at positions s0 .. s0 + T - 1:
//   X = E[tokens]                                            (fp32 [T][H])
//   per layer l:
//     H1 = rmsnorm(X) * w_attn[l]            as bf16 parts [T][H]
//     QKV GEMM, epilogue: RoPE; q -> Q (fp32 [T][n_heads * hd]); k, v ->
//       the KV cache (bf16) at positions s0 + t
//     (last layer: stop, the rest of it feeds no K,V)
//     attention (causal over positions 0 .. s0 + t, GQA) -> O, bf16 parts
//     X += O Wo^T;  H1 = rmsnorm(X) * w_ffn[l]
//     gate/up GEMM, epilogue silu(g) * u -> A, bf16 parts [T][F]
//     X += A Wd^T
// Every GEMM activation operand is split into bf16 parts, x = p0 + p1 (+
// p2) to 2^-18 (2^-27) relative (p0 = bf16(x), p1 = bf16(x - p0), p2 =
// bf16(x - p0 - p1); each subtraction is exact in fp32), and the parts are
// multiplied against the bf16 weights into one fp32 accumulator.  Three
// parts carry the activation's full fp32 precision, as the decode kernel's
// fp32 GEMVs do; two parts (the default) take two thirds of the tensor work
// (measured on the 8B shape: 50 instead of 71 ms for 2048 tokens) and leave
// ~0.3% of the first layer's bf16 K,V one step off the fp32 path (three
// parts: ~0.04%).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace amk {

constexpr int kPfBM = 128;      // tokens per GEMM tile (MMA M, TMEM lanes)
constexpr int kPfBN = 256;      // packed weight rows per GEMM tile at most (MMA N, TMEM columns)
constexpr int kPfBNNarrow = 224;   // the narrower tile width (a multiple of every Rt)
constexpr int kPfBK = 64;       // k per pipeline stage: one 128-byte swizzled row
constexpr int kPfParts = 3;     // bf16 parts of a GEMM activation operand at most (buffers, maps)
constexpr int kPfDefaultParts = 2;
// The tensor cores' fp32 accumulation truncates (measured: a bias toward
// zero that grows with K, ~1e-7 of the sum of |terms| at K = 4096 against
// ~1e-10 for an fp32 FMA chain), so the GEMM accumulates in TMEM only over
// segments of kPfSegKB k blocks (128 k) and promotes each segment's partial
// sums into fp32 registers of the epilogue warps, two TMEM buffers
// alternating so that the MMAs never wait for the promotion.
constexpr int kPfSegKB = 2;
// epilogue warps: two per TMEM lane quarter, each owning 128 accumulator columns
constexpr int kPfEpiWarps = 8;
constexpr int kPfGemmThreads = 64 + 32 * kPfEpiWarps;   // TMA warp, MMA warp, epilogue warps
constexpr int kPfQT = 16;       // query tokens of one attention warp (one m16 tile of one head)
constexpr int kPfKB = 32;       // cached positions per attention key block (two CTAs of 8 warps per SM)
constexpr int kPfDefaultChunk = 2048;

enum PrefillEpi : int32_t { PE_QKV = 0, PE_RESID = 1, PE_SWIGLU = 2 };

// One GEMM D[T][N] = A[T][K] . W[N][K]^T over a packed weight matrix and its
// epilogue.  A arrives through kPfParts 2-D tensor maps (its bf16 parts,
// each [rows][K], boxes of 64 x 128, 128-byte swizzle); W through a 4-D map
// over the decode kernel's tile layout ({Kt, Rt, nkt, n_rb}, boxes
// {64, Rt, 1, bn / Rt}, bn = kPfBN or kPfBNNarrow rows).
struct PrefillGemm {
  int32_t T;              // tokens (rows of D that are stored)
  int32_t N;              // packed weight rows (columns of D that are used)
  int32_t nk;             // k blocks of kPfBK over the padded K
  int32_t Kt, Rt;         // packed tile geometry of the weight matrix
  int32_t layer, s0;      // layer; position of token 0
  int32_t hd, group, n_kv, max_seq;
  float* x;               // PE_RESID: residual rows [T][ldx], += D
  int32_t ldx;
  float* q;               // PE_QKV: rotated q rows [T][ldq]
  int32_t ldq;
  uint16_t* kv;           // PE_QKV: KV cache bf16 [L][2][n_kv][max_seq][hd]
  const float2* rope;     // PE_QKV: (cos, sin) [max_seq][hd / 2]
  uint16_t* out[kPfParts];   // PE_SWIGLU: silu(g) * u as bf16 parts [T][ldo]
  int32_t ldo;
  int32_t parts;          // bf16 parts of the activations (2 or 3)
  uint32_t* status;       // device status words (a timed-out wait records ST_TIMEOUT)
  uint64_t timeout_ns;
  int32_t ctas;           // persistent CTAs (at most one per SM; fewer when there are fewer tiles)
};

// Causal GQA attention of a chunk: queries Q (fp32, RoPE applied) of
// tokens [0, T) at positions s0 + t against the cache's K,V of positions
// [0, s0 + t]; output O as bf16 parts [T][ldo] in head order.
struct PrefillAttn {
  const float* q;
  int32_t ldq;
  const uint16_t* kv;
  int32_t layer, n_kv, max_seq, group, hd;
  int32_t T, s0;
  uint16_t* o[kPfParts];
  int32_t ldo;
  int32_t parts;          // bf16 parts written (2 or 3)
  uint32_t* status;       // device status words (a timed-out wait records ST_TIMEOUT)
  uint64_t timeout_ns;
};

// Attention on the 5th-generation tensor cores (prefill_attn_tc_kernel):
// one CTA per 128 query rows (128 / group tokens x the group's query
// heads) and KV head, K,V blocks of kTcKeys positions by TMA.  Taken when
// head_dim is 64 or 128, the group divides 128 and the cache holds at least
// kTcKeys positions after the chunk (s0 + T >= kTcKeys: every key window
// lies inside written positions); otherwise the mma.sync kernel runs.
constexpr int kTcRows = 128;
constexpr int kTcKeys = 64;
bool prefill_attn_uses_tc(int head_dim, int group, int s0, int T);

int prefill_gemm_smem_bytes(int parts, int bn);

// Tile width of a GEMM with n_rows packed weight rows over T tokens on
// `sms` SMs: kPfBN or kPfBNNarrow, whichever finishes first when every SM
// runs one tile at a time and a tile takes time in proportion to its
// width (ceil(tiles / sms) rounds of width bn); ties go to kPfBN.
int prefill_gemm_bn(int n_rows, int T, int sms);
int prefill_attn_smem_bytes(int head_dim, int group);

// X[t][:] = float(embed[tokens[t]][:]) for t < T
cudaError_t launch_prefill_embed(const int32_t* tokens, int T, const uint16_t* embed, int hidden,
                                 float* x, cudaStream_t s);
// out[i][t][:] = the bf16 parts of rmsnorm(X[t]) * w for t < T (row stride hidden)
cudaError_t launch_prefill_norm(const float* x, int T, int hidden, const uint16_t* w, float eps,
                                uint16_t* const* out, int parts, cudaStream_t s);
// a: the g.parts tensor maps of the activation parts; w: the weight map,
// encoded with boxes of bn rows (kPfBN or kPfBNNarrow)
cudaError_t launch_prefill_gemm(int epi, const CUtensorMap* a, const CUtensorMap* w, int bn, const PrefillGemm& g,
                                cudaStream_t s);
// kv_map: the KV cache as rows of head_dim bf16 ([L][2][n_kv][max_seq]
// rows), boxes of 64 dims x kTcKeys rows, 128-byte swizzle (for the
// tensor-core kernel)
cudaError_t launch_prefill_attn(const PrefillAttn& a, const CUtensorMap* kv_map, cudaStream_t s);

}  // namespace amk
