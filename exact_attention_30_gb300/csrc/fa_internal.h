// fa_internal.h -- launch functions shared between the C-ABI layer (fa_api.cu)
// and the kernel translation units. Host-side only declarations; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Upper bound for any single mbarrier wait inside a kernel, in nanoseconds.
// Past it the kernel records FA_ERR_TIMEOUT in the status word and exits.
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;  // 1 s

// Device-side status word of the current device (created on first use).
int* device_status_ptr();

// ---- fp32 CUDA-core path (attn_f32.cu) ----
cudaError_t launch_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                           int BH, int N, int d, float scale, cudaStream_t st);
// Backward stage bits: preprocess, main, dQ convert.
enum : unsigned { kStagePre = 1u, kStageMain = 2u, kStageConvert = 4u, kStageAll = 7u };
cudaError_t launch_bwd_f32(const float* Q, const float* K, const float* V, const float* O,
                           const float* dO, const float* LSE, float* dQ, float* dK, float* dV,
                           float* Dws, int BH, int N, int d, float scale, unsigned stages,
                           cudaStream_t st);

// ---- bf16 tcgen05 path ----
// Tensor maps describe one [BH, N, d] bf16 tensor as 3-D (d, N, BH) with
// 64-element x 128-row boxes and 128-byte swizzle.
struct FwdArgs {
  CUtensorMap tmQ, tmK, tmV;
  void* O;      // bf16 [BH, N, d]
  float* LSE;   // [BH, N]
  int N;
  float scale_log2;  // scale * log2(e)
  int* status;
  unsigned long long wait_limit_ns;
};
cudaError_t launch_fwd_bf16(const FwdArgs& a, int BH, int d, cudaStream_t st);

struct BwdArgs {
  CUtensorMap tmQ, tmK, tmV, tmdO;
  CUtensorMap tmDQacc;  // fp32 [BH*Npad, d], 32 x 32 boxes, no swizzle (d = 128 only)
  const void* O;     // bf16 [BH, N, d]
  const void* dO;    // bf16 [BH, N, d]
  const float* LSE;  // [BH, N]
  void* dQ;          // bf16 [BH, N, d]
  void* dK;          // bf16 [BH, N, d]
  void* dV;          // bf16 [BH, N, d]
  float* dQacc;      // fp32 [BH, Npad, d]
  float* lse2;       // fp32 [BH, Npad]  LSE * log2(e); +inf past N
  float* Drow;       // fp32 [BH, Npad]  rowsum(dO o O); 0 past N
  int N, Npad;
  float scale;
  float scale_log2;
  int* status;
  unsigned long long wait_limit_ns;
};
cudaError_t launch_bwd_bf16(const BwdArgs& a, int BH, int d, unsigned stages, cudaStream_t st);
// Row padding used by the bf16 backward workspace.
constexpr int kBwdRowPad = 128;
// Query rows per streamed tile of the bf16 backward kernel (its Q/dO TMA box
// height); must match BwdCfg<d>::BQ.
constexpr int bwd_query_tile(int d) { return d > 0 ? 128 : 128; }

// Fused row softmax (softmax_rows.cu): rows x cols, fp32 or bf16, cols <= 32768.
constexpr int kSoftmaxMaxCols = 32768;
cudaError_t launch_softmax_rows(const void* X, void* Y, int rows, int cols, float scale, bool bf16,
                                cudaStream_t st);

// ---- KV-cache decode (decode_splitkv.cu) ----
constexpr int kDecodeMaxQueries = 8;
constexpr int kDecodeMaxSplits = 256;
struct DecodeArgs {
  CUtensorMap tmK, tmV;  // [BH, Nk, d] bf16 as 3-D (d, Nk, BH), 64 x 64 boxes, 128-byte swizzle
  const void* Q;         // bf16 [BH, Nq, d]
  void* O;               // bf16 [BH, Nq, d]
  float* LSE;            // [BH, Nq], natural log
  float* Opart;          // fp32 [splits, BH*Nq, d]: each split's normalised output
  float* LSEpart;        // fp32 [splits, BH*Nq]: each split's log-sum-exp, base 2
  int BH, Nq, Nk, splits, keys_per_split;
  float scale_log2;
  int* status;
  unsigned long long wait_limit_ns;
};
struct DecodePlan {
  int splits;          // 0 on failure
  int keys_per_split;  // a multiple of 64
};
// Split count for a problem on the current device (queries its SM count and
// the kernel's occupancy once per device).
DecodePlan plan_decode(int BH, int Nq, int Nk, int d);
// The same choice for a given number of resident CTAs on the GPU.
DecodePlan plan_decode_for_slots(int BH, int Nk, int slots);
cudaError_t launch_decode_bf16(const DecodeArgs& a, int d, cudaStream_t st);

// Bounded-wait probe (fa_debug_timeout_probe).
cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace fa
