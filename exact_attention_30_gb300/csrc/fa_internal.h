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

// Bounded-wait probe (fa_debug_timeout_probe).
cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace fa
