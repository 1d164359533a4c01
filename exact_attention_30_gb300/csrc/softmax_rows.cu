// softmax_rows.cu -- fused row softmax: Y[r, :] = softmax(scale * X[r, :]).
//
// The fusion example of "FlashAttention and Triton" §19.11: one pass per row
// that loads the row (a ragged tail reads as -inf), subtracts the row max,
// exponentiates, sums and divides, so the row crosses HBM once on the way in
// and once on the way out, instead of the several round trips of a composed
// max / sub / exp / sum / div sequence. exp(scale*(x - m)) is computed as
// 2^((x - m) * scale*log2(e)) with the hardware exp2.
//
// Layout: X, Y dense row-major [rows, cols]; fp32 or bf16 in and out,
// arithmetic in fp32.
//  * cols <= 2048: one warp per row, the row held in registers
//    (VPL = values per lane); 16-byte loads/stores when rows are 16-byte
//    aligned, scalar otherwise.
//  * 2048 < cols <= 32768: one block of 256-1024 threads per row, the row
//    held in registers (16 or 32 values per thread), reductions through
//    shared memory.
// HBM-bound: rows * cols * (bytes in + bytes out) per call. X and Y may be
// the same buffer: every thread reads its elements before it writes any.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row. Element e of the row is held by lane (e / VEC) % 32 in
// slot ((e / VEC) / 32) * VEC + e % VEC, so that each lane's VEC elements are
// contiguous (one 16-byte access when VECTOR).
template <typename T, int VPL, bool VECTOR>
__global__ void __launch_bounds__(256) softmax_warp_kernel(const T* X, T* Y,
                                                           int rows, int cols, float scale_log2) {
  constexpr int VEC = 16 / sizeof(T);  // elements per 16-byte access
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const T* x = X + (size_t)warp * cols;
  T* y = Y + (size_t)warp * cols;
  float v[VPL];
#pragma unroll
  for (int g = 0; g < VPL / VEC; ++g) {
    const int e0 = (g * 32 + lane) * VEC;
    if (VECTOR && e0 + VEC <= cols) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + e0);
      const T* t = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int k = 0; k < VEC; ++k) v[g * VEC + k] = to_f<T>(t[k]);
    } else {
#pragma unroll
      for (int k = 0; k < VEC; ++k) v[g * VEC + k] = (e0 + k < cols) ? to_f<T>(x[e0 + k]) : -INFINITY;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < VPL; ++k) m = fmaxf(m, v[k]);
  m = warp_max(m);
  const float nm = -m * scale_log2;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPL; ++k) {
    v[k] = ex2_approx(fmaf(v[k], scale_log2, nm));  // -inf -> 0
    s += v[k];
  }
  const float inv = 1.f / warp_sum(s);
#pragma unroll
  for (int g = 0; g < VPL / VEC; ++g) {
    const int e0 = (g * 32 + lane) * VEC;
    if (VECTOR && e0 + VEC <= cols) {
      uint4 u;
      T* t = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int k = 0; k < VEC; ++k) t[k] = from_f<T>(v[g * VEC + k] * inv);
      *reinterpret_cast<uint4*>(y + e0) = u;
    } else {
#pragma unroll
      for (int k = 0; k < VEC; ++k)
        if (e0 + k < cols) y[e0 + k] = from_f<T>(v[g * VEC + k] * inv);
    }
  }
}

// One block of THREADS threads per row, the row held in registers (VPT
// values per thread, in groups of VEC contiguous elements: element
// (g * THREADS + tid) * VEC + k). Max and sum are reduced within each warp by
// shuffles, then across warps through shared memory.
template <typename T, int THREADS, int VPT, bool VECTOR>
__global__ void __launch_bounds__(THREADS) softmax_block_kernel(const T* X, T* Y, int cols,
                                                                float scale_log2) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int NW = THREADS / 32;
  __shared__ float red_m[NW], red_s[NW];
  const T* x = X + (size_t)blockIdx.x * cols;
  T* y = Y + (size_t)blockIdx.x * cols;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float v[VPT];
#pragma unroll
  for (int g = 0; g < VPT / VEC; ++g) {
    const int e0 = (g * THREADS + tid) * VEC;
    if (VECTOR && e0 + VEC <= cols) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + e0);
      const T* t = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int k = 0; k < VEC; ++k) v[g * VEC + k] = to_f<T>(t[k]);
    } else {
#pragma unroll
      for (int k = 0; k < VEC; ++k) v[g * VEC + k] = (e0 + k < cols) ? to_f<T>(x[e0 + k]) : -INFINITY;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < VPT; ++k) m = fmaxf(m, v[k]);
  m = warp_max(m);
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  m = warp_max(lane < NW ? red_m[lane] : -INFINITY);
  const float nm = -m * scale_log2;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    v[k] = ex2_approx(fmaf(v[k], scale_log2, nm));  // -inf -> 0
    s += v[k];
  }
  s = warp_sum(s);
  if (lane == 0) red_s[warp] = s;
  __syncthreads();
  const float inv = 1.f / warp_sum(lane < NW ? red_s[lane] : 0.f);
#pragma unroll
  for (int g = 0; g < VPT / VEC; ++g) {
    const int e0 = (g * THREADS + tid) * VEC;
    if (VECTOR && e0 + VEC <= cols) {
      uint4 u;
      T* t = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int k = 0; k < VEC; ++k) t[k] = from_f<T>(v[g * VEC + k] * inv);
      *reinterpret_cast<uint4*>(y + e0) = u;
    } else {
#pragma unroll
      for (int k = 0; k < VEC; ++k)
        if (e0 + k < cols) y[e0 + k] = from_f<T>(v[g * VEC + k] * inv);
    }
  }
}

template <typename T, int THREADS, int VPT>
cudaError_t launch_block(const T* X, T* Y, int rows, int cols, float sl2, bool vector, cudaStream_t st) {
  if (vector) softmax_block_kernel<T, THREADS, VPT, true><<<rows, THREADS, 0, st>>>(X, Y, cols, sl2);
  else softmax_block_kernel<T, THREADS, VPT, false><<<rows, THREADS, 0, st>>>(X, Y, cols, sl2);
  return cudaGetLastError();
}

template <typename T, int VPL>
cudaError_t launch_warp(const T* X, T* Y, int rows, int cols, float sl2, bool vector, cudaStream_t st) {
  const unsigned blocks = (unsigned)(((long long)rows * 32 + 255) / 256);
  if (vector) softmax_warp_kernel<T, VPL, true><<<blocks, 256, 0, st>>>(X, Y, rows, cols, sl2);
  else softmax_warp_kernel<T, VPL, false><<<blocks, 256, 0, st>>>(X, Y, rows, cols, sl2);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void* Xv, void* Yv, int rows, int cols, float scale, cudaStream_t st) {
  const T* X = static_cast<const T*>(Xv);
  T* Y = static_cast<T*>(Yv);
  constexpr int VEC = 16 / sizeof(T);
  const float sl2 = scale * kLog2e;
  const bool vector = (cols % VEC == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(Y) % 16 == 0);
  // values per lane: the smallest of 4, 8, 16, 32, 64 (a multiple of VEC)
  // with 32 * VPL >= cols
  const int need = (cols + 31) / 32;
  constexpr int V4 = VEC > 4 ? VEC : 4;
  if (need <= 4) return launch_warp<T, V4>(X, Y, rows, cols, sl2, vector, st);
  if (need <= 8) return launch_warp<T, 8>(X, Y, rows, cols, sl2, vector, st);
  if (need <= 16) return launch_warp<T, 16>(X, Y, rows, cols, sl2, vector, st);
  if (need <= 32) return launch_warp<T, 32>(X, Y, rows, cols, sl2, vector, st);
  if (need <= 64) return launch_warp<T, 64>(X, Y, rows, cols, sl2, vector, st);
  // longer rows: one block per row, 16 or 32 values per thread
  if (cols <= 256 * 16) return launch_block<T, 256, 16>(X, Y, rows, cols, sl2, vector, st);
  if (cols <= 512 * 16) return launch_block<T, 512, 16>(X, Y, rows, cols, sl2, vector, st);
  if (cols <= 1024 * 16) return launch_block<T, 1024, 16>(X, Y, rows, cols, sl2, vector, st);
  return launch_block<T, 1024, 32>(X, Y, rows, cols, sl2, vector, st);
}

}  // namespace

cudaError_t launch_softmax_rows(const void* X, void* Y, int rows, int cols, float scale, bool bf16,
                                cudaStream_t st) {
  return bf16 ? launch_t<__nv_bfloat16>(X, Y, rows, cols, scale, st)
              : launch_t<float>(X, Y, rows, cols, scale, st);
}

}  // namespace fa
