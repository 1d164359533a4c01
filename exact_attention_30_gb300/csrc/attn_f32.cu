// attn_f32.cu -- float32 fused attention on CUDA cores (FFMA), any 1 <= d <= 128.
//
// Same algorithm as the tensor-core path: key/value tiles streamed through
// shared memory, an online softmax per query row (running max m, denominator
// l, accumulator rescaled by exp(m - m_new)), S and P never written to global
// memory ("Lesson 1: FlashAttention core idea" §3-§4). The backward pass
// rebuilds P from the saved log-sum-exp ("Lesson 1" §5).
//
// fp32 cannot go through bf16/tf32 tensor cores without losing the 1e-5
// accuracy this dtype promises, so these kernels use FFMA and the accurate
// expf/logf of the CUDA math library (this file is built without fast-math).
//
// Layout: one warp per query (forward, dQ) or key (dK/dV) row, 8 warps per
// block sharing a 32-row tile of the other operand in shared memory. Rows are
// addressed through the SeqArgs layout (fixed length or packed variable
// length); with causal attention query row r sees keys c <= r, and the key
// (query) loops stop (start) at the block's diagonal.
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.h"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int kWarps = 8;
constexpr int kTile = 32;  // rows of K/V (or Q/dO) per shared-memory tile

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

// Forward. grid = (ceil(N / kWarps), B*H), block = 32*kWarps.
// Shared: q rows [kWarps][d], K tile [kTile][d+1], V tile [kTile][d].
template <int DC>  // DC = ceil(d/32) output columns per lane
__global__ void __launch_bounds__(32 * kWarps)
fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
               const float* __restrict__ V, float* __restrict__ O, float* __restrict__ LSE,
               const SeqArgs sq, int* status, int d, float scale) {
  extern __shared__ float sm[];
  const int dp = d + 1;
  float* qs = sm;                    // kWarps * d
  float* ks = qs + kWarps * d;       // kTile * dp
  float* vs = ks + kTile * dp;       // kTile * d
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqView sv = seq_view(sq, blockIdx.y, status);
  const int N = sv.len;
  const int row0 = blockIdx.x * kWarps;
  if (row0 >= N) return;  // whole block
  const int row = row0 + warp;
  const bool live = row < N;
  const bool causal = sq.causal != 0;
  // keys this block needs: all, or up to its last row
  const int k_end = causal ? min(N, row0 + kWarps) : N;

  for (int c = lane; c < d; c += 32) qs[warp * d + c] = live ? Q[seq_row_offset(sq, sv, row) + c] : 0.f;

  float m = -INFINITY, l = 0.f;
  float acc[DC];
#pragma unroll
  for (int k = 0; k < DC; ++k) acc[k] = 0.f;

  for (int k0 = 0; k0 < k_end; k0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int r = e / d, c = e - r * d;
      const bool ok = k0 + r < N;
      ks[r * dp + c] = ok ? K[seq_row_offset(sq, sv, k0 + r) + c] : 0.f;
      vs[r * d + c] = ok ? V[seq_row_offset(sq, sv, k0 + r) + c] : 0.f;
    }
    __syncthreads();
    // lane j scores key k0 + j
    float s = -INFINITY;
    if (k0 + lane < N && (!causal || k0 + lane <= row)) {
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(qs[warp * d + c], ks[lane * dp + c], dot);
      s = dot * scale;
    }
    const float m_new = fmaxf(m, warp_max(s));
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float p = (s == -INFINITY) ? 0.f : expf(s - m_new);
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int k = 0; k < DC; ++k) acc[k] *= alpha;
    const int nk = min(kTile, N - k0);
    for (int j = 0; j < nk; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
      for (int k = 0; k < DC; ++k) {
        const int c = lane + 32 * k;
        if (c < d) acc[k] = fmaf(pj, vs[j * d + c], acc[k]);
      }
    }
    m = m_new;
  }
  if (live) {
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < DC; ++k) {
      const int c = lane + 32 * k;
      if (c < d) O[seq_row_offset(sq, sv, row) + c] = acc[k] * inv;
    }
    if (lane == 0) LSE[seq_stat_index(sq, sv, row)] = m + logf(l);
  }
}

// D_r = sum_c dO_rc * O_rc for every row of every plane (whichever sequence
// holds it). grid = (ceil(total/kWarps), planes); D has the LSE layout.
__global__ void __launch_bounds__(32 * kWarps)
bwd_pre_f32_kernel(const float* __restrict__ O, const float* __restrict__ dO,
                   float* __restrict__ Dv, const SeqArgs sq, int d) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  if (row >= sq.total) return;
  const size_t off = (size_t)blockIdx.y * (size_t)sq.plane_stride + (size_t)row * (size_t)sq.row_stride;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(dO[off + c], O[off + c], acc);
  acc = warp_sum(acc);
  if (lane == 0) Dv[(size_t)blockIdx.y * (size_t)sq.stat_plane + row] = acc;
}

// dQ_r = scale * sum_c P_rc (dP_rc - D_r) K_c, one warp per query row r.
// Shared: q, dO rows [kWarps][d] each; K, V tiles [kTile][d+1].
template <int DC>
__global__ void __launch_bounds__(32 * kWarps)
bwd_dq_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                  const float* __restrict__ V, const float* __restrict__ dO,
                  const float* __restrict__ LSE, const float* __restrict__ Dv,
                  float* __restrict__ dQ, const SeqArgs sq, int* status, int d, float scale) {
  extern __shared__ float sm[];
  const int dp = d + 1;
  float* qs = sm;
  float* dos = qs + kWarps * d;
  float* ks = dos + kWarps * d;
  float* vs = ks + kTile * dp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqView sv = seq_view(sq, blockIdx.y, status);
  const int N = sv.len;
  const int row0 = blockIdx.x * kWarps;
  if (row0 >= N) return;  // whole block
  const int row = row0 + warp;
  const bool live = row < N;
  const bool causal = sq.causal != 0;
  const int k_end = causal ? min(N, row0 + kWarps) : N;
  for (int c = lane; c < d; c += 32) {
    qs[warp * d + c] = live ? Q[seq_row_offset(sq, sv, row) + c] : 0.f;
    dos[warp * d + c] = live ? dO[seq_row_offset(sq, sv, row) + c] : 0.f;
  }
  const float lse = live ? LSE[seq_stat_index(sq, sv, row)] : 0.f;
  const float Dr = live ? Dv[seq_stat_index(sq, sv, row)] : 0.f;
  float acc[DC];
#pragma unroll
  for (int k = 0; k < DC; ++k) acc[k] = 0.f;

  for (int k0 = 0; k0 < k_end; k0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int r = e / d, c = e - r * d;
      const bool ok = k0 + r < N;
      ks[r * dp + c] = ok ? K[seq_row_offset(sq, sv, k0 + r) + c] : 0.f;
      vs[r * dp + c] = ok ? V[seq_row_offset(sq, sv, k0 + r) + c] : 0.f;
    }
    __syncthreads();
    float ds = 0.f;
    if (live && k0 + lane < N && (!causal || k0 + lane <= row)) {
      float s = 0.f, dpv = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(qs[warp * d + c], ks[lane * dp + c], s);
        dpv = fmaf(dos[warp * d + c], vs[lane * dp + c], dpv);
      }
      const float p = expf(s * scale - lse);
      ds = p * (dpv - Dr) * scale;
    }
    const int nk = min(kTile, N - k0);
    for (int j = 0; j < nk; ++j) {
      const float dsj = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
      for (int k = 0; k < DC; ++k) {
        const int c = lane + 32 * k;
        if (c < d) acc[k] = fmaf(dsj, ks[j * dp + c], acc[k]);
      }
    }
  }
  if (live) {
#pragma unroll
    for (int k = 0; k < DC; ++k) {
      const int c = lane + 32 * k;
      if (c < d) dQ[seq_row_offset(sq, sv, row) + c] = acc[k];
    }
  }
}

// dV_c = sum_r P_rc dO_r and dK_c = scale * sum_r P_rc (dP_rc - D_r) Q_r,
// one warp per key row c. Shared: k, v rows [kWarps][d]; Q, dO tiles
// [kTile][d+1]; LSE, D tile [kTile].
template <int DC>
__global__ void __launch_bounds__(32 * kWarps)
bwd_dkdv_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                    const float* __restrict__ V, const float* __restrict__ dO,
                    const float* __restrict__ LSE, const float* __restrict__ Dv,
                    float* __restrict__ dK, float* __restrict__ dV, const SeqArgs sq, int* status,
                    int d, float scale) {
  extern __shared__ float sm[];
  const int dp = d + 1;
  float* ksr = sm;
  float* vsr = ksr + kWarps * d;
  float* qs = vsr + kWarps * d;
  float* dos = qs + kTile * dp;
  float* ls = dos + kTile * dp;
  float* Ds = ls + kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqView sv = seq_view(sq, blockIdx.y, status);
  const int N = sv.len;
  const int c0 = blockIdx.x * kWarps;
  if (c0 >= N) return;  // whole block
  const int col = c0 + warp;  // key row
  const bool live = col < N;
  const bool causal = sq.causal != 0;
  // queries this block needs: all, or from its first key on
  const int r_begin = causal ? c0 / kTile * kTile : 0;
  for (int c = lane; c < d; c += 32) {
    ksr[warp * d + c] = live ? K[seq_row_offset(sq, sv, col) + c] : 0.f;
    vsr[warp * d + c] = live ? V[seq_row_offset(sq, sv, col) + c] : 0.f;
  }
  float adk[DC], adv[DC];
#pragma unroll
  for (int k = 0; k < DC; ++k) adk[k] = adv[k] = 0.f;

  for (int r0 = r_begin; r0 < N; r0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * d; e += blockDim.x) {
      const int r = e / d, c = e - r * d;
      const bool ok = r0 + r < N;
      qs[r * dp + c] = ok ? Q[seq_row_offset(sq, sv, r0 + r) + c] : 0.f;
      dos[r * dp + c] = ok ? dO[seq_row_offset(sq, sv, r0 + r) + c] : 0.f;
    }
    for (int r = threadIdx.x; r < kTile; r += blockDim.x) {
      const bool ok = r0 + r < N;
      ls[r] = ok ? LSE[seq_stat_index(sq, sv, r0 + r)] : 0.f;
      Ds[r] = ok ? Dv[seq_stat_index(sq, sv, r0 + r)] : 0.f;
    }
    __syncthreads();
    float p = 0.f, ds = 0.f;
    if (live && r0 + lane < N && (!causal || r0 + lane >= col)) {
      float s = 0.f, dpv = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(qs[lane * dp + c], ksr[warp * d + c], s);
        dpv = fmaf(dos[lane * dp + c], vsr[warp * d + c], dpv);
      }
      p = expf(s * scale - ls[lane]);
      ds = p * (dpv - Ds[lane]) * scale;
    }
    const int nr = min(kTile, N - r0);
    for (int i = 0; i < nr; ++i) {
      const float pi = __shfl_sync(0xffffffffu, p, i);
      const float dsi = __shfl_sync(0xffffffffu, ds, i);
#pragma unroll
      for (int k = 0; k < DC; ++k) {
        const int c = lane + 32 * k;
        if (c < d) {
          adv[k] = fmaf(pi, dos[i * dp + c], adv[k]);
          adk[k] = fmaf(dsi, qs[i * dp + c], adk[k]);
        }
      }
    }
  }
  if (live) {
#pragma unroll
    for (int k = 0; k < DC; ++k) {
      const int c = lane + 32 * k;
      if (c < d) {
        dK[seq_row_offset(sq, sv, col) + c] = adk[k];
        dV[seq_row_offset(sq, sv, col) + c] = adv[k];
      }
    }
  }
}

template <typename Kern>
cudaError_t set_smem(Kern kern, size_t smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int DC>
cudaError_t fwd_f32_dc(const float* Q, const float* K, const float* V, float* O, float* LSE,
                       const SeqArgs& sq, int* status, int BH, int d, float scale, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)kWarps * d + (size_t)kTile * (d + 1) + (size_t)kTile * d);
  dim3 grid((sq.N + kWarps - 1) / kWarps, BH);
  cudaError_t e = set_smem(fwd_f32_kernel<DC>, smem);
  if (e != cudaSuccess) return e;
  fwd_f32_kernel<DC><<<grid, 32 * kWarps, smem, st>>>(Q, K, V, O, LSE, sq, status, d, scale);
  return cudaGetLastError();
}

template <int DC>
cudaError_t bwd_f32_dc(const float* Q, const float* K, const float* V, const float* O,
                       const float* dO, const float* LSE, float* dQ, float* dK, float* dV,
                       float* Dws, const SeqArgs& sq, int* status, int BH, int d, float scale,
                       unsigned stages, cudaStream_t st) {
  dim3 grid((sq.N + kWarps - 1) / kWarps, BH);
  cudaError_t e = cudaSuccess;
  if (stages & kStagePre) {
    const int planes = sq.cu_seqlens ? sq.H : BH;
    bwd_pre_f32_kernel<<<dim3((sq.total + kWarps - 1) / kWarps, planes), 32 * kWarps, 0, st>>>(
        O, dO, Dws, sq, d);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (!(stages & kStageMain)) return cudaSuccess;  // the fp32 path has no separate convert
  const size_t smem_dq = sizeof(float) * (2 * (size_t)kWarps * d + 2 * (size_t)kTile * (d + 1));
  e = set_smem(bwd_dq_f32_kernel<DC>, smem_dq);
  if (e != cudaSuccess) return e;
  bwd_dq_f32_kernel<DC><<<grid, 32 * kWarps, smem_dq, st>>>(Q, K, V, dO, LSE, Dws, dQ, sq, status, d,
                                                             scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem_kv =
      sizeof(float) * (2 * (size_t)kWarps * d + 2 * (size_t)kTile * (d + 1) + 2 * (size_t)kTile);
  e = set_smem(bwd_dkdv_f32_kernel<DC>, smem_kv);
  if (e != cudaSuccess) return e;
  bwd_dkdv_f32_kernel<DC><<<grid, 32 * kWarps, smem_kv, st>>>(Q, K, V, dO, LSE, Dws, dK, dV, sq,
                                                               status, d, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                           const SeqArgs& sq, int* status, int BH, int d, float scale,
                           cudaStream_t st) {
  if (d <= 32) return fwd_f32_dc<1>(Q, K, V, O, LSE, sq, status, BH, d, scale, st);
  if (d <= 64) return fwd_f32_dc<2>(Q, K, V, O, LSE, sq, status, BH, d, scale, st);
  return fwd_f32_dc<4>(Q, K, V, O, LSE, sq, status, BH, d, scale, st);
}

cudaError_t launch_bwd_f32(const float* Q, const float* K, const float* V, const float* O,
                           const float* dO, const float* LSE, float* dQ, float* dK, float* dV,
                           float* Dws, const SeqArgs& sq, int* status, int BH, int d, float scale,
                           unsigned stages, cudaStream_t st) {
  if (d <= 32)
    return bwd_f32_dc<1>(Q, K, V, O, dO, LSE, dQ, dK, dV, Dws, sq, status, BH, d, scale, stages, st);
  if (d <= 64)
    return bwd_f32_dc<2>(Q, K, V, O, dO, LSE, dQ, dK, dV, Dws, sq, status, BH, d, scale, stages, st);
  return bwd_f32_dc<4>(Q, K, V, O, dO, LSE, dQ, dK, dV, Dws, sq, status, BH, d, scale, stages, st);
}

}  // namespace fa
