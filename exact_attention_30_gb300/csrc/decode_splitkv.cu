// decode_splitkv.cu -- attention of a few new queries against a long key/value
// cache, split along the keys.
//
// What it computes: for each (batch, head) and each of Nq <= 16 queries,
//   O = softmax(scale * q K^T) V  and  LSE = ln sum_j exp(scale * q.k_j)
// over all Nk cached keys: the inference use of "Interview Q15" (attention
// against a KV cache). The keys are cut into S contiguous splits. One CTA
// streams one split of one head and keeps, per query, the online-softmax
// state of "Lesson 1: FlashAttention core idea" §3 (running max m,
// denominator l, unnormalised output). A combine kernel merges the S partial
// results with the same rule, applied to whole splits:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  O = sum_s O_s l_s 2^(m_s - m) / l,
// where each split hands over its normalised O_s and its log-sum-exp
// m_s + log2 l_s (base-2 units inside the library).
//
// Decode is bound by HBM: each cached key and value is read once, 4 d bytes
// per key, against 4 d Nq FLOPs. With one query per head the scores and P V
// run on CUDA cores in packed f32x2 FMAs, and TMA keeps 64-key K/V tiles
// streaming through a shared-memory ring (128-byte swizzled rows: one lane
// per key reads its own row without bank conflicts). With 2..16 queries (for
// example the query heads that share one K/V head) the FMAs would no longer
// keep up with HBM, and both products run on the tensor cores instead
// (decode_tc_kernel).
//
// One query per head (decode_split_kernel below, instantiated for NQ = 1;
// several queries go to the tensor-core kernel further down): CTA of 3
// warps. Warp 2 (one lane) is the TMA producer. Warps 0 and 1 own keys
// 0-31 and 32-63 of every tile (lane = key) and keep separate online-softmax
// states; at the end warp 1 hands its state to warp 0 through shared memory
// (an mbarrier with a bounded wait) and warp 0 writes the split's result.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// tolerated growth of a query's running max (log2 units) before its output is rescaled
constexpr float kDecodeRescaleLog2 = 8.0f;

template <int D, int NQ>
struct DecCfg {
  static constexpr int BK = 64;                     // keys per tile
  static constexpr int STAGES = D == 128 ? 2 : 3;   // 2-3 CTAs per SM keep >= 2 tiles in flight each
  static constexpr int CH = D / 64;                 // 128-byte column chunks per row
  static constexpr int CHUNK = BK * 128;            // one [64 rows][128 B] swizzled chunk
  static constexpr int TILE = CH * CHUNK;           // a K or a V tile
  static constexpr int DL = D / 32;                 // output columns per lane
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_Q = OFF_V + STAGES * TILE;        // fp32 [NQ][D]
  static constexpr int OFF_P = OFF_Q + NQ * D * 4;           // fp32 [2 warps][32 keys][NQ]
  static constexpr int OFF_X = OFF_P + 2 * 32 * NQ * 4;      // warp 1 hand-over: m[NQ] l[NQ] acc[NQ][D]
  static constexpr int OFF_BAR = (OFF_X + (2 * NQ + NQ * D) * 4 + 7) / 8 * 8;
  static constexpr int NBAR = 2 * STAGES + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;   // base rounded up to 1024 (swizzle atom)
  static constexpr int THREADS = 96;
  static_assert(TILE % 1024 == 0 && OFF_Q % 16 == 0 && OFF_P % 16 == 0, "alignment");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Two bf16 (low half = lower index) widened exactly to a packed fp32 pair.
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t v) {
  return f2_pack(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

template <int D, int NQ>
__global__ void __launch_bounds__(96) decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  using C = DecCfg<D, NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  constexpr int B_FULL = 0, B_EMPTY = C::STAGES, B_MERGE = 2 * C::STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int nq = a.Nq;
  const int k_begin = split * a.keys_per_split;
  const int k_end = min(a.Nk, k_begin + a.keys_per_split);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + C::BK - 1) / C::BK : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(B_FULL + s), 1);
      mbar_init(BAR(B_EMPTY + s), 2);  // one arrival per consumer warp
    }
    mbar_init(BAR(B_MERGE), 1);
    fence_mbar_init();
  }
  // this head's queries, widened to fp32; rows nq..NQ-1 are zero (their
  // results are computed and dropped)
  float* qs = reinterpret_cast<float*>(smem + C::OFF_Q);
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.Q) + (size_t)bh * nq * D;
  for (int e = threadIdx.x; e < NQ * D; e += C::THREADS)
    qs[e] = e < nq * D ? __bfloat162float(qg[e]) : 0.f;
  __syncthreads();

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tmK);
      tma_prefetch_desc(&a.tmV);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % C::STAGES;
        if (!mbar_wait(BAR(B_EMPTY + s), ((t / C::STAGES) & 1) ^ 1, a.status, a.wait_limit_ns)) break;
        mbar_arrive_expect_tx(BAR(B_FULL + s), 2 * C::TILE);
        const int y = k_begin + t * C::BK;
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_3d(sbase + C::OFF_K + s * C::TILE + c * C::CHUNK, &a.tmK, BAR(B_FULL + s), c * 64, y, bh);
          tma_load_3d(sbase + C::OFF_V + s * C::TILE + c * C::CHUNK, &a.tmV, BAR(B_FULL + s), c * 64, y, bh);
        }
        issued = t + 1;
      }
      // do not leave the CTA with copies in flight (the consumers may have
      // stopped early on a timeout)
      for (int t = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; t < issued; ++t)
        mbar_wait(BAR(B_FULL + t % C::STAGES), (t / C::STAGES) & 1, a.status, a.wait_limit_ns);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const float c2 = a.scale_log2;
  float m[NQ], l[NQ];
  uint64_t acc[NQ][C::DL / 2];  // packed fp32 pairs: columns lane*DL + 2e, +1
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    m[q] = -INFINITY;
    l[q] = 0.f;
#pragma unroll
    for (int e = 0; e < C::DL / 2; ++e) acc[q][e] = 0ull;
  }
  const int j = warp * 32 + lane;  // this lane's key row within a tile
  float* pw = reinterpret_cast<float*>(smem + C::OFF_P) + warp * 32 * NQ;
  bool ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % C::STAGES;
    if (!mbar_wait_warp(BAR(B_FULL + s), (t / C::STAGES) & 1, a.status, a.wait_limit_ns)) {
      ok = false;
      break;
    }
    const uint8_t* kt = smem + C::OFF_K + s * C::TILE;
    const uint8_t* vt = smem + C::OFF_V + s * C::TILE;
    const bool valid = k_begin + t * C::BK + j < k_end;

    // scores of key j against every query: key row read once, in 16-byte
    // units (unit u of row r is stored at unit u ^ (r & 7))
    uint64_t sc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) sc[q] = 0ull;
#pragma unroll
    for (int c = 0; c < C::CH; ++c) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 kv = *reinterpret_cast<const uint4*>(kt + c * C::CHUNK + j * 128 + ((u ^ (j & 7)) << 4));
        const uint64_t k0 = bf2_to_f2(kv.x), k1 = bf2_to_f2(kv.y), k2 = bf2_to_f2(kv.z),
                       k3 = bf2_to_f2(kv.w);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(qs + q * D + c * 64 + u * 8);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(qs + q * D + c * 64 + u * 8 + 4);
          sc[q] = ffma2(qa.x, k0, sc[q]);
          sc[q] = ffma2(qa.y, k1, sc[q]);
          sc[q] = ffma2(qb.x, k2, sc[q]);
          sc[q] = ffma2(qb.y, k3, sc[q]);
        }
      }
    }
    // online-softmax update per query over this warp's 32 keys
    float p[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const float2 s2 = f2_unpack(sc[q]);
      const float x = valid ? (s2.x + s2.y) * c2 : -INFINITY;
      float mt = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m[q], mt);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;  // no valid key seen yet
      const float alpha = ex2_approx(m[q] - m_use);           // 0 while m = -inf
      p[q] = ex2_approx(x - m_use);                           // 0 for masked keys
      float ps = p[q];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[q] = fmaf(l[q], alpha, ps);
      m[q] = m_new;
      const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
      for (int e = 0; e < C::DL / 2; ++e) acc[q][e] = fmul2(acc[q][e], al2);
    }
    // hand the probabilities to the whole warp: pw[key][q]
    if constexpr (NQ % 4 == 0) {
#pragma unroll
      for (int q = 0; q < NQ; q += 4)
        *reinterpret_cast<float4*>(pw + lane * NQ + q) = make_float4(p[q], p[q + 1], p[q + 2], p[q + 3]);
    } else {
#pragma unroll
      for (int q = 0; q < NQ; ++q) pw[lane * NQ + q] = p[q];
    }
    __syncwarp();
    // O += p_j v_j for the warp's 32 keys; this lane owns columns lane*DL ..
    const int col = lane * C::DL;
    const int v_off = (col >> 6) * C::CHUNK + (((col & 63) >> 3) << 4) + (col & 7) * 2;
#pragma unroll 4
    for (int jj = 0; jj < 32; ++jj) {
      const int r = warp * 32 + jj;
      const uint8_t* vp = vt + r * 128 + (v_off ^ ((r & 7) << 4));
      uint64_t v2[C::DL / 2];
      if constexpr (C::DL == 4) {
        const uint2 vv = *reinterpret_cast<const uint2*>(vp);
        v2[0] = bf2_to_f2(vv.x);
        v2[1] = bf2_to_f2(vv.y);
      } else {
        v2[0] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(vp));
      }
      float pj[NQ];
      if constexpr (NQ % 4 == 0) {
#pragma unroll
        for (int q = 0; q < NQ; q += 4) {
          const float4 f = *reinterpret_cast<const float4*>(pw + jj * NQ + q);
          pj[q] = f.x; pj[q + 1] = f.y; pj[q + 2] = f.z; pj[q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) pj[q] = pw[jj * NQ + q];
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint64_t pp = f2_pack(pj[q], pj[q]);
#pragma unroll
        for (int e = 0; e < C::DL / 2; ++e) acc[q][e] = ffma2(pp, v2[e], acc[q][e]);
      }
    }
    __syncwarp();  // pw is rewritten for the next tile
    if (lane == 0) mbar_arrive(BAR(B_EMPTY + s));
  }

  // ------------------------------------------------------------ merge the two warps, write the split
  float* xs = reinterpret_cast<float*>(smem + C::OFF_X);  // m[NQ], l[NQ], acc[NQ][D]
  if (warp == 1) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (lane == 0) {
        xs[q] = m[q];
        xs[NQ + q] = l[q];
      }
#pragma unroll
      for (int e = 0; e < C::DL / 2; ++e)
        *reinterpret_cast<uint64_t*>(xs + 2 * NQ + q * D + lane * C::DL + 2 * e) = acc[q][e];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_MERGE));  // also after a timeout, so that warp 0 never waits long
    return;
  }
  const bool merged = mbar_wait_warp(BAR(B_MERGE), 0, a.status, a.wait_limit_ns);
  if (!merged || !ok) return;
  const int rows = a.BH * nq;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (q >= nq) break;
    const float m1 = xs[q], l1 = xs[NQ + q];
    const float mm = fmaxf(m[q], m1);
    const float mu = mm == -INFINITY ? 0.f : mm;
    const float a0 = ex2_approx(m[q] - mu), a1 = ex2_approx(m1 - mu);
    const float lsum = fmaf(l[q], a0, l1 * a1);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const size_t prow = (size_t)split * rows + (size_t)bh * nq + q;
    float* op = a.Opart + prow * D + lane * C::DL;
#pragma unroll
    for (int e = 0; e < C::DL / 2; ++e) {
      const float2 x0 = f2_unpack(acc[q][e]);
      const float2 x1 = *reinterpret_cast<const float2*>(xs + 2 * NQ + q * D + lane * C::DL + 2 * e);
      *reinterpret_cast<float2*>(op + 2 * e) =
          make_float2((x0.x * a0 + x1.x * a1) * inv, (x0.y * a0 + x1.y * a1) * inv);
    }
    // a split with no key would give -inf; the planner never makes one
    if (lane == 0) a.LSEpart[prow] = lsum > 0.f ? mm + __log2f(lsum) : -INFINITY;
  }
}

// Merge the S split results of each (head, query) row: one warp per row.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a) {
  constexpr int DL = D / 32;
  const int row = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5);  // bh * Nq + q
  const int lane = threadIdx.x & 31;
  const int rows = a.BH * a.Nq;
  if (row >= rows) return;
  const int S = a.splits;
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, a.LSEpart[(size_t)s * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float mu = mx == -INFINITY ? 0.f : mx;
  float wsum = 0.f;
  for (int s = lane; s < S; s += 32) wsum += ex2_approx(a.LSEpart[(size_t)s * rows + row] - mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  float o_acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) o_acc[e] = 0.f;
#pragma unroll 4
  for (int s = 0; s < S; ++s) {
    const float w = ex2_approx(a.LSEpart[(size_t)s * rows + row] - mu);
    const float* op = a.Opart + ((size_t)s * rows + row) * D + lane * DL;
    if constexpr (DL == 4) {
      const float4 v = *reinterpret_cast<const float4*>(op);
      o_acc[0] = fmaf(w, v.x, o_acc[0]);
      o_acc[1] = fmaf(w, v.y, o_acc[1]);
      o_acc[2 % DL] = fmaf(w, v.z, o_acc[2 % DL]);
      o_acc[3 % DL] = fmaf(w, v.w, o_acc[3 % DL]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(op);
      o_acc[0] = fmaf(w, v.x, o_acc[0]);
      o_acc[1 % DL] = fmaf(w, v.y, o_acc[1 % DL]);
    }
  }
  const float inv = 1.f / wsum;
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.O) + (size_t)row * D + lane * DL;
  if constexpr (DL == 4) {
    uint2 w;
    w.x = pack_bf16x2(o_acc[0] * inv, o_acc[1] * inv);
    w.y = pack_bf16x2(o_acc[2 % DL] * inv, o_acc[3 % DL] * inv);
    *reinterpret_cast<uint2*>(o) = w;
  } else {
    *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(o_acc[0] * inv, o_acc[1 % DL] * inv);
  }
  if (lane == 0) a.LSE[row] = (mx + __log2f(wsum)) * 0.6931471805599453f;
}

template <int D, int NQ>
cudaError_t launch_dq(const DecodeArgs& a, cudaStream_t st) {
  using C = DecCfg<D, NQ>;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, NQ><<<dim3(a.splits, a.BH), C::THREADS, C::SMEM_ALLOC, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = (long long)a.BH * a.Nq;
  decode_combine_kernel<D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D, int NQ>
int resident_ctas_per_sm() {
  using C = DecCfg<D, NQ>;
  if (cudaFuncSetAttribute(decode_split_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_ALLOC) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<D, NQ>, C::THREADS,
                                                    C::SMEM_ALLOC) != cudaSuccess)
    return 0;
  return n;
}


// ---------------------------------------------------------------------------
// Tensor-core variant for 2..16 queries per head (grouped-query decode).
// With several queries the CUDA-core FMAs above no longer keep up with HBM;
// here both products run on tcgen05 with keys (scores) and head dimension
// (output) on the TMEM lanes, the queries padded to the MMA's N = 16:
//   S^T = K_j Q^T         M = 128 keys, N = 16, K = d       (A, B K-major)
//   O^T += V_j^T P_j^T    M = d,        N = 16, K = 128 keys (A MN-major)
// Warps: 0 TMA producer (K_j, V_j ring), 1 MMA issuer (converged, elected
// lane), 2-5 softmax: one thread per key of the tile (its TMEM lane). Per
// tile the softmax warps exchange their per-query maxima through shared
// memory behind an mbarrier (bounded wait), exponentiate against a
// reference max that moves only when a query's maximum grows by more than
// 2^8 (then O^T is rescaled in TMEM), keep per-thread partial sums l, and
// write bf16 P^T[q][key] into a swizzled tile that the second MMA reads as a
// K-major operand. At d = 64 the second MMA still has M = 128: its upper 64
// rows read a neighbouring shared-memory region and land in TMEM lanes that
// are never read.
template <int D>
struct DecTcCfg {
  static constexpr int BK = 128;   // keys per tile
  static constexpr int NQP = 16;   // queries padded to the MMA's N
  // d = 128: one CTA per SM, three 64 KB K+V stages keep two tiles loading
  // while one is processed; d = 64: three CTAs per SM (96 registers each)
  // with two 32 KB stages each
  static constexpr int STAGES = D == 128 ? 3 : 2;
  static constexpr int CH = D / 64;
  static constexpr int CHUNK = BK * 128;     // 128 rows x 128 bytes, swizzled
  static constexpr int TILE = CH * CHUNK;    // a K or a V tile
  static constexpr int QCHUNK = NQP * 128;   // 16 rows x 128 bytes
  // V ring first: at d = 64 the upper half of the M = 128 V^T operand reads
  // C::TILE past each V stage, which stays inside the V and K rings
  static constexpr int OFF_V = 0;
  static constexpr int OFF_K = STAGES * TILE;
  static constexpr int OFF_Q = 2 * STAGES * TILE;    // [16 q][d] bf16, CH chunks
  static constexpr int OFF_P = OFF_Q + CH * QCHUNK;  // 2 buffers x [16 q][128 keys] bf16
  static constexpr int OFF_RED = OFF_P + 2 * 2 * QCHUNK;  // fp32 max[2][4][16], sum[4][16]
  static constexpr int OFF_BAR = OFF_RED + (2 * 4 * 16 + 4 * 16) * 4;
  // barriers: full[S], empty[S], q_ready, s_full[2], s_empty[2], p_full[2],
  // p_empty[2], o_done, red, drain
  static constexpr int NBAR = 2 * STAGES + 1 + 8 + 3;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  // d = 64: no alignment slack, so that three CTAs fit on an SM (the kernel
  // checks that the dynamic shared memory starts on a 1024-byte boundary)
  static constexpr int SMEM_ALLOC = D == 64 ? SMEM : SMEM + 1024;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 64;  // S^T x 2 (16 columns each), O^T (16)
  static constexpr uint32_t COL_S = 0, COL_O = 32;
  static_assert(TILE % 1024 == 0 && OFF_P % 1024 == 0 && OFF_Q % 1024 == 0, "swizzle atoms");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Maximum (or sum) over the 32 lanes of each of 16 values: returns, on every
// lane, the result for query q = 8*b4 + 4*b3 + 2*b2 + b1 (bits of the lane
// index); lanes 2i and 2i+1 hold the same query.
template <bool MAX>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
  float a8[8], a4[4], a2[2];
  const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4, h1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = h4 ? v[i] : v[i + 8];
    const float keep = h4 ? v[i + 8] : v[i];
    a8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = h3 ? a8[i] : a8[i + 4];
    const float keep = h3 ? a8[i + 4] : a8[i];
    a4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = h2 ? a4[i] : a4[i + 2];
    const float keep = h2 ? a4[i + 2] : a4[i];
    a2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = h1 ? a2[0] : a2[1];
  const float keep = h1 ? a2[1] : a2[0];
  const float a1 = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}
__device__ __forceinline__ int reduce16_query(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

template <int D>
__global__ void __launch_bounds__(192, D == 64 ? 3 : 1) decode_tc_kernel(const __grid_constant__ DecodeArgs a) {
  using C = DecTcCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = ((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw);
  if (pad + C::SMEM > (uint32_t)C::SMEM_ALLOC) {
    // cannot place the swizzled tiles: report and leave before touching anything
    if (threadIdx.x == 0) report_status(a.status, kStatusTimeout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  constexpr int B_FULL = 0, B_EMPTY = C::STAGES, B_QREADY = 2 * C::STAGES, B_SFULL = B_QREADY + 1,
                B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2, B_PEMPTY = B_PFULL + 2,
                B_ODONE = B_PEMPTY + 2, B_RED = B_ODONE + 1, B_DRAIN = B_RED + 1;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  float* red_max = reinterpret_cast<float*>(smem + C::OFF_RED);  // [2][4][16]
  float* red_sum = red_max + 2 * 4 * 16;                         // [4][16]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int nq = a.Nq;
  const int k_begin = split * a.keys_per_split;
  const int k_end = min(a.Nk, k_begin + a.keys_per_split);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + C::BK - 1) / C::BK : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(B_FULL + s), 1);
      mbar_init(BAR(B_EMPTY + s), 1);
    }
    mbar_init(BAR(B_QREADY), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(B_SFULL + b), 1);
      mbar_init(BAR(B_SEMPTY + b), 4);
      mbar_init(BAR(B_PFULL + b), 4);
      mbar_init(BAR(B_PEMPTY + b), 1);
    }
    mbar_init(BAR(B_ODONE), 1);
    mbar_init(BAR(B_RED), 4);
    mbar_init(BAR(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32((const void*)tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&a.tmK);
      tma_prefetch_desc(&a.tmV);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        if (*abort_flag) break;
        const int s = t % C::STAGES;
        if (!mbar_wait(BAR(B_EMPTY + s), ((t / C::STAGES) & 1) ^ 1, a.status, a.wait_limit_ns)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(BAR(B_FULL + s), 2 * C::TILE);
        const int y = k_begin + t * C::BK;
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {
          tma_load_3d(sbase + C::OFF_K + s * C::TILE + c * C::CHUNK, &a.tmK, BAR(B_FULL + s), c * 64, y, bh);
          tma_load_3d(sbase + C::OFF_V + s * C::TILE + c * C::CHUNK, &a.tmV, BAR(B_FULL + s), c * 64, y, bh);
        }
        issued = t + 1;
      }
      for (int t = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; t < issued; ++t)
        mbar_wait(BAR(B_FULL + t % C::STAGES), (t / C::STAGES) & 1, a.status, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    constexpr uint32_t id_s = idesc_bf16_f32(128, C::NQP, false, false);
    constexpr uint32_t id_o = idesc_bf16_f32(128, C::NQP, true, false);
    const uint64_t dK0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
    const uint64_t dQ0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
    // V^T as an MN-major A operand: d in 64-element column blocks C::CHUNK
    // apart (d = 64: rows 64-127 of the product read the region C::TILE
    // ahead, the next V stage or the first K stage, and are never used)
    const uint64_t dV0 = sdesc_sw128(sbase + C::OFF_V, D == 128 ? C::CHUNK : C::TILE, 1024);
    const uint64_t dP0 = sdesc_sw128(sbase + C::OFF_P, 16, 1024);
    auto wait = [&](int b, uint32_t parity) {
      return mbar_wait_warp(BAR(b), parity, a.status, a.wait_limit_ns);
    };
    auto issue_pv = [&](int t) {
      const int s = t % C::STAGES, pb = t & 1;
      const uint64_t vb = dV0 + (uint64_t)((s * C::TILE) >> 4);
      const uint64_t pbd = dP0 + (uint64_t)((pb * 2 * C::QCHUNK) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::BK / 16; ++kk) {
        const uint64_t voff = (uint64_t)((kk * 2048) >> 4);  // 16 key rows of 128 bytes
        const uint64_t poff = (uint64_t)(((kk >> 2) * C::QCHUNK + (kk & 3) * 32) >> 4);
        mma_ss(tmem + C::COL_O, vb + voff, pbd + poff, id_o, (t > 0 || kk > 0) ? 1u : 0u, leader);
      }
    };
    bool ok = n_tiles > 0 && wait(B_QREADY, 0);
    for (int t = 0; ok && t < n_tiles; ++t) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int s = t % C::STAGES, sb = t & 1;
      if (!wait(B_FULL + s, (t / C::STAGES) & 1)) { ok = false; break; }
      if (t >= 2 && !wait(B_SEMPTY + sb, ((t >> 1) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      {
        const uint64_t kb = dK0 + (uint64_t)((s * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t koff = (uint64_t)(((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4);
          const uint64_t qoff = (uint64_t)(((kk >> 2) * C::QCHUNK + (kk & 3) * 32) >> 4);
          mma_ss(tmem + C::COL_S + 16 * sb, kb + koff, dQ0 + qoff, id_s, kk > 0 ? 1u : 0u, leader);
        }
        mma_commit(BAR(B_SFULL + sb), leader);
      }
      if (t >= 1) {
        const int tp = t - 1;
        if (!wait(B_PFULL + (tp & 1), (tp >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        issue_pv(tp);
        mma_commit(BAR(B_PEMPTY + (tp & 1)), leader);
        mma_commit(BAR(B_ODONE), leader);
        mma_commit(BAR(B_EMPTY + tp % C::STAGES), leader);
      }
    }
    if (ok) {
      const int tp = n_tiles - 1;
      if (wait(B_PFULL + (tp & 1), (tp >> 1) & 1)) {
        tc_fence_after();
        issue_pv(tp);
        mma_commit(BAR(B_PEMPTY + (tp & 1)), leader);
        mma_commit(BAR(B_ODONE), leader);
        mma_commit(BAR(B_EMPTY + tp % C::STAGES), leader);
      } else {
        ok = false;
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
    mma_commit(BAR(B_DRAIN), leader);
    wait(B_DRAIN, 0);
  } else {
    // ------------------------------------------------------------ softmax (warps 2-5)
    const int wq = warp & 3;            // TMEM lane quarter
    const int k = wq * 32 + lane;       // key of the tile / d index of O^T (TMEM lane)
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float c2 = a.scale_log2;
    // stage Q (rows >= nq zero) into the swizzled [16][d] operand tile
    {
      const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(a.Q) + (size_t)bh * nq * D;
      constexpr int UPR = D / 8;  // 16-byte units per row
      for (int e = k; e < C::NQP * UPR; e += 128) {
        const int r = e / UPR, uu = e - r * UPR, c = uu >> 3, u = uu & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < nq) v = *reinterpret_cast<const uint4*>(qg + (size_t)r * D + uu * 8);
        *reinterpret_cast<uint4*>(smem + C::OFF_Q + c * C::QCHUNK + r * 128 + ((u ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_QREADY));
    }
    float m[16], lp[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      m[q] = -INFINITY;
      lp[q] = 0.f;
    }
    bool ok = n_tiles > 0;
    for (int t = 0; ok && t < n_tiles; ++t) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int sb = t & 1;
      if (!mbar_wait_warp(BAR(B_SFULL + sb), (t >> 1) & 1, a.status, a.wait_limit_ns)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[16];
      tmem_ld16(lane_addr + C::COL_S + 16 * sb, sr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_SEMPTY + sb));  // S^T(t) read: the buffer may be reused
      const bool valid = k_begin + t * C::BK + k < k_end;
      float x[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) x[q] = valid ? __uint_as_float(sr[q]) * c2 : -INFINITY;
      // tile maximum of every query over the 128 keys: within the warp, then
      // across the four warps through shared memory
      {
        const float wm = warp_reduce16<true>(x, lane);
        float* slot = red_max + (t & 1) * 64 + wq * 16;
        if ((lane & 1) == 0) slot[reduce16_query(lane)] = wm;
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_RED));
      }
      if (!mbar_wait_warp(BAR(B_RED), t & 1, a.status, a.wait_limit_ns)) { ok = false; break; }
      float mt[16];
      {
        const float4* r4 = reinterpret_cast<const float4*>(red_max + (t & 1) * 64);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float4 w0 = r4[g], w1 = r4[4 + g], w2 = r4[8 + g], w3 = r4[12 + g];
          mt[4 * g + 0] = fmaxf(fmaxf(w0.x, w1.x), fmaxf(w2.x, w3.x));
          mt[4 * g + 1] = fmaxf(fmaxf(w0.y, w1.y), fmaxf(w2.y, w3.y));
          mt[4 * g + 2] = fmaxf(fmaxf(w0.z, w1.z), fmaxf(w2.z, w3.z));
          mt[4 * g + 3] = fmaxf(fmaxf(w0.w, w1.w), fmaxf(w2.w, w3.w));
        }
      }
      // the reference max moves only when a query's tile max exceeds it by
      // more than 2^8 (always on the first tile); the decision is the same on
      // every thread
      bool need = false;
#pragma unroll
      for (int q = 0; q < 16; ++q) need |= mt[q] > m[q] + kDecodeRescaleLog2;
      if (need) {
        float alpha[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const bool up = mt[q] > m[q] + kDecodeRescaleLog2;
          const float mn = up ? mt[q] : m[q];
          alpha[q] = up ? ex2_approx(m[q] - mn) : 1.f;  // 0 on the first tile
          m[q] = mn;
          lp[q] *= alpha[q];
        }
        if (t > 0) {
          // O^T (d on the lanes, queries on the columns) after P V of tile t-1
          if (!mbar_wait_warp(BAR(B_ODONE), (t - 1) & 1, a.status, a.wait_limit_ns)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(lane_addr + C::COL_O, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
          tmem_st16(lane_addr + C::COL_O, o);
          tmem_st_wait();
        }
      }
      // P^T of this key for the 16 queries -> row q, column k of the P tile
      if (t >= 2 && !mbar_wait_warp(BAR(B_PEMPTY + sb), ((t >> 1) & 1) ^ 1, a.status, a.wait_limit_ns)) {
        ok = false;
        break;
      }
      uint8_t* pt = smem + C::OFF_P + sb * 2 * C::QCHUNK + (k >> 6) * C::QCHUNK + (k & 7) * 2;
      const int ku = (k & 63) >> 3;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float p = ex2_approx(x[q] - m[q]);  // 0 for masked keys
        lp[q] += p;
        *reinterpret_cast<__nv_bfloat16*>(pt + q * 128 + ((ku ^ (q & 7)) << 4)) = __float2bfloat16_rn(p);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL + sb));
    }
    if (ok) {
      // l of every query: the per-thread partial sums over all 128 keys
      const float ws = warp_reduce16<false>(lp, lane);
      if ((lane & 1) == 0) red_sum[wq * 16 + reduce16_query(lane)] = ws;
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_RED));
      const bool w1 = mbar_wait_warp(BAR(B_RED), n_tiles & 1, a.status, a.wait_limit_ns);
      const bool w2 = w1 && mbar_wait_warp(BAR(B_ODONE), (n_tiles - 1) & 1, a.status, a.wait_limit_ns);
      ok = w2;
    }
    if (ok) {
      tc_fence_after();
      uint32_t o[16];
      tmem_ld16(lane_addr + C::COL_O, o);
      tmem_ld_wait();
      const int rows = a.BH * nq;
      if (k < D) {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (q < nq) {
            const float l = red_sum[q] + red_sum[16 + q] + red_sum[32 + q] + red_sum[48 + q];
            const size_t prow = (size_t)split * rows + (size_t)bh * nq + q;
            a.Opart[prow * D + k] = l > 0.f ? __uint_as_float(o[q]) / l : 0.f;
            if (k == q) a.LSEpart[prow] = l > 0.f ? m[q] + __log2f(l) : -INFINITY;
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_tc(const DecodeArgs& a, cudaStream_t st) {
  using C = DecTcCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<D><<<dim3(a.splits, a.BH), C::THREADS, C::SMEM_ALLOC, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = (long long)a.BH * a.Nq;
  decode_combine_kernel<D><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D>
int resident_tc_ctas_per_sm() {
  using C = DecTcCfg<D>;
  if (cudaFuncSetAttribute(decode_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_ALLOC) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tc_kernel<D>, C::THREADS, C::SMEM_ALLOC) !=
      cudaSuccess)
    return 0;
  return n;
}

// One query per head runs on the CUDA-core kernel (bandwidth-bound at HBM
// speed); from two queries on, the tensor-core kernel.
bool use_tc(int nq) { return nq >= 2; }
// Keys per tile of the kernel a problem runs on (split sizes are multiples of it).
int decode_tile(int nq) { return use_tc(nq) ? 128 : 64; }

constexpr int kMaxDevices = 64;
std::mutex g_plan_mu;
int g_slots[kMaxDevices][2][2] = {};  // [device][d == 128][tensor-core path] -> resident CTAs

int gpu_slots(int d, int nq) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  int& slot = g_slots[dev][d == 128][use_tc(nq)];
  if (slot == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    int per_sm = 0;
    if (use_tc(nq)) per_sm = d == 128 ? resident_tc_ctas_per_sm<128>() : resident_tc_ctas_per_sm<64>();
    else per_sm = d == 128 ? resident_ctas_per_sm<128, 1>() : resident_ctas_per_sm<64, 1>();
    slot = sms * per_sm;
  }
  return slot;
}

}  // namespace

DecodePlan plan_decode_for_slots(int BH, int Nk, int slots, int tile) {
  DecodePlan p{0, 0};
  if (slots <= 0 || BH < 1 || Nk < 1 || tile < 1) return p;
  // Pick S in [1, kDecodeMaxSplits] minimising waves(S) * (keys per split +
  // a fixed per-CTA cost of ~128 keys for filling the pipeline), so that the
  // last wave is as full as possible; ties go to the smaller S. Every split
  // gets at least one key.
  const long long tiles = ((long long)Nk + tile - 1) / tile;
  const int s_max = (int)(tiles < kDecodeMaxSplits ? tiles : kDecodeMaxSplits);
  long long best = -1;
  for (int s = 1; s <= s_max; ++s) {
    const long long kps = ((Nk + (long long)s - 1) / s + tile - 1) / tile * tile;
    if ((Nk + kps - 1) / kps != s) continue;  // would leave an empty split
    const long long waves = ((long long)BH * s + slots - 1) / slots;
    const long long cost = waves * (kps + 128);
    if (best < 0 || cost < best) {
      best = cost;
      p.splits = s;
      p.keys_per_split = (int)kps;
    }
  }
  return p;
}

DecodePlan plan_decode(int BH, int Nq, int Nk, int d) {
  return plan_decode_for_slots(BH, Nk, gpu_slots(d, Nq), decode_tile(Nq));
}

int decode_tile_keys(int Nq) { return decode_tile(Nq); }

cudaError_t launch_decode_bf16(const DecodeArgs& a, int d, cudaStream_t st) {
  if (a.keys_per_split % decode_tile(a.Nq) != 0) return cudaErrorInvalidValue;
  if (use_tc(a.Nq)) {
    if (d == 128) return launch_tc<128>(a, st);
    if (d == 64) return launch_tc<64>(a, st);
    return cudaErrorInvalidValue;
  }
  if (a.Nq != 1) return cudaErrorInvalidValue;
  if (d == 128) return launch_dq<128, 1>(a, st);
  if (d == 64) return launch_dq<64, 1>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
