// decode_splitkv.cu -- attention of a few new queries against a long key/value
// cache, split along the keys.
//
// What it computes: for each (batch, head) and each of Nq <= 8 queries,
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
// per key, against 4 d Nq FLOPs. So the scores and P V run on CUDA cores in
// packed f32x2 FMAs, and TMA keeps 64-key K/V tiles streaming through a
// shared-memory ring (128-byte swizzled rows: one lane per key reads its own
// row without bank conflicts).
//
// CTA: 3 warps. Warp 2 (one lane) is the TMA producer. Warps 0 and 1 own keys
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

int nq_bucket(int nq) { return nq <= 1 ? 1 : nq <= 2 ? 2 : nq <= 4 ? 4 : 8; }

template <int D>
int resident_ctas_d(int nqb) {
  switch (nqb) {
    case 1: return resident_ctas_per_sm<D, 1>();
    case 2: return resident_ctas_per_sm<D, 2>();
    case 4: return resident_ctas_per_sm<D, 4>();
    default: return resident_ctas_per_sm<D, 8>();
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_plan_mu;
int g_slots[kMaxDevices][2][4] = {};  // [device][d == 128][nq bucket] -> resident CTAs on the GPU

int gpu_slots(int d, int nq) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int nqb = nq_bucket(nq);
  const int bi = nqb == 1 ? 0 : nqb == 2 ? 1 : nqb == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  int& slot = g_slots[dev][d == 128][bi];
  if (slot == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    const int per_sm = d == 128 ? resident_ctas_d<128>(nqb) : resident_ctas_d<64>(nqb);
    slot = sms * per_sm;
  }
  return slot;
}

}  // namespace

DecodePlan plan_decode_for_slots(int BH, int Nk, int slots) {
  DecodePlan p{0, 0};
  if (slots <= 0 || BH < 1 || Nk < 1) return p;
  // Pick S in [1, kDecodeMaxSplits] minimising waves(S) * (keys per split +
  // a fixed per-CTA cost of ~128 keys for filling the pipeline), so that the
  // last wave is as full as possible; ties go to the smaller S. Every split
  // gets at least one key.
  const long long tiles = ((long long)Nk + 63) / 64;
  const int s_max = (int)(tiles < kDecodeMaxSplits ? tiles : kDecodeMaxSplits);
  long long best = -1;
  for (int s = 1; s <= s_max; ++s) {
    const long long kps = ((Nk + (long long)s - 1) / s + 63) / 64 * 64;
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
  return plan_decode_for_slots(BH, Nk, gpu_slots(d, Nq));
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, int d, cudaStream_t st) {
  const int nqb = nq_bucket(a.Nq);
  if (d == 128) {
    switch (nqb) {
      case 1: return launch_dq<128, 1>(a, st);
      case 2: return launch_dq<128, 2>(a, st);
      case 4: return launch_dq<128, 4>(a, st);
      default: return launch_dq<128, 8>(a, st);
    }
  }
  if (d == 64) {
    switch (nqb) {
      case 1: return launch_dq<64, 1>(a, st);
      case 2: return launch_dq<64, 2>(a, st);
      case 4: return launch_dq<64, 4>(a, st);
      default: return launch_dq<64, 8>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
