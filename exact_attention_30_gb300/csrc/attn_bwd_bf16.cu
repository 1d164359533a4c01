// attn_bwd_bf16.cu -- exact-attention backward with recomputation on sm_103a.
//
// What it computes ("Lesson 1: FlashAttention core idea" §5): with the
// forward pass's per-row log-sum-exp as the only saved statistic,
//   P  = exp(scale * Q K^T - LSE)          (rebuilt tile by tile)
//   dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D) * scale,  D_r = rowsum(dO o O)_r
//   dQ = dS K,    dK = dS^T Q.
// D uses the identity rowsum(dP o P) = rowsum(dO o O) (O = P V), so the row
// sum over the full row is available before any tile is visited.
//
// Three kernels on the caller's stream:
//  1. bwd_pre:   D and LSE*log2(e) per row into the workspace (rows padded to
//                a multiple of 128: D = 0, LSE*log2(e) = +inf past N, which
//                makes P = 0 there), and zero the fp32 dQ accumulator.
//  2. bwd_main:  one CTA per (batch*head, 128-key tile j); K_j, V_j stay in
//                shared memory while the query tiles i stream through a TMA
//                ring. All products run on tcgen05 with fp32 accumulators in
//                TMEM, keys on the TMEM lanes:
//                  S^T = K_j Q_i^T,  dP^T = V_j dO_i^T   (recompute)
//                  dV += P^T dO_i,   dK += dS^T Q_i      (stay in TMEM)
//                  dQ_i (+)= dS K_j  -> fp32 atomics into the accumulator
//                The softmax warpgroup (one thread per key) turns S^T, dP^T
//                into bf16 P^T and dS^T tiles in swizzled shared memory,
//                which feed both the dV/dK and the dQ products. S^T/dP^T of
//                the next query tile are computed while it works.
//  3. dq_convert: fp32 accumulator -> bf16 dQ.
// d = 128 uses 64-query tiles and computes dQ^T = K_j^T dS^T (M = d);
// d = 64 uses 128-query tiles and computes dQ = dS K_j (M = queries); both
// keep every TMEM operand at M = 128 within 512 columns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// ----------------------------------------------------------------------------
// 1. preprocess
// ----------------------------------------------------------------------------
// One group of D/8 lanes per row; each lane reads 8 bf16 of O and dO.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a, int BH) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, l = lane % LPR;
  const long long prow = (long long)warp_global * RPW + sub;  // padded row index
  const long long total = (long long)BH * a.Npad;
  float acc = 0.f;
  bool live = false;
  long long bh = 0, n = 0;
  if (prow < total) {
    bh = prow / a.Npad;
    n = prow - bh * a.Npad;
    live = n < a.N;
    if (live) {
      const size_t off = ((size_t)bh * a.N + (size_t)n) * D + (size_t)l * 8;
      const uint4 uo = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.O) + off);
      const uint4 ud = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.dO) + off);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&uo);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&ud);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fo = __bfloat1622float2(o2[i]);
        const float2 fd = __bfloat1622float2(d2[i]);
        acc = fmaf(fo.x, fd.x, acc);
        acc = fmaf(fo.y, fd.y, acc);
      }
    }
    float4* z = reinterpret_cast<float4*>(a.dQacc + (size_t)prow * D + (size_t)l * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (prow < total && l == 0) {
    a.Drow[prow] = live ? acc : 0.f;
    a.lse2[prow] = live ? a.LSE[(size_t)bh * a.N + (size_t)n] * 1.4426950408889634f : INFINITY;
  }
}

// ----------------------------------------------------------------------------
// 3. dQ convert
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BwdArgs a, int BH) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 elements
  const long long groups = (long long)BH * a.N * (D / 8);
  if (idx >= groups) return;
  const long long row = idx / (D / 8);
  const int g = (int)(idx - row * (D / 8));
  const long long bh = row / a.N, n = row - bh * a.N;
  const float4* src = reinterpret_cast<const float4*>(a.dQacc + ((size_t)bh * a.Npad + n) * D + g * 8);
  const float4 x = src[0], y = src[1];
  uint4 u;
  u.x = pack_bf16x2(x.x, x.y);
  u.y = pack_bf16x2(x.z, x.w);
  u.z = pack_bf16x2(y.x, y.y);
  u.w = pack_bf16x2(y.z, y.w);
  *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.dQ) + (size_t)row * D + g * 8) = u;
}

// ----------------------------------------------------------------------------
// 2. main kernel
// ----------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  static constexpr bool DQ_T = (D == 128);   // compute dQ^T (M = d) instead of dQ (M = queries)
  static constexpr int BK = 128;             // keys per CTA (TMEM lanes)
  static constexpr int BQ = DQ_T ? 64 : 128; // queries per streamed tile
  static constexpr int CH = D / 64;          // 128-byte chunks per K/V/Q/dO row
  static constexpr int QCH = BQ / 64;        // 128-byte chunks per P^T/dS^T row
  // Q/dO ring depth: a slot is busy from the S^T prefetch of its tile until
  // the dK/dV products one iteration later, so loads need >= 3 slots to run
  // ahead of use; the P^T/dS^T tiles are single-buffered to make room.
  static constexpr int STAGES = 3;
  static constexpr int NPS = 1;  // P^T/dS^T shared-memory buffers
  static constexpr int KV_CHUNK = BK * 128;          // 16 KB
  static constexpr int Q_CHUNK = BQ * 128;           // 8 or 16 KB
  static constexpr int KV_TILE = CH * KV_CHUNK;
  static constexpr int Q_TILE = CH * Q_CHUNK;
  static constexpr int PS_CHUNK = BK * 128;          // 16 KB: [128 keys][64 queries] bf16
  static constexpr int PS_TILE = QCH * PS_CHUNK;
  static constexpr int STAT_BYTES = 2 * BQ * 4;      // lse2 + D for one query tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_P = OFF_DO + STAGES * Q_TILE;      // NPS buffers
  static constexpr int OFF_DS = OFF_P + NPS * PS_TILE;        // NPS buffers
  static constexpr int OFF_STAT = OFF_DS + NPS * PS_TILE;     // STAGES x STAT_BYTES
  static constexpr int OFF_BAR = OFF_STAT + STAGES * STAT_BYTES;
  // barriers: kv_full, q_full[S], qdo_empty[S], s_full, s_consumed, p_ready[2],
  //           pds_empty[2], dq_full[2], dq_empty[2], acc_done, drain
  static constexpr int NBAR = 1 + 2 * STAGES + 2 + 2 + 2 + 2 + 2 + 2;
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;
  static constexpr int THREADS = 384;
  // TMEM columns
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BQ;
  static constexpr int DQC = DQ_T ? BQ : D;  // columns of one dQ buffer
  static constexpr uint32_t COL_DQ = 2 * BQ;
  static constexpr uint32_t COL_DV = 2 * BQ + 2 * DQC;
  static constexpr uint32_t COL_DK = COL_DV + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_DK + D <= 512, "TMEM budget");
  static_assert(BQ == bwd_query_tile(D), "host tensor-map box height");
};

template <int D>
__global__ void __launch_bounds__(384, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const int B_KV = 0, B_QFULL = 1, B_QEMPTY = 1 + C::STAGES, B_SFULL = 1 + 2 * C::STAGES,
            B_SCONS = B_SFULL + 1, B_PREADY = B_SCONS + 1, B_PSEMPTY = B_PREADY + 2,
            B_DQFULL = B_PSEMPTY + 2, B_DQEMPTY = B_DQFULL + 2, B_ACC = B_DQEMPTY + 2,
            B_DRAIN = B_ACC + 1;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  const float* stat_smem = reinterpret_cast<const float*>(smem + C::OFF_STAT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int k0 = blockIdx.x * C::BK;
  const int N = a.N;
  const int n_q = a.Npad / C::BQ;

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_KV), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(B_QFULL + s), 1);
      mbar_init(BAR(B_QEMPTY + s), 1);
    }
    mbar_init(BAR(B_SFULL), 1);
    mbar_init(BAR(B_SCONS), 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(B_PREADY + b), 128);
      mbar_init(BAR(B_PSEMPTY + b), 1);
      mbar_init(BAR(B_DQFULL + b), 1);
      mbar_init(BAR(B_DQEMPTY + b), 128);
    }
    mbar_init(BAR(B_ACC), 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&a.tmQ);
      tma_prefetch_desc(&a.tmK);
      tma_prefetch_desc(&a.tmV);
      tma_prefetch_desc(&a.tmdO);
      mbar_arrive_expect_tx(BAR(B_KV), 2 * C::KV_TILE);
      for (int c = 0; c < C::CH; ++c) {
        tma_load_3d(sbase + C::OFF_K + c * C::KV_CHUNK, &a.tmK, BAR(B_KV), c * 64, k0, bh);
        tma_load_3d(sbase + C::OFF_V + c * C::KV_CHUNK, &a.tmV, BAR(B_KV), c * 64, k0, bh);
      }
      int last[C::STAGES];
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last[s] = -1;
      for (int i = 0; i < n_q; ++i) {
        if (*abort_flag) break;
        const int s = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        if (!mbar_wait(BAR(B_QEMPTY + s), ph ^ 1, a.status, a.wait_limit_ns)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(BAR(B_QFULL + s), 2 * C::Q_TILE + C::STAT_BYTES);
        for (int c = 0; c < C::CH; ++c) {
          tma_load_3d(sbase + C::OFF_Q + s * C::Q_TILE + c * C::Q_CHUNK, &a.tmQ, BAR(B_QFULL + s),
                      c * 64, i * C::BQ, bh);
          tma_load_3d(sbase + C::OFF_DO + s * C::Q_TILE + c * C::Q_CHUNK, &a.tmdO,
                      BAR(B_QFULL + s), c * 64, i * C::BQ, bh);
        }
        const size_t row0 = (size_t)bh * a.Npad + (size_t)i * C::BQ;
        bulk_load(sbase + C::OFF_STAT + s * C::STAT_BYTES, a.lse2 + row0, C::BQ * 4, BAR(B_QFULL + s));
        bulk_load(sbase + C::OFF_STAT + s * C::STAT_BYTES + C::BQ * 4, a.Drow + row0, C::BQ * 4,
                  BAR(B_QFULL + s));
        last[s] = i;
      }
      mbar_wait(BAR(B_KV), 0, a.status, a.wait_limit_ns);
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s)
        if (last[s] >= 0) mbar_wait(BAR(B_QFULL + s), (last[s] / C::STAGES) & 1, a.status, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, C::BQ, false, false);   // S^T, dP^T
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, false, true);      // dV, dK
      constexpr uint32_t id_dq = C::DQ_T ? idesc_bf16_f32(128, C::BQ, true, true)   // dQ^T = K^T dS^T
                                         : idesc_bf16_f32(128, D, true, true);      // dQ = dS K
      // S^T = K Q_i^T and dP^T = V dO_i^T  (A K-major [keys x d], B K-major [queries x d])
      auto issue_s = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          const uint32_t offb = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::COL_S, sdesc_sw128(sbase + C::OFF_K + offa, 16, 1024),
                 sdesc_sw128(sbase + C::OFF_Q + s * C::Q_TILE + offb, 16, 1024), id_s, kk > 0);
          mma_ss(tmem + C::COL_DP, sdesc_sw128(sbase + C::OFF_V + offa, 16, 1024),
                 sdesc_sw128(sbase + C::OFF_DO + s * C::Q_TILE + offb, 16, 1024), id_s, kk > 0);
        }
      };
      // dV += P^T dO_i, dK += dS^T Q_i  (A K-major [keys x queries], B MN-major [queries x d])
      auto issue_acc = [&](int s, int b, bool acc) {
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * C::PS_CHUNK + (kk & 3) * 32;
          const uint32_t offb = kk * 2048;
          mma_ss(tmem + C::COL_DV, sdesc_sw128(sbase + C::OFF_P + b * C::PS_TILE + offa, 16, 1024),
                 sdesc_sw128(sbase + C::OFF_DO + s * C::Q_TILE + offb, C::Q_CHUNK, 1024), id_acc,
                 (acc || kk > 0) ? 1u : 0u);
          mma_ss(tmem + C::COL_DK, sdesc_sw128(sbase + C::OFF_DS + b * C::PS_TILE + offa, 16, 1024),
                 sdesc_sw128(sbase + C::OFF_Q + s * C::Q_TILE + offb, C::Q_CHUNK, 1024), id_acc,
                 (acc || kk > 0) ? 1u : 0u);
        }
      };
      // dQ^T = K^T dS^T (d = 128) or dQ = dS K (d = 64); K-dimension = keys.
      auto issue_dq = [&](int b, int bp) {
        const uint32_t dcol = tmem + C::COL_DQ + b * C::DQC;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          const uint32_t off = kk * 2048;
          const uint64_t kd = sdesc_sw128(sbase + C::OFF_K + off, C::KV_CHUNK, 1024);
          const uint64_t sd = sdesc_sw128(sbase + C::OFF_DS + bp * C::PS_TILE + off, C::PS_CHUNK, 1024);
          if (C::DQ_T) mma_ss(dcol, kd, sd, id_dq, kk > 0);
          else mma_ss(dcol, sd, kd, id_dq, kk > 0);
        }
      };
      bool ok = mbar_wait(BAR(B_KV), 0, a.status, a.wait_limit_ns) &&
                mbar_wait(BAR(B_QFULL + 0), 0, a.status, a.wait_limit_ns);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(BAR(B_SFULL));
      }
      for (int i = 0; ok && i < n_q; ++i) {
        if (*abort_flag) { ok = false; break; }
        const int s = i % C::STAGES;
        const int b = i & 1;                  // dQ TMEM buffer
        const int bp = i % C::NPS;            // P^T/dS^T buffer
        const uint32_t php = (i / C::NPS) & 1;
        if (i + 1 < n_q) {
          const int s1 = (i + 1) % C::STAGES;
          const uint32_t ph1 = ((i + 1) / C::STAGES) & 1;
          if (!mbar_wait(BAR(B_QFULL + s1), ph1, a.status, a.wait_limit_ns) ||
              !mbar_wait(BAR(B_SCONS), i & 1, a.status, a.wait_limit_ns)) { ok = false; break; }
          tc_fence_after();
          issue_s(s1);
          mma_commit(BAR(B_SFULL));
        }
        if (!mbar_wait(BAR(B_PREADY + bp), php, a.status, a.wait_limit_ns)) { ok = false; break; }
        tc_fence_after();
        issue_acc(s, bp, i > 0);
        mma_commit(BAR(B_QEMPTY + s));  // Q_i, dO_i, stats: last use was dK/dV
        if (!mbar_wait(BAR(B_DQEMPTY + b), ((i >> 1) & 1) ^ 1, a.status, a.wait_limit_ns)) { ok = false; break; }
        tc_fence_after();
        issue_dq(b, bp);
        mma_commit(BAR(B_DQFULL + b));
        mma_commit(BAR(B_PSEMPTY + bp));
      }
      if (ok) mma_commit(BAR(B_ACC));
      else *abort_flag = 1;
      mma_commit(BAR(B_DRAIN));
      mbar_wait(BAR(B_DRAIN), 0, a.status, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax: P^T, dS^T
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row within the tile == TMEM lane
    const bool key_live = k0 + r < N;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const float c2 = a.scale_log2, scale = a.scale;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int s = i % C::STAGES;
      const int b = i % C::NPS;
      bool w = mbar_wait(BAR(B_SFULL), i & 1, a.status, a.wait_limit_ns) &&
               mbar_wait(BAR(B_QFULL + s), (i / C::STAGES) & 1, a.status, a.wait_limit_ns) &&
               mbar_wait(BAR(B_PSEMPTY + b), ((i / C::NPS) & 1) ^ 1, a.status, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      const float* lse2 = stat_smem + s * (C::STAT_BYTES / 4);
      const float* drow = lse2 + C::BQ;
      uint8_t* pbuf = smem + C::OFF_P + b * C::PS_TILE;
      uint8_t* dsbuf = smem + C::OFF_DS + b * C::PS_TILE;
#pragma unroll
      for (int h = 0; h < C::QCH; ++h) {
        uint32_t sr[64], dr[64];
        {
          uint32_t t0[32], t1[32];
          tmem_ld32(lane_addr + C::COL_S + 64 * h, t0);
          tmem_ld32(lane_addr + C::COL_S + 64 * h + 32, t1);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) { sr[k] = t0[k]; sr[32 + k] = t1[k]; }
          tmem_ld32(lane_addr + C::COL_DP + 64 * h, t0);
          tmem_ld32(lane_addr + C::COL_DP + 64 * h + 32, t1);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) { dr[k] = t0[k]; dr[32 + k] = t1[k]; }
        }
        if (h == C::QCH - 1) {
          tc_fence_before();
          mbar_arrive(BAR(B_SCONS));
        }
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4) {
          const int q = 64 * h + 4 * k4;
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + q);
          const float4 d4 = *reinterpret_cast<const float4*>(drow + q);
          const float lq[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dq[4] = {d4.x, d4.y, d4.z, d4.w};
          float p[4], ds[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            p[u] = ex2_approx(fmaf(__uint_as_float(sr[4 * k4 + u]), c2, -lq[u]));
            ds[u] = p[u] * (__uint_as_float(dr[4 * k4 + u]) - dq[u]) * scale;
            if (!key_live) p[u] = ds[u] = 0.f;
          }
          pk[2 * k4] = pack_bf16x2(p[0], p[1]);
          pk[2 * k4 + 1] = pack_bf16x2(p[2], p[3]);
          dk[2 * k4] = pack_bf16x2(ds[0], ds[1]);
          dk[2 * k4 + 1] = pack_bf16x2(ds[2], ds[3]);
        }
        // row r of a 128-byte-swizzled [128 x 64] bf16 tile: 16-byte chunk c at c ^ (r & 7)
        uint8_t* prow = pbuf + h * C::PS_CHUNK + r * 128;
        uint8_t* drow_s = dsbuf + h * C::PS_CHUNK + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int pc = (c ^ (r & 7)) * 16;
          *reinterpret_cast<uint4*>(prow + pc) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          *reinterpret_cast<uint4*>(drow_s + pc) = make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(BAR(B_PREADY + b));
    }
    if (ok) {
      const bool w = mbar_wait(BAR(B_ACC), 0, a.status, a.wait_limit_ns);
      ok = __all_sync(0xffffffffu, w);
    }
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const size_t out_row = ((size_t)bh * N + (size_t)(k0 + r)) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::COL_DV : C::COL_DK;
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which == 0 ? a.dV : a.dK) + out_row;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t v[32];
          tmem_ld32(lane_addr + col + 32 * q, v);
          tmem_ld_wait();
          if (key_live) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * q);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              d4[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]), __uint_as_float(v[8 * u + 1])),
                                 pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                                 pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                                 pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ reduction
    const int wq = warp & 3;
    const int t = wq * 32 + lane;  // TMEM lane: d index (dQ^T) or query row (dQ)
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    for (int i = 0; i < n_q; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int b = i & 1;
      const bool w = mbar_wait(BAR(B_DQFULL + b), (i >> 1) & 1, a.status, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, w)) { *abort_flag = 1; break; }
      tc_fence_after();
      uint32_t v[64];
      {
        uint32_t t0[32], t1[32];
        tmem_ld32(lane_addr + C::COL_DQ + b * C::DQC, t0);
        tmem_ld32(lane_addr + C::COL_DQ + b * C::DQC + 32, t1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) { v[k] = t0[k]; v[32 + k] = t1[k]; }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_DQEMPTY + b));
      const size_t row0 = (size_t)bh * a.Npad + (size_t)i * C::BQ;
      if (C::DQ_T) {
        // lane t holds dQ[row0 + q][t] for q = 0..63: warp-coalesced 128-byte reductions
        float* base = a.dQacc + row0 * D + t;
#pragma unroll
        for (int q = 0; q < 64; ++q) atomicAdd(base + (size_t)q * D, __uint_as_float(v[q]));
      } else {
        // lane t holds the whole dQ row (64 values) of query row0 + t
        float4* base = reinterpret_cast<float4*>(a.dQacc + (row0 + t) * D);
#pragma unroll
        for (int q = 0; q < 16; ++q)
          atomicAdd(base + q, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                          __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, int BH, unsigned stages, cudaStream_t st) {
  using C = BwdCfg<D>;
  static_assert(C::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaSuccess;
  if (stages & kStagePre) {
    constexpr int RPW = 32 / (D / 8);
    const long long rows = (long long)BH * a.Npad;
    const long long warps = (rows + RPW - 1) / RPW;
    const long long blocks = (warps * 32 + 255) / 256;
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(a, BH);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kStageMain) {
    e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + C::BK - 1) / C::BK, BH);
    bwd_main_kernel<D><<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kStageConvert) {
    const long long groups = (long long)BH * a.N * (D / 8);
    dq_convert_kernel<D><<<(unsigned)((groups + 255) / 256), 256, 0, st>>>(a, BH);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdArgs& a, int BH, int d, unsigned stages, cudaStream_t st) {
  if (d == 128) return launch_bwd_d<128>(a, BH, stages, st);
  if (d == 64) return launch_bwd_d<64>(a, BH, stages, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
