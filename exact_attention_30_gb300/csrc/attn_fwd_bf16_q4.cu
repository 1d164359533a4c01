// attn_fwd_bf16_q4.cu -- the d = 64 forward with four query tiles per CTA.
//
// Same computation as fwd_bf16_kernel ("Lesson 1: FlashAttention core idea"
// §3-§4; "FlashAttention and Triton" §19.4-§19.6): per query row
//   O_r = sum_c exp(s_rc - m_r) V_c / l_r,  LSE_r = m_r + ln(l_r),  s = scale * q.k
// with S and P held only in tensor memory and registers, and the same online
// softmax rule (base 2, reference max raised only when a tile's max exceeds it
// by more than kRescaleLog2Q4, O rescaled in TMEM before the next P V
// product). Each 64-column row of S is read in one TMEM round trip and its max
// found first, so every exponential is computed once.
//
// Why a second d = 64 kernel. At d = 64 every CTA of the two-tile kernel
// spends most of its time in a serial chain (S -> softmax -> P V) that the
// other tile's products cannot cover, and short sequences leave 1-2 partly
// filled waves of CTAs. Here a CTA keeps four 128-row query tiles in flight
// against 64-key K/V tiles: TMEM holds, per query tile t, S_t (64 fp32
// columns, P_t written over it as bf16) and O_t (64 columns), 4 x 128 = 512
// columns. The tensor core then always has three other tiles' products queued
// while one tile's softmax runs, and a 1024-key head needs only two CTAs.
// The price: S = Q K^T has N = 64 (keys), which the tensor core runs at the
// time of an N = 128 product, like P V (N = d = 64) in both kernels.
//
// CTA = one (batch*head, 512-row query block). Warps (18):
//   warp 0       TMA producer: the four Q tiles (one barrier each), then
//                K_j / V_j (64 keys) through a ring of STAGES slots.
//   warp 1       TMEM allocation; the converged warp runs the MMA schedule,
//                one elected lane issues: per key tile j and query tile t,
//                P_t(j) V_j then S_t(j+1) = Q_t K_{j+1}^T (P over S: the next
//                S is ordered after the P V product that reads P).
//   warps 2-17   softmax, warpgroup g = query tile g, one thread per row.
// Fixed-length problems, causal or not (packed variable-length batches go to
// the two-tile kernel). Causal attention: query tile t of a 512-row block
// runs the 64-key tiles up to its diagonal (two tiles more than tile t - 1),
// the last two of them masked per row; the grid lists the blocks with the
// most key tiles first. Every wait is bounded; on expiry the kernel records a
// timeout, drains its copies and products, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kRescaleLog2Q4 = 8.0f;  // tolerated growth of the running max before O is rescaled

struct Q4Cfg {
  static constexpr int D = 64;
  static constexpr int BM = 128;  // query rows per tile (TMEM lanes)
  static constexpr int QT = 4;    // query tiles per CTA
  static constexpr int BN = 64;   // keys per K/V tile
  static constexpr int STAGES = 4;
  static constexpr int Q_BYTES = BM * 128;   // 128 rows x 64 bf16, 128-byte swizzle
  static constexpr int KV_BYTES = BN * 128;  // 64 rows x 64 bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // barriers: q_full[QT], k_full[S], v_full[S], k_empty[S], v_empty[S],
  //           s_full[QT], p_full[QT], o_done[QT], drain
  static constexpr int NBAR = QT + 4 * STAGES + 3 * QT + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1024-byte alignment
  static constexpr int SW0 = 2;                          // first softmax warp
  static constexpr int THREADS = 32 * (SW0 + 4 * QT);    // 576
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL(int t) { return 128u * t; }        // P_t over its first 32
  static constexpr uint32_t O_COL(int t) { return 128u * t + 64u; }
};
static_assert(Q4Cfg::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(Q4Cfg::O_COL(Q4Cfg::QT - 1) + Q4Cfg::D <= Q4Cfg::TMEM_COLS, "TMEM budget");

// One 32-column chunk of a score row: p = 2^(s*c2 - m) for column pairs
// (packed fp32 arithmetic), row sums in four packed accumulators, P as bf16
// pairs.
__device__ __forceinline__ void q4_chunk32(const uint32_t (&r)[32], uint32_t (&pk)[16], uint64_t c22,
                                           uint64_t nm2, uint64_t (&sm2)[4]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c22, nm2));
    const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
    sm2[i & 3] = fadd2(sm2[i & 3], f2_pack(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(Q4Cfg::THREADS, 1) fwd_bf16_q4_kernel(const __grid_constant__ FwdArgs a) {
  using C = Q4Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const int B_QFULL = 0, B_KFULL = C::QT, B_VFULL = C::QT + C::STAGES,
            B_KEMPTY = C::QT + 2 * C::STAGES, B_VEMPTY = C::QT + 3 * C::STAGES,
            B_SFULL = C::QT + 4 * C::STAGES, B_PFULL = B_SFULL + C::QT, B_ODONE = B_PFULL + C::QT,
            B_DRAIN = B_ODONE + C::QT;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool causal = CAUSAL;  // a separate instance: the unmasked path stays as lean as before
  int bh, qblk;
  if (causal) {
    // causal grids: (heads of a group, query blocks from the last = most key
    // tiles to the first, head groups): longest first within a group
    bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    qblk = (int)(gridDim.y - 1 - blockIdx.y);
  } else {
    const int qblocks = (a.seq.N + C::BM * C::QT - 1) / (C::BM * C::QT);
    bh = (int)blockIdx.x / qblocks;
    qblk = (int)blockIdx.x - bh * qblocks;
  }
  if (bh >= a.BH) return;
  const int N = a.seq.N;
  const int q0 = qblk * (C::BM * C::QT);
  const int n_kv = (N + C::BN - 1) / C::BN;
  const int plane = bh;
  // query tiles with at least one row inside the sequence
  const int n_tiles = min(C::QT, (N - q0 + C::BM - 1) / C::BM);
  // key tiles of query tile t: all of them, or (causal) those up to its
  // diagonal, which ends at key q0 + 128 (t + 1) - 1
  auto n_own = [&](int t) { return causal ? min(n_kv, (q0 + C::BM * (t + 1)) / C::BN) : n_kv; };
  const int n_max = n_own(n_tiles - 1);  // the last live tile sees the most keys

  if (threadIdx.x == 0) {
    for (int t = 0; t < C::QT; ++t) mbar_init(BAR(B_QFULL + t), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(B_KFULL + s), 1);
      mbar_init(BAR(B_VFULL + s), 1);
      mbar_init(BAR(B_KEMPTY + s), 1);
      mbar_init(BAR(B_VEMPTY + s), 1);
    }
    for (int t = 0; t < C::QT; ++t) {
      mbar_init(BAR(B_SFULL + t), 1);
      mbar_init(BAR(B_PFULL + t), 4);  // one arrival per softmax warp of the tile
      mbar_init(BAR(B_ODONE + t), 1);
    }
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
      auto load_q = [&](int t) {
        mbar_arrive_expect_tx(BAR(B_QFULL + t), C::Q_BYTES);
        tma_load_3d(sbase + C::OFF_Q + t * C::Q_BYTES, &a.tmQ, BAR(B_QFULL + t), 0, q0 + t * C::BM, plane);
      };
      // Q tile 0, then K_0, then the other Q tiles: S_0(0) needs only the first two
      load_q(0);
      int q_loaded = 1;
      int last_k[C::STAGES], last_v[C::STAGES];  // last tile loaded into each slot
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) last_k[s] = last_v[s] = -1;
      for (int j = 0; j < n_max; ++j) {
        if (*abort_flag) break;
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        if (!mbar_wait(BAR(B_KEMPTY + s), ph ^ 1, a.status, a.wait_limit_ns)) { *abort_flag = 1; break; }
        if (j != a.debug_skip_kv) {
          mbar_arrive_expect_tx(BAR(B_KFULL + s), C::KV_BYTES);
          tma_load_3d(sbase + C::OFF_K + s * C::KV_BYTES, &a.tmK, BAR(B_KFULL + s), 0, j * C::BN, plane);
          last_k[s] = j;
        }
        if (j == 0)
          for (; q_loaded < n_tiles; ++q_loaded) load_q(q_loaded);
        if (!mbar_wait(BAR(B_VEMPTY + s), ph ^ 1, a.status, a.wait_limit_ns)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(BAR(B_VFULL + s), C::KV_BYTES);
        tma_load_3d(sbase + C::OFF_V + s * C::KV_BYTES, &a.tmV, BAR(B_VFULL + s), 0, j * C::BN, plane);
        last_v[s] = j;
      }
      // drain: the last load issued into each slot must have landed before exit
      for (int t = 0; t < q_loaded; ++t) mbar_wait(BAR(B_QFULL + t), 0, a.status, a.wait_limit_ns);
#pragma unroll
      for (int s = 0; s < C::STAGES; ++s) {
        if (last_k[s] >= 0)
          mbar_wait(BAR(B_KFULL + s), (last_k[s] / C::STAGES) & 1, a.status, a.wait_limit_ns);
        if (last_v[s] >= 0)
          mbar_wait(BAR(B_VFULL + s), (last_v[s] / C::STAGES) & 1, a.status, a.wait_limit_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, C::BN, false, false);  // S = Q K^T
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, C::D, false, true);    // O += P V
    // Descriptors built once; K-steps add byte offsets >> 4 (every operand
    // lies below 256 KB, so the 14-bit address field cannot carry over).
    const uint64_t dQ0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
    const uint64_t dV0 = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
    auto issue_s = [&](int t, int s) {
      const uint64_t qa = dQ0 + (uint64_t)((t * C::Q_BYTES) >> 4);
      const uint64_t kb = dK0 + (uint64_t)((s * C::KV_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk)
        mma_ss(tmem + C::S_COL(t), qa + (uint64_t)(kk * 2), kb + (uint64_t)(kk * 2), idesc_s, kk > 0 ? 1u : 0u,
               leader);  // 16 elements = 32 bytes per K-step
    };
    auto issue_pv = [&](int t, int s, bool acc) {
      const uint64_t vb = dV0 + (uint64_t)((s * C::KV_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ts(tmem + C::O_COL(t), tmem + C::S_COL(t) + kk * 8, vb + (uint64_t)((kk * 2048) >> 4), idesc_o,
               (acc || kk > 0) ? 1u : 0u, leader);  // 16 keys = 16 rows of 128 bytes
    };
    auto wait = [&](int b, uint32_t parity) {
      return mbar_wait_warp(BAR(b), parity, a.status, a.wait_limit_ns);
    };
    bool ok = wait(B_KFULL + 0, 0);
    for (int t = 0; ok && t < n_tiles; ++t) {
      if (!wait(B_QFULL + t, 0)) { ok = false; break; }
      tc_fence_after();
      issue_s(t, 0);
      mma_commit(BAR(B_SFULL + t), leader);
    }
    if (ok) mma_commit(BAR(B_KEMPTY + 0), leader);
    for (int j = 0; ok && j < n_max; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const int s = j % C::STAGES, s1 = (j + 1) % C::STAGES;
      const uint32_t ph = (j / C::STAGES) & 1, ph1 = ((j + 1) / C::STAGES) & 1;
      const bool more = j + 1 < n_max;
      if (!wait(B_VFULL + s, ph)) { ok = false; break; }
      if (more && !wait(B_KFULL + s1, ph1)) { ok = false; break; }
      for (int t = 0; t < n_tiles; ++t) {
        const int nt = n_own(t);
        if (j >= nt) continue;  // (causal) this query tile is past its diagonal
        // P_t(j) V_j, then S_t(j+1) over the columns P_t(j) occupies
        if (!wait(B_PFULL + t, j & 1)) { ok = false; break; }
        tc_fence_after();
        issue_pv(t, s, j > 0);
        mma_commit(BAR(B_ODONE + t), leader);
        if (j + 1 < nt) {
          issue_s(t, s1);
          mma_commit(BAR(B_SFULL + t), leader);
        }
      }
      if (!ok) break;
      mma_commit(BAR(B_VEMPTY + s), leader);
      if (more) mma_commit(BAR(B_KEMPTY + s1), leader);
    }
    if (!ok && lane == 0) *abort_flag = 1;
    // drain every MMA issued before TMEM can be released
    mma_commit(BAR(B_DRAIN), leader);
    wait(B_DRAIN, 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - C::SW0) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;             // TMEM lane quarter
    const int row_in_tile = wq * 32 + lane;
    const int row = q0 + t * C::BM + row_in_tile;
    const bool live_tile = t < n_tiles;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + C::S_COL(t);
    const uint32_t o_addr = lane_addr + C::O_COL(t);
    const uint64_t c22 = f2_pack(a.scale_log2, a.scale_log2);
    const int nt = live_tile ? n_own(t) : 0;
    const int key_end = causal ? min(N, row + 1) : N;  // keys this row sees: [0, key_end)
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      const bool w = mbar_wait(BAR(B_SFULL + t), j & 1, a.status, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      // Keys past N (the sequence's last key tile) and, causal, keys after
      // this row (the last two key tiles of the query tile) are masked.
      const int valid = key_end - j * C::BN;
      const bool mask = valid < C::BN;
      // Both 32-column halves of the row are loaded at once (one TMEM round
      // trip); the row max comes first, so every exponential is computed
      // once, against the final reference max of this tile.
      uint32_t ra[32], rb[32];
      tmem_ld32(s_addr, ra);
      tmem_ld32(s_addr + 32, rb);
      tmem_ld_wait_dep(ra);
      tmem_ld_wait_dep(rb);
      if (mask) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          ra[i] = i >= valid ? __float_as_uint(-INFINITY) : ra[i];
          rb[i] = 32 + i >= valid ? __float_as_uint(-INFINITY) : rb[i];
        }
      }
      float mx[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx[u] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        mx[i & 3] = fmax3(mx[i & 3], __uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
        mx[(i + 2) & 3] = fmax3(mx[(i + 2) & 3], __uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
      }
      // raise the reference max only when the tile's max exceeds it by more
      // than kRescaleLog2Q4 (always on the first tile)
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
      const bool need = mt > m_ref + kRescaleLog2Q4;
      const float m_new = need ? mt : m_ref;
      const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;  // 0 on the first tile
      m_ref = m_new;
      uint64_t sm2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sm2[u] = 0ull;
      {
        // P (bf16 pairs) over the first 32 S columns, each half stored as soon
        // as it is computed: the S columns it covers are already in registers
        const uint64_t nm2 = f2_pack(-m_new, -m_new);
        uint32_t pk[16];
        q4_chunk32(ra, pk, c22, nm2, sm2);
        tmem_st16(s_addr, pk);
        q4_chunk32(rb, pk, c22, nm2, sm2);
        tmem_st16(s_addr + 16, pk);
      }
      const float2 sa = f2_unpack(fadd2(fadd2(sm2[0], sm2[1]), fadd2(sm2[2], sm2[3])));
      l = l * alpha + (sa.x + sa.y);
      // P_t(j-1) V_{j-1} completed before S_t(j) (committed after it), so O
      // can be rescaled here, before P_t(j) V_j is issued.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int q = 0; q < C::D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(o_addr + 32 * q, o);
          tmem_ld_wait_dep(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(o_addr + 32 * q, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL + t));
    }
    tmem_st_wait();  // no TMEM store may be in flight when the loop is left early
    if (ok && live_tile) {
      const bool w = mbar_wait(BAR(B_ODONE + t), (nt - 1) & 1, a.status, a.wait_limit_ns);
      ok = __all_sync(0xffffffffu, w);
    }
    // the tile's four warps take one decision (they share the store barrier)
    if (t == 0) ok = named_bar_and<1>(128, ok);
    else if (t == 1) ok = named_bar_and<2>(128, ok);
    else if (t == 2) ok = named_bar_and<3>(128, ok);
    else ok = named_bar_and<4>(128, ok);
    if (!ok) *abort_flag = 1;
    if (ok && live_tile) {
      // Epilogue: O / l as bf16 into the tile's Q slot (its last S product has
      // read it) in the 128-byte swizzle of the TMA box, then one tensor
      // store of 64 columns x 128 rows (rows past N are not written).
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint8_t* stage = smem + C::OFF_Q + t * C::Q_BYTES;
#pragma unroll
      for (int q = 0; q < C::D / 32; ++q) {
        uint32_t r[32];
        tmem_ld32(o_addr + 32 * q, r);
        tmem_ld_wait_dep(r);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
          u.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
          u.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
          u.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
          const int k = 4 * q + v;  // 16-byte unit of the 128-byte row
          *reinterpret_cast<uint4*>(stage + row_in_tile * 128 + ((k ^ (row_in_tile & 7)) << 4)) = u;
        }
      }
      fence_proxy_async_smem();
      if (t == 0) named_bar_sync<1>(128);
      else if (t == 1) named_bar_sync<2>(128);
      else if (t == 2) named_bar_sync<3>(128);
      else named_bar_sync<4>(128);
      if (wq == 0 && lane == 0) {
        tma_store_3d(&a.tmO, smem_u32(stage), 0, q0 + t * C::BM, plane);
        bulk_commit_group();
        bulk_wait_group_read<0>();  // the slot is read before the CTA exits; the writes land before the kernel ends
      }
      if (row < N) a.LSE[(size_t)plane * (size_t)a.seq.stat_plane + row] = (m_ref + __log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_fwd_bf16_q4(const FwdArgs& a, int BH, cudaStream_t st) {
  using C = Q4Cfg;
  if (a.seq.cu_seqlens || a.splits != 1) return cudaErrorInvalidValue;
  auto kernel = a.seq.causal ? fwd_bf16_q4_kernel<true> : fwd_bf16_q4_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long long qblocks = ((long long)a.seq.N + C::BM * C::QT - 1) / (C::BM * C::QT);
  dim3 grid((unsigned)(qblocks * BH));
  if (a.seq.causal) {
    // every CTA of a head streams the head's K and V (budget: most of L2)
    const int hpg = causal_heads_per_group(BH, 4ll * a.seq.N * C::D, 96ll << 20);
    grid = dim3((unsigned)hpg, (unsigned)qblocks, (unsigned)((BH + hpg - 1) / hpg));
  }
  kernel<<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
