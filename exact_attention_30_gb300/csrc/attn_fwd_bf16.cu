// attn_fwd_bf16.cu -- fused exact-attention forward on sm_103a tensor cores.
//
// What it computes ("Lesson 1: FlashAttention core idea" §4, query tiles
// outer / key-value tiles inner; "FlashAttention and Triton" §19.4-§19.6):
//   per query row r:  O_r = sum_c exp(s_rc - m_r) V_c / l_r,
//                     LSE_r = m_r + ln(l_r),  s = scale * q.k
// with S and P held only in tensor memory (TMEM) and registers.
//
// CTA = one (batch*head, 256-row query block) = two 128-row query tiles.
// Warp roles (10 warps):
//   warp 0      TMA producer: Q tiles once, then K_j / V_j through a ring of
//               STAGES shared-memory slots (full/empty mbarrier pairs).
//   warp 1      TMEM allocation; the converged warp runs the MMA schedule
//               and one elected lane issues every tcgen05.mma:
//                 S_t = Q_t K_j^T   (SS form, fp32 accumulator in TMEM)
//                 O_t += P_t V_j    (TS form: P read from TMEM, V from smem)
//               in the order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) (d = 128),
//               so the tensor core works on one query tile while the softmax
//               warps work on the other; at d = 64, where P has TMEM columns
//               of its own, S_t(j+1) goes before PV_t(j), as soon as the
//               softmax has read S_t(j).
//   warps 2-5   softmax for query tile 0, one thread per row (TMEM lane);
//   warps 6-9   softmax for query tile 1.
// Online softmax ("Lesson 1" §3) in the log2 domain: x = s * scale*log2(e),
// p = 2^(x - m_ref), l = l * 2^(m_ref_old - m_ref) + rowsum(p). The reference
// max m_ref is only raised when the tile max exceeds it by more than
// kRescaleLog2 (p <= 2^kRescaleLog2 meanwhile); O and l always share the same
// m_ref, so the result is exact in real arithmetic (the argument of
// "Lesson 1" §4: every term is normalised to one common max). When m_ref
// moves, the row of O in TMEM is multiplied by 2^(m_old - m_new) before the
// next P V product is issued. P is rounded to bf16 and written over the S
// columns it came from (d = 128), or into columns of its own (d = 64, where
// TMEM has room); either way it is the A operand of the TS MMA.
// Epilogue: O / l to bf16 through the tile's Q slot and TMA tensor stores,
// LSE = (m_ref + log2 l) * ln 2, rows >= N skipped.
//
// Grid (non-causal): one CTA per unit (batch*head, 256-row block), head-major.
// When the last wave of CTAs is only partly filled, the caller's scratch lets
// its units run as 2-4 key ranges each; a range writes its normalised fp32 O
// and base-2 LSE, and fwd_tail_merge_kernel combines the ranges afterwards.
//
// Sequences: a CTA works on one sequence of the SeqArgs layout (fixed length,
// or one entry of a packed variable-length batch); keys past the sequence's
// end are masked like a ragged tail. Causal attention (query row r sees keys
// c <= r) visits only the key tiles up to each query tile's diagonal and
// masks the diagonal tile; the grid then lists the CTAs with the most key
// tiles first (longest-processing-time order), so the short ones fill the
// last wave.
//
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the status word, drains its in-flight TMA loads and MMAs, frees TMEM and
// exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr float kRescaleLog2 = 8.0f;  // tolerated growth of the running max before O is rescaled
constexpr int kMaxTailSplits = 4;     // key ranges of a split unit (the host plan's bound)

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;  // query rows per tile (TMEM lanes)
  static constexpr int QT = 2;    // query tiles per CTA
  static constexpr int BN = 128;  // keys per KV tile
  static constexpr int CH = D / 64;  // 128-byte column chunks per row
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int CHUNK_BYTES = 128 * 128;  // one 128-row x 128-byte swizzled chunk
  static constexpr int TILE_BYTES = CH * CHUNK_BYTES;  // 128 rows x D bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QT * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE_BYTES;
  static constexpr int NBAR = QT + 4 * STAGES + 4 * QT + 1;
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1024-byte alignment
  // warps: 0 producer, 1 MMA, 2-5 and 6-9 the softmax warpgroups of query
  // tiles 0 and 1 (any four consecutive warps cover the four TMEM lane
  // quarters); 320 threads leave 200 registers per thread
  static constexpr int SW0 = 2;
  static constexpr int THREADS = 32 * (SW0 + 4 * QT);
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S_t at 128*t, O_t at 256 + D*t. With d = 64 the last 128
  // columns are free and hold P_t (64 columns of bf16 pairs each), so P can
  // be written while S is still being read; with d = 128 P goes over S.
  static constexpr bool P_OWN = (D == 64);
  static constexpr uint32_t S_COL(int t) { return 128u * t; }
  static constexpr uint32_t O_COL(int t) { return 256u + (uint32_t)D * t; }
  static constexpr uint32_t P_COL(int t) { return P_OWN ? 256u + 2u * D + 64u * t : S_COL(t); }
};

// Scores past `valid` (ragged tail, causal diagonal) become -inf.
__device__ __forceinline__ void mask_cols32(uint32_t (&r)[32], int c0, int valid) {
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = c0 + i >= valid ? __float_as_uint(-INFINITY) : r[i];
}

// One 32-column chunk of a row of S: p = 2^(s*c2 - m) for column pairs
// (packed fp32 arithmetic), the row sums in four packed accumulators, the row
// max alongside when asked, and the chunk's P as bf16 pairs.
template <bool WITH_MAX>
__device__ __forceinline__ void softmax_chunk32(const uint32_t (&r)[32], uint32_t (&pk)[16],
                                                uint64_t c22, uint64_t nm2, float (&mx)[4],
                                                uint64_t (&sm2)[4]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float s0 = __uint_as_float(r[2 * i]), s1 = __uint_as_float(r[2 * i + 1]);
    if (WITH_MAX) mx[i & 3] = fmax3(mx[i & 3], s0, s1);
    const float2 x = f2_unpack(ffma2(f2_pack(s0, s1), c22, nm2));
    const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
    sm2[i & 3] = fadd2(sm2[i & 3], f2_pack(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
  }
}

// A 128-column row of S read in four 32-column chunks, each load in flight
// while the chunk before it is exponentiated; each chunk's P goes to TMEM
// columns of its own. Before the first P store the thread waits for the
// previous P V product to finish reading those columns (o_wait, on the
// o_done barrier); false if that bounded wait expired (nothing stored then).
template <bool WITH_MAX>
__device__ __forceinline__ bool softmax_pass_own_p(uint32_t s_addr, uint32_t p_addr,
                                                   bool mask_tile, int valid, uint64_t c22,
                                                   uint64_t nm2, float (&mx)[4],
                                                   uint64_t (&sm2)[4], bool o_wait,
                                                   uint32_t o_done, uint32_t o_parity,
                                                   int* status, unsigned long long limit_ns) {
  uint32_t ra[32], rb[32], pk[16];
  tmem_ld32(s_addr, ra);
  tmem_ld_wait_dep(ra);
  // not unrolled: fully unrolled, ptxas batches the exponentials of all the
  // chunks and runs out of registers
#pragma unroll 1
  for (int c = 0; c < 4; c += 2) {
    tmem_ld32(s_addr + 32 * (c + 1), rb);
    if (mask_tile) mask_cols32(ra, 32 * c, valid);
    softmax_chunk32<WITH_MAX>(ra, pk, c22, nm2, mx, sm2);
    if (c == 0 && o_wait &&
        !__all_sync(0xffffffffu, mbar_wait(o_done, o_parity, status, limit_ns))) {
      tmem_ld_wait();  // the load in flight lands before its registers go away
      return false;
    }
    tmem_st16(p_addr + 16 * c, pk);
    tmem_ld_wait_dep(rb);
    if (c + 2 < 4) tmem_ld32(s_addr + 32 * (c + 2), ra);
    if (mask_tile) mask_cols32(rb, 32 * (c + 1), valid);
    softmax_chunk32<WITH_MAX>(rb, pk, c22, nm2, mx, sm2);
    tmem_st16(p_addr + 16 * (c + 1), pk);
    if (c + 2 < 4) tmem_ld_wait_dep(ra);
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1) fwd_bf16_kernel(const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  // barrier indices
  const uint32_t bar0 = smem_u32(bars);
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const int B_QFULL = 0;  // + query tile: each Q tile has its own barrier
  const int B_KFULL = C::QT, B_VFULL = C::QT + C::STAGES, B_KEMPTY = C::QT + 2 * C::STAGES,
            B_VEMPTY = C::QT + 3 * C::STAGES;
  const int B_SFULL = C::QT + 4 * C::STAGES, B_PFULL = B_SFULL + C::QT, B_ODONE = B_PFULL + C::QT;
  const int B_SFREE = B_ODONE + C::QT;  // S read by the softmax (own-P layout only)
  const int B_DRAIN = B_SFREE + C::QT;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);


  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool causal = a.seq.causal != 0;
  int bh, qblk;
  int tail_unit = -1, part = 0;  // split units: index among them, key part
  if (causal) {
    // causal grids: (heads of a group, query blocks from the last = most key
    // tiles to the first, head groups)
    bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    qblk = (int)(gridDim.y - 1 - blockIdx.y);
  } else {
    // one CTA per unit (head, 256-row block), head-major; the units from
    // n_full on are split into a.splits key ranges, one CTA each
    const int qblocks = (a.seq.N + C::BM * C::QT - 1) / (C::BM * C::QT);
    int u = (int)blockIdx.x;
    if (u >= a.n_full) {
      const int r = u - a.n_full;
      tail_unit = r / a.splits;
      part = r - tail_unit * a.splits;
      u = a.n_full + tail_unit;
    }
    bh = u / qblocks;
    qblk = u - bh * qblocks;
  }
  if (bh >= a.BH) return;  // past the last head of the last group
  const SeqView sv = seq_view(a.seq, bh, a.status);
  const int N = sv.len;  // queries = keys of this sequence
  const int q0 = qblk * (C::BM * C::QT);
  if (q0 >= N) return;  // the whole CTA: nothing of this sequence here
  const int n_kv = (N + C::BN - 1) / C::BN;
  // key tiles kt0 + j, j < n_t0 (query tile 0) or n_t1 (tile 1): all of
  // them, up to the diagonal (causal), or this CTA's part of a split unit
  int kt0 = 0, kt_end = n_kv;
  if (tail_unit >= 0) {
    kt0 = (int)((long long)part * n_kv / a.splits);
    kt_end = (int)((long long)(part + 1) * n_kv / a.splits);
  }
  const int qt0 = q0 / C::BM;
  const int n_t0 = causal ? min(qt0 + 1, n_kv) : kt_end - kt0;
  const int n_t1 = causal ? min(qt0 + 2, n_kv) : kt_end - kt0;  // >= n_t0
  const int n_max = n_t1;
  const int y0 = sv.start;  // first row of the sequence in the TMA views
  const int plane = sv.plane;

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
      mbar_init(BAR(B_PFULL + t), 4);  // one arrival per softmax warp
      mbar_init(BAR(B_ODONE + t), 1);
      mbar_init(BAR(B_SFREE + t), 4);
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
      // Q tile 0, then K_0, then the other Q tiles: S_0(0) needs only the first two
      auto load_q = [&](int t) {
        mbar_arrive_expect_tx(BAR(B_QFULL + t), C::TILE_BYTES);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d(sbase + C::OFF_Q + (t * C::CH + c) * C::CHUNK_BYTES, &a.tmQ, BAR(B_QFULL + t),
                      c * 64, y0 + q0 + t * C::BM, plane);
      };
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
          mbar_arrive_expect_tx(BAR(B_KFULL + s), C::TILE_BYTES);
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d(sbase + C::OFF_K + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &a.tmK,
                        BAR(B_KFULL + s), c * 64, y0 + (kt0 + j) * C::BN, plane);
          last_k[s] = j;
        }
        if (j == 0)
          for (; q_loaded < C::QT; ++q_loaded) load_q(q_loaded);
        if (!mbar_wait(BAR(B_VEMPTY + s), ph ^ 1, a.status, a.wait_limit_ns)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(BAR(B_VFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d(sbase + C::OFF_V + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &a.tmV,
                      BAR(B_VFULL + s), c * 64, y0 + (kt0 + j) * C::BN, plane);
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
    // The whole warp runs this loop converged (waits, descriptor arithmetic);
    // tcgen05.mma and tcgen05.commit are issued by the one elected lane.
    {
      const uint32_t leader = elect_one();
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      // Descriptors are built once; advancing along K only adds a byte offset
      // (>> 4) to the 14-bit start-address field, which cannot carry out of it
      // because every operand lies below 256 KB of shared memory.
      const uint64_t dQ0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sbase + C::OFF_V, C::CHUNK_BYTES, 1024);
      auto issue_s = [&](int t, int s) {
        const uint64_t qa = dQ0 + (uint64_t)((t * C::TILE_BYTES) >> 4);
        const uint64_t kb = dK0 + (uint64_t)((s * C::TILE_BYTES) >> 4);
        const uint32_t dcol = tmem + C::S_COL(t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4);
          mma_ss(dcol, qa + off, kb + off, idesc_s, kk > 0 ? 1u : 0u, leader);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint64_t vb = dV0 + (uint64_t)((s * C::TILE_BYTES) >> 4);
        const uint32_t dcol = tmem + C::O_COL(t), acol = tmem + C::P_COL(t);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ts(dcol, acol + kk * 8, vb + (uint64_t)((kk * 2048) >> 4), idesc_o,
                 (acc || kk > 0) ? 1u : 0u, leader);
      };
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait_warp(BAR(b), parity, a.status, a.wait_limit_ns);
      };
      bool ok = wait(B_QFULL + 0, 0) && wait(B_KFULL + 0, 0);
      for (int t = 0; ok && t < C::QT; ++t) {
        if (t > 0 && !wait(B_QFULL + t, 0)) { ok = false; break; }
        tc_fence_after();
        issue_s(t, 0);
        mma_commit(BAR(B_SFULL + t), leader);
      }
      if (ok) mma_commit(BAR(B_KEMPTY + 0), leader);
      for (int j = 0; ok && j < n_max; ++j) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        const int s1 = (j + 1) % C::STAGES;
        const uint32_t ph1 = ((j + 1) / C::STAGES) & 1;
        bool k_next = false;  // K_{j+1} has landed
        bool v_here = false;  // V_j has landed
        for (int t = 0; t < C::QT; ++t) {
          const int n_own = t == 0 ? n_t0 : n_t1;
          if (j >= n_own) continue;  // this query tile is past its diagonal
          if constexpr (C::P_OWN) {
            // P has its own columns: S_{j+1} may overwrite S_j as soon as the
            // softmax has read it, so it goes first and is ready when the
            // softmax of tile j is done; P_j V_j follows.
            if (j + 1 < n_own) {
              if (!wait(B_SFREE + t, j & 1)) { ok = false; break; }
              if (!k_next && !wait(B_KFULL + s1, ph1)) { ok = false; break; }
              k_next = true;
              tc_fence_after();
              issue_s(t, s1);
              mma_commit(BAR(B_SFULL + t), leader);
            }
            if (!wait(B_PFULL + t, j & 1)) { ok = false; break; }
            if (!v_here && !wait(B_VFULL + s, ph)) { ok = false; break; }
            v_here = true;
            tc_fence_after();
            issue_pv(t, s, j > 0);
            mma_commit(BAR(B_ODONE + t), leader);
          } else {
            // P overwrites S: P_j V_j must be issued before S_{j+1}.
            if (!v_here && !wait(B_VFULL + s, ph)) { ok = false; break; }
            v_here = true;
            if (!wait(B_PFULL + t, j & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, s, j > 0);
            mma_commit(BAR(B_ODONE + t), leader);
            if (j + 1 < n_own) {
              if (!k_next && !wait(B_KFULL + s1, ph1)) { ok = false; break; }
              k_next = true;
              tc_fence_after();
              issue_s(t, s1);
              mma_commit(BAR(B_SFULL + t), leader);
            }
          }
        }
        if (!ok) break;
        mma_commit(BAR(B_VEMPTY + s), leader);
        if (j + 1 < n_max) mma_commit(BAR(B_KEMPTY + s1), leader);
      }
      if (!ok && lane == 0) *abort_flag = 1;
      // drain every MMA issued before TMEM can be released
      mma_commit(BAR(B_DRAIN), leader);
      wait(B_DRAIN, 0);
    }
  } else if (warp >= C::SW0) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - C::SW0) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;             // TMEM lane quarter
    const int row_in_tile = wq * 32 + lane;
    const int row = q0 + t * C::BM + row_in_tile;  // within the sequence
    const int n_own = t == 0 ? n_t0 : n_t1;
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + C::S_COL(t);
    const uint32_t o_addr = lane_addr + C::O_COL(t);
    const float c2 = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_own; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      bool w = mbar_wait(BAR(B_SFULL + t), j & 1, a.status, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      // Raw scores of this row (d = 128: 64 columns at a time, two 32-column
      // loads, one wait). Only the last key tile of a query tile can hold masked columns:
      // keys past the sequence's end, and (causal) keys after this row.
      uint32_t r[64];
      const bool mask_tile = j == n_own - 1;
      int valid = N - (kt0 + j) * C::BN;  // >= 128 unless this is the sequence's last tile
      if (causal) valid = min(valid, row - j * C::BN + 1);
      auto load_half = [&](int h) {
        tmem_ld32(s_addr + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(s_addr + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld_wait();
        if (mask_tile) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            r[i] = 64 * h + i >= valid ? __float_as_uint(-INFINITY) : r[i];
        }
      };
      // Speculative pass: exponentiate against the current reference max while
      // this tile's row max is computed alongside (max, exp2 and the sums run
      // on different pipes). Only when the tile max exceeds the reference by
      // more than kRescaleLog2 -- always on the first tile, rarely later -- is
      // the tile redone against the new max, from S re-read out of TMEM (P is
      // written over S only after this decision). Scale > 0 commutes with max.
      // Pairs of columns go through packed fp32 arithmetic (fma/add .f32x2)
      // and a three-input max: fewer issued instructions per score, which
      // also leaves issue slots to the MMA warp sharing these sub-partitions.
      float mx[4];
      uint64_t sm2[4];
      const uint64_t c22 = f2_pack(c2, c2);
#pragma unroll
      for (int u = 0; u < 4; ++u) { mx[u] = -INFINITY; sm2[u] = 0ull; }
      float mt;
      bool need;
      float alpha = 1.f;
      if constexpr (C::P_OWN) {
        // P has columns of its own: S is read in 32-column chunks, the next
        // chunk's load in flight while the current one is exponentiated, and
        // each chunk's P goes to TMEM at once (no register copy of the tile).
        // S_j was issued before P_{j-1} V_{j-1}, which must have finished
        // reading P's columns before the first store.
        const uint32_t p_addr = lane_addr + C::P_COL(t);
        const float neg_m = (j > 0) ? -m_ref : 0.f;
        if (!softmax_pass_own_p<true>(s_addr, p_addr, mask_tile, valid, c22, f2_pack(neg_m, neg_m),
                                      mx, sm2, j > 0, BAR(B_ODONE + t), (uint32_t)(j - 1) & 1u,
                                      a.status, a.wait_limit_ns)) {
          ok = false;
          break;
        }
        mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
        need = mt > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mt : m_ref;
          alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) sm2[u] = 0ull;
          tmem_st_wait();  // the speculative P is overwritten below
          softmax_pass_own_p<false>(s_addr, p_addr, mask_tile, valid, c22, f2_pack(-m_new, -m_new),
                                    mx, sm2, false, 0u, 0u, a.status, a.wait_limit_ns);
          m_ref = m_new;
        }
        // S_j has been read: S_{j+1} may be written over it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_SFREE + t));
      } else {
        uint32_t pk[64];
        {
          const float neg_m = (j > 0) ? -m_ref : 0.f;
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            load_half(h);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float s0 = __uint_as_float(r[2 * i]), s1 = __uint_as_float(r[2 * i + 1]);
              mx[i & 3] = fmax3(mx[i & 3], s0, s1);
              const float2 x = f2_unpack(ffma2(f2_pack(s0, s1), c22, nm2));
              const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
              sm2[i & 3] = fadd2(sm2[i & 3], f2_pack(p0, p1));
              pk[32 * h + i] = pack_bf16x2(p0, p1);
            }
          }
        }
        mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
        need = mt > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // redo for the whole warp (rows that keep their max recompute the
          // same values)
          const float m_new = need ? mt : m_ref;
          alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
          const uint64_t nm2 = f2_pack(-m_new, -m_new);
#pragma unroll
          for (int u = 0; u < 4; ++u) sm2[u] = 0ull;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            load_half(h);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c22, nm2));
              const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
              sm2[i & 3] = fadd2(sm2[i & 3], f2_pack(p0, p1));
              pk[32 * h + i] = pack_bf16x2(p0, p1);
            }
          }
          m_ref = m_new;
        }
        // P (bf16) over the first 64 S columns
        tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      }
      const float2 sa = f2_unpack(fadd2(fadd2(sm2[0], sm2[1]), fadd2(sm2[2], sm2[3])));
      l = l * alpha + (sa.x + sa.y);
      // P V of the previous tile is complete here: with P over S, S of this
      // tile was committed after it (a commit tracks every earlier MMA); with
      // P in its own columns the pass above waited on o_done. So O can be
      // rescaled at once.
      if (j > 0) {
        if (__any_sync(0xffffffffu, need)) {  // alpha == 1 on rows whose max did not move
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            tmem_ld32(o_addr + 32 * q, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(o_addr + 32 * q, o);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL + t));
    }
    tmem_st_wait();  // no TMEM store may be in flight when the loop is left early
    if (ok && n_own > 0) {
      const bool w = mbar_wait(BAR(B_ODONE + t), (n_own - 1) & 1, a.status, a.wait_limit_ns);
      ok = __all_sync(0xffffffffu, w);
    }
    // Every warp that shares an epilogue barrier takes the same decision: a
    // warp that gave up must not leave the others waiting at a barrier it
    // never reaches. Split units: both tiles' warps (they stage into shared
    // memory the other tile may still read); otherwise the tile's own four.
    if (tail_unit >= 0) ok = named_bar_and<1>(256, ok);
    else if (t == 0) ok = named_bar_and<2>(128, ok);
    else ok = named_bar_and<3>(128, ok);
    if (!ok) *abort_flag = 1;
    if (tail_unit >= 0) {
      // One key part of a split unit: its normalised partial O (fp32) and
      // base-2 LSE go to the workspace; fwd_tail_merge_kernel, launched after
      // this kernel, combines the parts. Both tiles' products are complete
      // past the barrier above, so all of shared memory is free: tile t
      // stages its rows in [OFF_Q + t * D * 512, ...) as 32-column boxes of
      // 128 rows in the TMA 128-byte swizzle, and one thread stores them.
      const int rows_unit = C::BM * C::QT;
      const int prow0 = (tail_unit * a.splits + part) * rows_unit + t * C::BM;  // tile's first workspace row
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        uint8_t* stage = smem + C::OFF_Q + t * (D * 512);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(o_addr + 32 * q, r);
          tmem_ld_wait();
          uint8_t* box = stage + q * 16384 + row_in_tile * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(box + ((k ^ (row_in_tile & 7)) << 4)) =
                make_float4(__uint_as_float(r[4 * k]) * inv_l, __uint_as_float(r[4 * k + 1]) * inv_l,
                            __uint_as_float(r[4 * k + 2]) * inv_l, __uint_as_float(r[4 * k + 3]) * inv_l);
        }
        a.Lpart[prow0 + row_in_tile] = m_ref + __log2f(l);
        fence_proxy_async_smem();
      }
      if (t == 0) named_bar_sync<2>(128);
      else named_bar_sync<3>(128);
      if (ok && warp == C::SW0 + 4 * t && lane == 0) {
        const uint8_t* stage = smem + C::OFF_Q + t * (D * 512);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) tma_store_2d(&a.tmOpart, smem_u32(stage + q * 16384), q * 32, prow0);
        bulk_commit_group();
        bulk_wait_group_read<0>();  // the staging read; the writes land before the kernel ends
      }
    } else if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      // A tile that cannot reach past its sequence's rows in the tensor (fixed
      // length: rows past N are outside the map and not written) leaves
      // through the tile's Q slot, which its last S product has finished
      // reading: bf16 rows in the 128-byte swizzle of the TMA box (16-byte
      // unit k of row r at k ^ (r % 8), so the 32 lanes' stores spread over
      // all banks), then tensor stores of 64 columns x 128 rows. The other
      // tiles (a packed sequence's last, partial tile) store row by row.
      const bool tma_out = a.seq.cu_seqlens == nullptr || q0 + (t + 1) * C::BM <= N;
      if (tma_out) {
        uint8_t* stage = smem + C::OFF_Q + t * C::TILE_BYTES;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(o_addr + 32 * q, r);
          tmem_ld_wait();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c0 = 32 * q + 8 * v;  // first column of this 16-byte unit
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
            u.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
            u.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
            u.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
            const int k = (c0 & 63) >> 3;
            *reinterpret_cast<uint4*>(stage + (c0 >> 6) * C::CHUNK_BYTES + row_in_tile * 128 +
                                      ((k ^ (row_in_tile & 7)) << 4)) = u;
          }
        }
        fence_proxy_async_smem();
        if (t == 0) named_bar_sync<2>(128);  // this tile's softmax warps
        else named_bar_sync<3>(128);
        if (warp == C::SW0 + 4 * t && lane == 0) {
#pragma unroll
          for (int c = 0; c < C::CH; ++c)
            tma_store_3d(&a.tmO, smem_u32(stage + c * C::CHUNK_BYTES), c * 64, y0 + q0 + t * C::BM, plane);
          bulk_commit_group();
          bulk_wait_group_read<0>();  // the slot read before the CTA exits; the writes land before the kernel ends
        }
      } else {
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.O) + seq_row_offset(a.seq, sv, row);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(o_addr + 32 * q, r);
          tmem_ld_wait();
          if (row < N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * q);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 u;
              u.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
              u.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
              u.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
              u.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
              dst[v] = u;
            }
          }
        }
      }
      if (row < N) a.LSE[seq_stat_index(a.seq, sv, row)] = (m_ref + __log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Combines the key parts of the split units ("Lesson 1: FlashAttention core
// idea" §3: partial softmaxes merge through their maxima and sums): row r
// gets O = sum_p w_p O_p / sum_p w_p with w_p = 2^(L_p - max L), and LSE =
// (max L + log2 sum_p w_p) ln 2. Warp-wide rows (lanes along d, coalesced),
// 16 / S rows per warp with every part's loads in flight (S = a.splits).
template <int D, int S>
__global__ void __launch_bounds__(256) fwd_tail_merge_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int PER = D / 32;  // floats of a row per lane
  constexpr int RPW = 16 / S;  // rows per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_unit = 256;
  const int qblocks = (a.seq.N + rows_unit - 1) / rows_unit;
  const long long r_first = (long long)blockIdx.x * (8 * RPW) + warp * RPW;  // merged row: tail unit * 256 + row
  float lp[RPW][S];
  float x[RPW][S][PER];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const long long mr = r_first + i;
    const long long tu = mr / rows_unit, ru = mr - tu * rows_unit;
#pragma unroll
    for (int p = 0; p < S; ++p) {
      lp[i][p] = -INFINITY;
#pragma unroll
      for (int e = 0; e < PER; ++e) x[i][p][e] = 0.f;
      if (tu < a.n_tail) {
        const size_t pr = (size_t)(tu * S + p) * rows_unit + ru;
        lp[i][p] = a.Lpart[pr];
        const float* src = a.Opart + pr * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          x[i][p][0] = v.x; x[i][p][1] = v.y; x[i][p][2] = v.z; x[i][p][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          x[i][p][0] = v.x; x[i][p][1] = v.y;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const long long mr = r_first + i;
    const long long tu = mr / rows_unit, ru = mr - tu * rows_unit;
    if (tu >= a.n_tail) continue;
    const long long u = a.n_full + tu;
    const long long bh = u / qblocks;
    const long long row = (u - bh * qblocks) * rows_unit + ru;
    if (row >= a.seq.N) continue;
    float L = -INFINITY;
#pragma unroll
    for (int p = 0; p < S; ++p) L = fmaxf(L, lp[i][p]);
    float w[S], wsum = 0.f;
#pragma unroll
    for (int p = 0; p < S; ++p) {
      w[p] = exp2f(lp[i][p] - L);
      wsum += w[p];
    }
    const float inv_w = 1.f / wsum;
    float y[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      float acc = 0.f;
#pragma unroll
      for (int p = 0; p < S; ++p) acc = fmaf(w[p], x[i][p][e], acc);
      y[e] = acc * inv_w;
    }
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.O) + (size_t)bh * (size_t)a.seq.plane_stride +
                          (size_t)row * (size_t)a.seq.row_stride + lane * PER;
    if constexpr (PER == 4)
      *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
    else
      *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(y[0], y[1]);
    if (lane == 0) a.LSE[(size_t)bh * (size_t)a.seq.stat_plane + row] = (L + __log2f(wsum)) * 0.69314718055994531f;
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, int BH, cudaStream_t st) {
  using C = FwdCfg<D>;
  static_assert(C::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(C::QT * D * 512 <= C::OFF_BAR - C::OFF_Q, "split-part staging fits the tile buffers");
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const unsigned qblocks = (unsigned)((a.seq.N + C::BM * C::QT - 1) / (C::BM * C::QT));
  if (a.splits < 1 || a.splits > kMaxTailSplits || a.n_full < 0 || a.n_tail < 0 ||
      (a.splits == 1) != (a.n_tail == 0) ||
      (long long)a.n_full + a.n_tail != (long long)qblocks * BH ||
      (a.splits > 1 && (a.seq.causal || a.seq.cu_seqlens || a.Opart == nullptr || a.Lpart == nullptr)))
    return cudaErrorInvalidValue;
  dim3 grid((unsigned)((long long)a.n_full + (long long)a.n_tail * a.splits));
  if (a.seq.causal) {
    // every CTA of a head streams the head's K and V (budget: most of L2)
    const int hpg = causal_heads_per_group(BH, 4ll * a.seq.N * D, 96ll << 20);
    grid = dim3((unsigned)hpg, qblocks, (unsigned)((BH + hpg - 1) / hpg));
  }
  fwd_bf16_kernel<D><<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(a);
  cudaError_t e2 = cudaGetLastError();
  if (e2 != cudaSuccess || a.splits == 1) return e2;
  const long long merge_rows = (long long)a.n_tail * C::BM * C::QT;
  auto blocks = [&](int rows_per_warp) {
    return (unsigned)((merge_rows + 8 * rows_per_warp - 1) / (8 * rows_per_warp));
  };
  if (a.splits == 2) fwd_tail_merge_kernel<D, 2><<<blocks(8), 256, 0, st>>>(a);
  else if (a.splits == 3) fwd_tail_merge_kernel<D, 3><<<blocks(5), 256, 0, st>>>(a);
  else fwd_tail_merge_kernel<D, 4><<<blocks(4), 256, 0, st>>>(a);
  return cudaGetLastError();
}

std::mutex g_slots_mu;
int g_slots[16] = {};

}  // namespace

FwdTailPlan plan_fwd_tail(long long units, int n_kv, int slots) {
  FwdTailPlan p{(int)units, 0, 1};
  if (units < 1 || slots < 1 || n_kv < 1) return p;
  const long long rem = units % slots;
  if (units < slots || rem == 0) return p;  // no whole wave before the tail, or no tail
  // Split the tail's units into as many key ranges as fit into one wave, at
  // most four and with at least four key tiles per range.
  long long sp = slots / rem;
  if (sp > 4) sp = 4;
  if (sp > n_kv / 4) sp = n_kv / 4;
  if (sp < 2) return p;
  p.n_full = (int)(units - rem);
  p.n_tail = (int)rem;
  p.splits = (int)sp;
  return p;
}

size_t fwd_tail_workspace_bytes(const FwdTailPlan& p, int d) {
  if (p.splits <= 1 || p.n_tail <= 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)p.n_tail * p.splits * 256;
  return up(rows * d * 4) + up(rows * 4);
}

int fwd_slots() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return 0;
  std::lock_guard<std::mutex> lk(g_slots_mu);
  if (g_slots[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_slots[dev] = sms;  // one forward CTA per SM (all of TMEM, most of shared memory)
  }
  return g_slots[dev];
}

cudaError_t launch_fwd_bf16(const FwdArgs& a, int BH, int d, cudaStream_t st) {
  if (d == 128) return launch_fwd_d<128>(a, BH, st);
  if (d == 64) return launch_fwd_d<64>(a, BH, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
