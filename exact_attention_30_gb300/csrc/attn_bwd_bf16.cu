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
//  1. bwd_pre:   -D and -LSE*log2(e) per row into the workspace (rows
//                padded to a multiple of 128: 0 and -inf past N, which makes
//                P = 0 there), and zero the fp32 dQ accumulator.
//  2. bwd_main:  per unit (batch*head, 128-key tile j): K_j, V_j stay in
//                shared memory while 128-query tiles i stream through a TMA
//                ring. A persistent grid (one CTA per SM) takes the units:
//                by stride when they have one length, else longest first
//                from a device counter (causal, packed batches). All products run on tcgen05 with fp32 accumulators in
//                TMEM (every MMA M = N = 128):
//                  S^T = K_j Q_i^T,  dP^T = V_j dO_i^T   (recompute; keys on lanes)
//                  dV += P^T dO_i (P^T read from TMEM), dK += dS^T Q_i
//                  dQ_i^T = K_j^T dS^T (d = 128) or dQ_i = dS K_j (d = 64)
//                  -> added into the fp32 accumulator (TMA tensor reduce-add
//                  from shared-memory staging blocks)
//                A softmax warpgroup (one thread per key) first writes bf16
//                P^T over the S^T columns, then, once dP^T is there, writes
//                bf16 dS^T into a swizzled shared-memory tile that feeds both
//                dK (K-major view) and dQ (MN-major view). dQ_i is computed
//                into the dP^T columns; a dQ warpgroup reads it out and adds
//                it to the accumulator as above. dV_j and dK_j leave TMEM
//                through a staging pass that stores whole 128-byte rows. Per query tile the
//                MMA order is dV(i), S^T(i+1), dQ(i), dK(i), dP^T(i+1), so the
//                next tile's recompute overlaps this tile's softmax.
//  3. dq_convert: fp32 accumulator times scale -> bf16 dQ.
// TMEM (512 columns): S^T|P^T, dP^T|dQ, dV, dK (P^T: queries 0-63 in columns
// 0-31, queries 64-127 in columns 64-95, bf16 pairs).
//
// Sequences (SeqArgs): preprocess and convert work on rows of whole planes;
// the main kernel works on one sequence of the layout. Keys past the
// sequence's end give P = 0 on their rows, queries past it (the next
// sequence of a packed batch) P = 0 in their columns. Causal attention
// visits only the query tiles at or after the key tile's diagonal and masks
// the diagonal tile (key r, query q: P = 0 where r > q); the grid then lists
// the key tiles with the most query tiles first.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

// ----------------------------------------------------------------------------
// 1. preprocess
// ----------------------------------------------------------------------------
// One group of D/8 lanes per row; each lane reads 8 bf16 of O and dO.
// Rows of whole planes: plane p, row n < ws_rows; rows n < total are data
// (of whichever sequence holds them), the rest padding.
// Packed batches: the main kernel's item list, longest sequence first. One
// block of the preprocess launch: each sequence's length (0 for an invalid
// pair of offsets), its rank by length (descending, then index; index order
// past 1024 sequences), and per rank the prefix sum of its units (H * key
// tiles): schedule ints [0] the item counter (zeroed), [1] the item total,
// [2 ..] the order, then the B + 1 prefix sums.
template <int BK>
__device__ void bwd_sched_block(const BwdArgs& a) {
  int* sched = a.item_counter;
  const int B = a.nseq, H = a.seq.H;
  int* order = sched + 2;
  int* prefix = order + B;
  __shared__ int lens[1024];
  __shared__ int part[256];
  const int t = threadIdx.x;
  auto len_of = [&](int b) {
    const int c0 = a.seq.cu_seqlens[b], c1 = a.seq.cu_seqlens[b + 1];
    return (0 <= c0 && c0 <= c1 && c1 <= a.seq.total && c1 - c0 <= a.seq.N) ? c1 - c0 : 0;
  };
  if (B <= 1024) {
    for (int b = t; b < B; b += 256) lens[b] = len_of(b);
    __syncthreads();
    for (int b = t; b < B; b += 256) {
      const int lb = lens[b];
      int r = 0;
      for (int b2 = 0; b2 < B; ++b2) r += (lens[b2] > lb) || (lens[b2] == lb && b2 < b);
      order[r] = b;
    }
  } else {
    for (int b = t; b < B; b += 256) order[b] = b;
  }
  __syncthreads();  // order[] (global, this block's writes) visible to the block
  const int per = (B + 255) / 256;
  const int r0 = min(B, t * per), r1 = min(B, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += H * ((len_of(order[r]) + BK - 1) / BK);
  part[t] = sum;
  __syncthreads();
  if (t == 0) {
    int acc = 0;
    for (int i = 0; i < 256; ++i) {
      const int v = part[i];
      part[i] = acc;
      acc += v;
    }
    sched[0] = 0;
    sched[1] = acc;
    prefix[B] = acc;
  }
  __syncthreads();
  int acc = part[t];
  for (int r = r0; r < r1; ++r) {
    prefix[r] = acc;
    acc += H * ((len_of(order[r]) + BK - 1) / BK);
  }
}

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
  if (a.nseq > 0 && blockIdx.x == gridDim.x - 1) {  // the extra block: the packed batch's schedule
    bwd_sched_block<128>(a);
    return;
  }
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, l = lane % LPR;
  const long long prow = (long long)warp_global * RPW + sub;  // workspace row index
  const long long total = (long long)a.planes * a.ws_rows;
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.item_counter != nullptr) *a.item_counter = 0;  // the main kernel's item counter
  float acc = 0.f;
  bool live = false;
  long long plane = 0, n = 0;
  if (prow < total) {
    plane = prow / a.ws_rows;
    n = prow - plane * a.ws_rows;
    live = n < a.seq.total;
    if (live) {
      const size_t off = (size_t)plane * (size_t)a.seq.plane_stride + (size_t)n * (size_t)a.seq.row_stride +
                         (size_t)l * 8;
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
  // Stored negated so that the main kernel forms P = 2^(s*c - LSE*log2e) with
  // one fused multiply-add and dP - D with one add (exact when they are equal).
  if (prow < total && l == 0) {
    a.Drow[prow] = live ? -acc : 0.f;
    a.lse2[prow] = live ? -a.LSE[(size_t)plane * (size_t)a.seq.stat_plane + (size_t)n] * 1.4426950408889634f
                        : -INFINITY;
  }
}

// ----------------------------------------------------------------------------
// 3. dQ convert
// ----------------------------------------------------------------------------
template <int D>
__device__ void bwd_tail_merge_rows(const BwdArgs& a, long long w);

// Blocks past the conversion's own (`conv_blocks`) add up the partial dK and
// dV of the split units (bwd_tail_merge_rows), in the same launch.
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const BwdArgs a, unsigned conv_blocks) {
  if (blockIdx.x >= conv_blocks) {
    bwd_tail_merge_rows<D>(a, ((long long)(blockIdx.x - conv_blocks) * blockDim.x + threadIdx.x) >> 5);
    return;
  }
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 elements
  const long long groups = (long long)a.planes * a.seq.total * (D / 8);
  if (idx >= groups) return;
  const long long row = idx / (D / 8);
  const int g = (int)(idx - row * (D / 8));
  const long long plane = row / a.seq.total, n = row - plane * a.seq.total;
  const float4* src = reinterpret_cast<const float4*>(a.dQacc + ((size_t)plane * a.ws_rows + n) * D + g * 8);
  const float4 x = src[0], y = src[1];
  uint4 u;
  const float f = a.scale;  // the softmax scale of dS, applied once here
  u.x = pack_bf16x2(f * x.x, f * x.y);
  u.y = pack_bf16x2(f * x.z, f * x.w);
  u.z = pack_bf16x2(f * y.x, f * y.y);
  u.w = pack_bf16x2(f * y.z, f * y.w);
  *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.dQ) + (size_t)plane * (size_t)a.seq.plane_stride +
                             (size_t)n * (size_t)a.seq.row_stride + g * 8) = u;
}

// The query ranges of a split unit summed ("Lesson 1" §5: dK_j and dV_j are
// sums over the query tiles), dK times the softmax scale, to bf16. One warp
// per key row w = tail unit * 128 + row of a split unit, lanes along d.
template <int D>
__device__ void bwd_tail_merge_rows(const BwdArgs& a, long long w) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  if (w >= (long long)a.n_tail * 128) return;
  const int tu = (int)(w >> 7), r = (int)(w & 127);
  const int kblocks = (a.seq.N + 127) / 128;
  const int u = a.n_full + tu;
  const int bh = u / kblocks, kb = u - bh * kblocks;
  const int key = kb * 128 + r;
  if (key >= a.seq.N) return;
  float sv[PER], sk[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) sv[e] = sk[e] = 0.f;
  for (int p = 0; p < a.splits; ++p) {
    const float* base = a.dKVpart + ((size_t)(tu * a.splits + p) * 2) * 128 * D + (size_t)r * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      sv[e] += base[e];
      sk[e] += base[(size_t)128 * D + e];
    }
  }
  const size_t off = (size_t)bh * (size_t)a.seq.plane_stride + (size_t)key * (size_t)a.seq.row_stride + lane * PER;
  __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(a.dV) + off;
  __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(a.dK) + off;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    *reinterpret_cast<uint32_t*>(dv + e) = pack_bf16x2(sv[e], sv[e + 1]);
    *reinterpret_cast<uint32_t*>(dk + e) = pack_bf16x2(a.scale * sk[e], a.scale * sk[e + 1]);
  }
}

// ----------------------------------------------------------------------------
// 2. main kernel
// ----------------------------------------------------------------------------
template <int D>
struct BwdCfg {
  static constexpr int BK = 128;  // keys per CTA: TMEM lanes of S^T, dP^T, dV, dK
  static constexpr int BQ = 128;  // queries per streamed tile
  // d = 128 computes dQ^T = K^T dS^T (d on the TMEM lanes: a warp's lanes
  // fill one 128-byte row segment of a staging block); d = 64 computes
  // dQ = dS K (queries on the lanes; an M = 64 product would be needed
  // otherwise) and stages each lane's row through a swizzled block
  static constexpr bool DQ_T = (D == 128);
  static constexpr int CH = D / 64;                  // 128-byte chunks per K/V/Q/dO row
  // Q_i (with its LSE/D statistics) is read by S^T(i), issued one tile
  // early, and last by dK(i); dO_i by dP^T(i), also issued one tile early,
  // and last by dV(i), the first product of tile i. So Q needs a deep ring
  // for its loads to run ahead, while one dO slot already gives its load
  // most of a tile of lead time.
  static constexpr int QSTAGES = (D == 128) ? 2 : 4;  // d = 128: room for the dQ staging
  static constexpr int DOSTAGES = (D == 128) ? 1 : 2;
  static constexpr int ROW_CHUNK = 128 * 128;        // 128 rows x 128 bytes, swizzled
  static constexpr int TILE = CH * ROW_CHUNK;        // 128 rows x D bf16
  static constexpr int DS_TILE = 2 * ROW_CHUNK;      // dS^T: [128 keys][128 queries] bf16
  static constexpr int STAT_BYTES = 2 * BQ * 4;      // LSE*log2(e) and D of one query tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_DS = OFF_V + TILE;
  static constexpr int OFF_Q = OFF_DS + DS_TILE;
  static constexpr int OFF_DO = OFF_Q + QSTAGES * TILE;
  static constexpr int OFF_STAT = OFF_DO + DOSTAGES * TILE;
  static constexpr int STATSTAGES = 2;  // LSE*log2e and D, read by both softmax phases
  // dQ reduction staging: per dQ warp 2 x [32 queries][32 d] fp32, added
  // into the global accumulator by the TMA engine (tensor bulk reduce-add)
  // instead of fp32 atomics. 1024-byte aligned (the d = 64 blocks are
  // written in the TMA 128-byte swizzle).
  static constexpr int DQ_ROWS = 32;
  static constexpr int DQ_BLOCK_BYTES = DQ_ROWS * 32 * 4;  // 4 KB
  static constexpr int OFF_DQS = OFF_STAT + STATSTAGES * STAT_BYTES;
  static constexpr int OFF_BAR = OFF_DQS + 4 * 2 * DQ_BLOCK_BYTES;
  static_assert(OFF_DQS % 1024 == 0, "swizzled staging alignment");
  // barriers: kv_full, q_full[QS], q_empty[QS], do_full[DS], do_empty[DS], st_full[2],
  //           st_empty[2], s_full, dp_full, pt_ready, ds_ready, ds_empty, dq_full,
  //           dq_empty, acc_done, drain, kv_empty, acc_empty, item_full[IRING],
  //           item_empty[IRING]
  static constexpr int IRING = 4;  // items published ahead by the producer
  static constexpr int NBAR = 1 + 2 * QSTAGES + 2 * DOSTAGES + 2 * STATSTAGES + 11 + 2 * IRING;
  // after the barriers: TMEM base, abort flag, 8 bytes free, the item ring
  // (IRING published items, 8 ints each)
  static constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 32 * IRING;
  static constexpr int SMEM_MAX = 227 * 1024;
  // request 1 KB of alignment slack when it fits; the kernel checks alignment
  static constexpr int SMEM_ALLOC = (SMEM_BYTES + 1024 <= SMEM_MAX) ? SMEM_BYTES + 1024 : SMEM_MAX;
  static constexpr int THREADS = 512;  // 16 warps: producers/MMA, 2 softmax WGs, dQ WG
  // TMEM columns: S^T (P^T as bf16 in columns 0-31 and 64-95), dP^T (dQ after dP^T is
  // consumed), dV, dK.
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = 128;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= SMEM_MAX, "shared memory budget");
  static_assert(BQ == bwd_query_tile(D), "host tensor-map box height");
};

// One work item of the main kernel: a unit (batch*head, 128-key tile), or one
// query range of a split unit.
struct BwdItem {
  SeqView sv;
  int kb;         // key tile
  int i_begin;    // first query tile
  int n_it;       // query tiles
  int tail_unit;  // index among the split units, or -1
  int part;       // query range of a split unit
};

// Item w of the 1-D item list of a fixed-length problem (non-causal: units
// key tile fastest, those from n_full on as `splits` query ranges each;
// causal: head groups, then key tiles in increasing order, then the heads of
// the group), or, with list == false, this CTA's unit of the 2-D/3-D grids
// (packed batches). False: nothing to do (a head past the last one, a key
// tile past the sequence's end). Out of line: every role decodes each of its items, and
// one shared copy keeps the kernel's code (and instruction-cache footprint)
// small.
template <int BK, int BQ>
__device__ __noinline__ bool bwd_item(const BwdArgs& a, bool list, int w, BwdItem& it) {
  const bool causal = a.seq.causal != 0;
  int bh;
  it.tail_unit = -1;
  it.part = 0;
  if (w < 0) return false;
  if (list && a.seq.cu_seqlens != nullptr) {
    // packed batch: sequences longest first (the preprocess's order), then
    // heads, then key tiles; the rank by binary search of the unit prefix
    const int* order = a.item_counter + 2;
    const int* prefix = order + a.nseq;
    int lo = 0, hi = a.nseq;  // prefix[lo] <= w < prefix[hi]
    if (w >= prefix[hi]) return false;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= w) lo = mid;
      else hi = mid;
    }
    const int b = order[lo], local = w - prefix[lo];
    const int c0 = a.seq.cu_seqlens[b], c1 = a.seq.cu_seqlens[b + 1];
    const int kblocks = (c1 - c0 + BK - 1) / BK;  // >= 1 (the rank has units)
    if (kblocks < 1) return false;
    const int h = local / kblocks;
    it.kb = local - h * kblocks;
    bh = b * a.seq.H + h;
  } else if (list && causal) {
    // (heads of a group, key tiles in increasing order = most query tiles
    // first, head groups): the order of the one-CTA-per-unit causal grid
    const int kblocks = (a.seq.N + BK - 1) / BK;
    const int x = w % a.causal_hpg, rest = w / a.causal_hpg;
    it.kb = rest % kblocks;
    bh = (rest / kblocks) * a.causal_hpg + x;
  } else if (list) {
    const int kblocks = (a.seq.N + BK - 1) / BK;
    int u = w;
    if (u >= a.n_full) {
      const int r = u - a.n_full;
      it.tail_unit = r / a.splits;
      it.part = r - it.tail_unit * a.splits;
      u = a.n_full + it.tail_unit;
    }
    bh = u / kblocks;
    it.kb = u - bh * kblocks;
  } else {
    // causal grids: (heads of a group, key tiles in increasing order = most
    // query tiles first, head groups)
    bh = causal ? (int)(blockIdx.z * gridDim.x + blockIdx.x) : (int)blockIdx.y;
    it.kb = causal ? (int)blockIdx.y : (int)blockIdx.x;
  }
  if (bh >= a.BH) return false;
  it.sv = seq_view(a.seq, bh, a.status);
  const int N = it.sv.len;  // queries = keys of this sequence
  if (it.kb * BK >= N) return false;
  // query tiles i_begin .. i_end-1: all of them, those at or after the
  // diagonal (causal: the earlier ones see no key of this tile), or this
  // item's range of a split unit
  const int n_q = (N + BQ - 1) / BQ;
  int i_end = n_q;
  it.i_begin = causal ? it.kb : 0;
  if (it.tail_unit >= 0) {  // part < splits <= 4: no overflow
    it.i_begin = it.part * n_q / a.splits;
    i_end = (it.part + 1) * n_q / a.splits;
  }
  it.n_it = i_end - it.i_begin;
  return it.n_it > 0;
}

// The main kernel runs as a persistent grid (a.items > 0): one CTA per SM
// takes items from the list, its first one by block index and, fixed-length
// non-causal (items of one length), every gridDim.x-th after it; causal and
// packed batches, each next one from a device counter (zeroed by the
// preprocess), so the SMs take the items, longest first, as they become
// free.
// The set-up, the TMEM allocation and the CTA turnaround are paid once per SM,
// and the next item's first loads and products overlap this item's last
// tile and epilogue. The rings and the
// per-tile barriers continue across items (global tile index g), the K/V
// tile and the dV/dK accumulators are handed over per item (kv_empty; the
// next item's first dV and dK products come after the epilogue: acc_empty
// from the dQ warps, or the softmax warps' next pt_ready and ds_ready
// arrivals).
// DYN: the causal and packed-batch item lists, taken from the counter and
// published decoded through the item ring; otherwise every role steps
// through the items itself (list: by stride gridDim.x; grid: its one unit),
// and no ring or counter code is compiled in.
template <int D, bool DYN>
__global__ void __launch_bounds__(512, 1) bwd_main_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  // Who writes an item's dV and dK: the dQ warps (the softmax warps go
  // straight on to the next item), except in the counter kernel (DYN) at
  // d = 128, where the softmax warps do (there the dQ warps' register budget
  // spills). Measured both ways; each is the faster one where it is used.
  constexpr bool EPI_DQ = (D == 64) || !DYN;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  if (pad + C::SMEM_BYTES > (uint32_t)C::SMEM_ALLOC) {
    // cannot place the swizzled tiles: report and leave before touching anything
    if (threadIdx.x == 0) report_status(a.status, kStatusTimeout);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  const int B_KV = 0, B_QFULL = 1, B_QEMPTY = 1 + C::QSTAGES, B_DOFULL = 1 + 2 * C::QSTAGES,
            B_DOEMPTY = B_DOFULL + C::DOSTAGES, B_STFULL = B_DOEMPTY + C::DOSTAGES,
            B_STEMPTY = B_STFULL + C::STATSTAGES, B_SFULL = B_STEMPTY + C::STATSTAGES,
            B_DPFULL = B_SFULL + 1, B_PTREADY = B_SFULL + 2, B_DSREADY = B_SFULL + 3,
            B_DSEMPTY = B_SFULL + 4, B_DQFULL = B_SFULL + 5, B_DQEMPTY = B_SFULL + 6,
            B_ACC = B_SFULL + 7, B_DRAIN = B_SFULL + 8, B_KVEMPTY = B_SFULL + 9,
            B_ACCEMPTY = B_SFULL + 10, B_ITF = B_SFULL + 11, B_ITE = B_ITF + C::IRING;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 16);
  auto ring_item = [&](int slot) {
    const volatile int* p = item_ring + 8 * slot;
    BwdItem it;
    it.sv.plane = p[0];
    it.sv.start = p[1];
    it.sv.len = p[2];
    it.kb = p[3];
    it.i_begin = p[4];
    it.n_it = p[5];
    it.tail_unit = p[6];
    it.part = p[7];
    return it;
  };
  const float* stat_smem = reinterpret_cast<const float*>(smem + C::OFF_STAT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool causal = a.seq.causal != 0;
  const bool list = a.items > 0;
  // item indices >= n_items end the walk (a packed batch's total is in its schedule)
  const int n_items = !list ? 1 : (a.seq.cu_seqlens != nullptr ? a.item_counter[1] : a.items);
  if (list && (int)blockIdx.x >= n_items) return;
  if (!list) {
    BwdItem it0;
    if (!bwd_item<C::BK, C::BQ>(a, false, 0, it0)) return;  // no key of a sequence here
  }

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_KV), 1);
    for (int s = 0; s < C::QSTAGES; ++s) {
      mbar_init(BAR(B_QFULL + s), 1);
      mbar_init(BAR(B_QEMPTY + s), 1);
    }
    for (int s = 0; s < C::DOSTAGES; ++s) {
      mbar_init(BAR(B_DOFULL + s), 1);
      mbar_init(BAR(B_DOEMPTY + s), 1);
    }
    for (int s = 0; s < C::STATSTAGES; ++s) {
      mbar_init(BAR(B_STFULL + s), 1);   // the statistics warp's lane 0
      mbar_init(BAR(B_STEMPTY + s), 8);  // one arrival per softmax warp
    }
    mbar_init(BAR(B_SFULL), 1);
    mbar_init(BAR(B_DPFULL), 1);
    mbar_init(BAR(B_PTREADY), 8);  // one arrival per softmax warp (two warpgroups)
    mbar_init(BAR(B_DSREADY), 8);
    mbar_init(BAR(B_DSEMPTY), 1);
    mbar_init(BAR(B_DQFULL), 1);
    mbar_init(BAR(B_DQEMPTY), 4);  // one arrival per dQ warp
    mbar_init(BAR(B_ACC), 1);
    mbar_init(BAR(B_DRAIN), 1);
    mbar_init(BAR(B_KVEMPTY), 1);
    mbar_init(BAR(B_ACCEMPTY), 4);  // one arrival per dQ warp, after its epilogue
    for (int s = 0; s < C::IRING; ++s) {
      mbar_init(BAR(B_ITF + s), 1);   // the producer
      mbar_init(BAR(B_ITE + s), 14);  // one arrival per consuming warp: MMA, statistics, 8 softmax, 4 dQ
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32((const void*)tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The n-th item of this CTA for a consuming warp (warp-uniform), into
  // `it`: 0 an item, 1 the end of the walk, 2 nothing here (skip), -1 the wait
  // ran out (abort raised). DYN: the item the producer decoded and published
  // (its slot is held until release_item(n)); otherwise the n-th of the
  // CTA's stride, decoded here.
  auto get_item = [&](int n, BwdItem& it) -> int {
    if constexpr (DYN) {
      const int slot = n % C::IRING;
      if (!mbar_wait_warp(BAR(B_ITF + slot), (n / C::IRING) & 1, a.status, a.wait_limit_ns)) {
        if (lane == 0) *abort_flag = 1;
        return -1;
      }
      it = ring_item(slot);
      return it.n_it == 0 ? 1 : 0;
    } else {
      const int w = list ? (int)blockIdx.x + n * (int)gridDim.x : n;
      if (w >= n_items) return 1;
      return bwd_item<C::BK, C::BQ>(a, list, w, it) ? 0 : 2;
    }
  };
  // The n-th item again (the epilogues read it again: that keeps the tile
  // loops' registers free).
  auto reload_item = [&](int n, BwdItem& it) {
    if constexpr (DYN) it = ring_item(n % C::IRING);
    else bwd_item<C::BK, C::BQ>(a, list, list ? (int)blockIdx.x + n * (int)gridDim.x : n, it);
  };
  // DYN: this warp is done with the n-th item's ring slot.
  auto release_item = [&](int n) {
    if constexpr (DYN) {
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_ITE + n % C::IRING));
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer: K, V, Q ring
    if (lane == 0) {
      tma_prefetch_desc(&a.tmQ);
      tma_prefetch_desc(&a.tmK);
      tma_prefetch_desc(&a.tmV);
      int last[C::QSTAGES];  // global tile index of the last load into each slot
#pragma unroll
      for (int s = 0; s < C::QSTAGES; ++s) last[s] = -1;
      int ui = 0, g0 = 0;  // items and query tiles before this item
      bool ok = true;
      int w = list ? (int)blockIdx.x : 0;
      // The item after this one: DYN (items of different lengths: causal,
      // packed batches) from the counter, taken once this item's last Q load
      // is issued (a few tiles before it ends: an earlier claim would hold a
      // long item's successor back while other SMs run dry); the others (all
      // of one length) by stride.
      auto take_next = [&]() {
        int wn = n_items;
        if constexpr (DYN) {
          const int c = atomicAdd(a.item_counter, 1);
          wn = c >= 0 && c < n_items ? (int)gridDim.x + c : n_items;
        } else {
          if (list) wn = w + (int)gridDim.x;
        }
        return wn;
      };
      for (int n = 0; ok; ++n) {
        // the item, past any with nothing to do (heads padding the last
        // causal head group)
        BwdItem it{};
        bool end = false;
        for (;;) {
          if (w >= n_items) { end = true; break; }
          if (bwd_item<C::BK, C::BQ>(a, list, w, it)) break;
          w = take_next();
        }
        if constexpr (DYN) {
          // publish the decoded item (n_it = 0: the end of the walk)
          const int slot = n % C::IRING;
          if (n >= C::IRING &&
              !mbar_wait(BAR(B_ITE + slot), ((n / C::IRING) - 1) & 1, a.status, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          volatile int* p = item_ring + 8 * slot;
          p[0] = it.sv.plane;
          p[1] = it.sv.start;
          p[2] = it.sv.len;
          p[3] = it.kb;
          p[4] = it.i_begin;
          p[5] = end ? 0 : it.n_it;
          p[6] = it.tail_unit;
          p[7] = it.part;
          mbar_arrive(BAR(B_ITF + slot));
        }
        if (end) break;
        const int plane = it.sv.plane, qrow0 = it.sv.start + it.i_begin * C::BQ;
        auto load_q = [&](int i) {  // query tile i_begin + i into its ring slot
          const int g = g0 + i;
          const int s = g % C::QSTAGES;
          if (!mbar_wait(BAR(B_QEMPTY + s), ((g / C::QSTAGES) & 1) ^ 1, a.status, a.wait_limit_ns)) return false;
          if (g != a.debug_skip_q) {
            mbar_arrive_expect_tx(BAR(B_QFULL + s), C::TILE);
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(sbase + C::OFF_Q + s * C::TILE + c * C::ROW_CHUNK, &a.tmQ, BAR(B_QFULL + s),
                          c * 64, qrow0 + i * C::BQ, plane);
            last[s] = g;
          }
          return true;
        };
        int i = 0;
        if (ui > 0) {
          // The slots of this item's first QSTAGES-1 query tiles were
          // released by dK products issued before the previous item's last
          // dQ, so they load ahead of K and V, which wait for that dQ.
          for (; ok && i < it.n_it && i < C::QSTAGES - 1; ++i) ok = *abort_flag == 0 && load_q(i);
          ok = ok && mbar_wait(BAR(B_KVEMPTY), (ui - 1) & 1, a.status, a.wait_limit_ns);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(B_KV), 2 * C::TILE);
        for (int c = 0; c < C::CH; ++c) {
          tma_load_3d(sbase + C::OFF_K + c * C::ROW_CHUNK, &a.tmK, BAR(B_KV), c * 64,
                      it.sv.start + it.kb * C::BK, plane);
          tma_load_3d(sbase + C::OFF_V + c * C::ROW_CHUNK, &a.tmV, BAR(B_KV), c * 64,
                      it.sv.start + it.kb * C::BK, plane);
        }
        ++ui;
        for (; ok && i < it.n_it; ++i) ok = *abort_flag == 0 && load_q(i);
        g0 += it.n_it;
        const int w_next = take_next();
        if (ok && w_next < n_items) {
          // the next item's K and V into L2 now, a few tiles before this
          // item's last dQ releases the buffer they load into
          BwdItem nx;
          if (bwd_item<C::BK, C::BQ>(a, list, w_next, nx))
            for (int c = 0; c < C::CH; ++c) {
              tma_prefetch_l2_3d(&a.tmK, c * 64, nx.sv.start + nx.kb * C::BK, nx.sv.plane);
              tma_prefetch_l2_3d(&a.tmV, c * 64, nx.sv.start + nx.kb * C::BK, nx.sv.plane);
            }
        }
        w = w_next;
      }
      if (!ok) *abort_flag = 1;
      // drain: the last load issued into each buffer must have landed before exit
      if (ui > 0) mbar_wait(BAR(B_KV), (ui - 1) & 1, a.status, a.wait_limit_ns);
#pragma unroll
      for (int s = 0; s < C::QSTAGES; ++s)
        if (last[s] >= 0) mbar_wait(BAR(B_QFULL + s), (last[s] / C::QSTAGES) & 1, a.status, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ producer: stats, dO ring
    // Each query tile's two statistics rows: with the fixed-length layout one
    // bulk copy each (rows past N hold the neutral padding); in a packed
    // batch, where a sequence may start at any row and the tile's last rows
    // may belong to the next sequence, the whole warp copies them with plain
    // loads (lane k: rows 4k..4k+3) and sets -LSE*log2e = -inf past the
    // sequence, so that P = 0 there. Lane 0 issues the dO tile loads.
    const bool stat_bulk = a.seq.cu_seqlens == nullptr;  // rows 16-byte aligned, padded
    if (lane == 0) tma_prefetch_desc(&a.tmdO);
    int last = -1;       // lane 0: global tile index of the last dO tile issued
    int last_stat = -1;  // lane 0: last statistics tile issued by bulk copies
    int g0 = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      BwdItem it;
      const int got = get_item(n, it);
      if (got < 0) { ok = false; break; }
      if (got == 1) break;
      if (got == 2) continue;
      const int N = it.sv.len, plane = it.sv.plane;
      const size_t ws_row0 = (size_t)plane * a.ws_rows + (size_t)it.sv.start;  // workspace row of query 0
      for (int i = 0; i < it.n_it; ++i) {
        const int g = g0 + i;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        const int q_row = (it.i_begin + i) * C::BQ;  // first query row of the tile, within the sequence
        {
          const int t = g % C::STATSTAGES;
          const uint32_t pt = (g / C::STATSTAGES) & 1;
          if (!mbar_wait_warp(BAR(B_STEMPTY + t), pt ^ 1, a.status, a.wait_limit_ns)) {
            if (lane == 0) *abort_flag = 1;
            ok = false;
            break;
          }
          if (stat_bulk) {
            if (lane == 0) {
              mbar_arrive_expect_tx(BAR(B_STFULL + t), C::STAT_BYTES);
              bulk_load(sbase + C::OFF_STAT + t * C::STAT_BYTES, a.lse2 + ws_row0 + q_row, C::BQ * 4,
                        BAR(B_STFULL + t));
              bulk_load(sbase + C::OFF_STAT + t * C::STAT_BYTES + C::BQ * 4, a.Drow + ws_row0 + q_row,
                        C::BQ * 4, BAR(B_STFULL + t));
              last_stat = g;
            }
          } else {
            const size_t row0 = ws_row0 + (size_t)q_row + 4 * lane;
            const int live = N - q_row - 4 * lane;  // rows of this lane inside the sequence
            float* dst = reinterpret_cast<float*>(smem + C::OFF_STAT + t * C::STAT_BYTES) + 4 * lane;
            const float4 l4 = make_float4(live > 0 ? a.lse2[row0] : -INFINITY,
                                          live > 1 ? a.lse2[row0 + 1] : -INFINITY,
                                          live > 2 ? a.lse2[row0 + 2] : -INFINITY,
                                          live > 3 ? a.lse2[row0 + 3] : -INFINITY);
            const float4 d4 = make_float4(a.Drow[row0], a.Drow[row0 + 1], a.Drow[row0 + 2], a.Drow[row0 + 3]);
            *reinterpret_cast<float4*>(dst) = l4;
            *reinterpret_cast<float4*>(dst + C::BQ) = d4;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_STFULL + t));
          }
        }
        if (lane == 0) {
          const int s = g % C::DOSTAGES;
          const uint32_t ph = (g / C::DOSTAGES) & 1;
          if (!mbar_wait(BAR(B_DOEMPTY + s), ph ^ 1, a.status, a.wait_limit_ns)) {
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(BAR(B_DOFULL + s), C::TILE);
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(sbase + C::OFF_DO + s * C::TILE + c * C::ROW_CHUNK, &a.tmdO,
                          BAR(B_DOFULL + s), c * 64, it.sv.start + q_row, plane);
            last = g;
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      g0 += it.n_it;
      release_item(n);
    }
    if (lane == 0) {
      // the last dO and statistics copies issued into each slot must have
      // landed before exit (after an abort nobody else waits for them)
      for (int i = last - C::DOSTAGES + 1 < 0 ? 0 : last - C::DOSTAGES + 1; i <= last; ++i)
        mbar_wait(BAR(B_DOFULL + i % C::DOSTAGES), (i / C::DOSTAGES) & 1, a.status, a.wait_limit_ns);
      for (int i = last_stat - C::STATSTAGES + 1 < 0 ? 0 : last_stat - C::STATSTAGES + 1; i <= last_stat; ++i)
        mbar_wait(BAR(B_STFULL + i % C::STATSTAGES), (i / C::STATSTAGES) & 1, a.status, a.wait_limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged (waits, descriptor arithmetic);
    // tcgen05.mma and tcgen05.commit are issued by the one elected lane.
    {
      const uint32_t leader = elect_one();
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait_warp(BAR(b), parity, a.status, a.wait_limit_ns);
      };
      constexpr uint32_t id_s = idesc_bf16_f32(128, C::BQ, false, false);  // S^T, dP^T
      constexpr uint32_t id_dv = idesc_bf16_f32(128, D, false, true);      // dV (A from TMEM)
      constexpr uint32_t id_dk = idesc_bf16_f32(128, D, false, true);      // dK
      constexpr uint32_t id_dq = C::DQ_T ? idesc_bf16_f32(128, C::BQ, true, true)  // dQ^T = K^T dS^T
                                         : idesc_bf16_f32(128, D, true, true);    // dQ = dS K
      // descriptors built once; K-steps only add byte offsets >> 4
      const uint64_t dKk = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t dKmn = sdesc_sw128(sbase + C::OFF_K, C::ROW_CHUNK, 1024);
      const uint64_t dVk = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      const uint64_t dQk = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dQmn = sdesc_sw128(sbase + C::OFF_Q, C::ROW_CHUNK, 1024);
      const uint64_t dOk = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
      const uint64_t dOmn = sdesc_sw128(sbase + C::OFF_DO, C::ROW_CHUNK, 1024);
      const uint64_t dSk = sdesc_sw128(sbase + C::OFF_DS, 16, 1024);
      const uint64_t dSmn = sdesc_sw128(sbase + C::OFF_DS, C::ROW_CHUNK, 1024);
      const auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * C::ROW_CHUNK + (kk & 3) * 32) >> 4); };
      const auto roff = [](int kk) { return (uint64_t)((kk * 2048) >> 4); };  // 16 rows of 128 B
      const auto soff = [](int s) { return (uint64_t)((s * C::TILE) >> 4); };  // ring slot s
      // S^T = K Q_i^T, dP^T = V dO_i^T (K-dimension = d)
      auto issue_s = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::COL_S, dKk + koff(kk), dQk + soff(s) + koff(kk), id_s, kk > 0, leader);
      };
      auto issue_dp = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::COL_DP, dVk + koff(kk), dOk + soff(s) + koff(kk), id_s, kk > 0, leader);
      };
      // dV += P^T dO_i (P^T from TMEM), dK += dS^T Q_i (K-dimension = queries)
      auto issue_dv = [&](int s, bool acc) {
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          // P^T of queries 16kk..16kk+15: packed bf16 in the S^T columns of the
          // softmax warpgroup that owns them (64 queries per group)
          mma_ts(tmem + C::COL_DV, tmem + C::COL_S + 64 * (kk >> 2) + 8 * (kk & 3), dOmn + soff(s) + roff(kk), id_dv,
                 (acc || kk > 0) ? 1u : 0u, leader);
      };
      auto issue_dk = [&](int s, bool acc) {
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          mma_ss(tmem + C::COL_DK, dSk + koff(kk), dQmn + soff(s) + roff(kk), id_dk,
                 (acc || kk > 0) ? 1u : 0u, leader);
      };
      // dQ_i (K-dimension = keys), into the dP^T columns; both operands MN-major
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          if (C::DQ_T) mma_ss(tmem + C::COL_DP, dKmn + roff(kk), dSmn + roff(kk), id_dq, kk > 0, leader);
          else mma_ss(tmem + C::COL_DP, dSmn + roff(kk), dKmn + roff(kk), id_dq, kk > 0, leader);
        }
      };
      bool ok = true;
      int ui = 0, g0 = 0;  // items and query tiles before this item
      for (int n = 0; ok; ++n) {
        BwdItem it;
        const int got = get_item(n, it);
        if (got < 0) { ok = false; break; }
        if (got == 1) break;
        if (got == 2) continue;
        const int n_it = it.n_it;
        {
          // the item's first S^T and dP^T (S^T overwrites P^T of the previous
          // item's last tile: ordered after the dV products that read it)
          const int s = g0 % C::QSTAGES, so = g0 % C::DOSTAGES;
          ok = wait(B_KV, ui & 1) && wait(B_QFULL + s, (g0 / C::QSTAGES) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(s);
          mma_commit(BAR(B_SFULL), leader);
          // dP^T reuses the dQ columns once the dQ warps have read the
          // previous tile's dQ
          ok = (g0 == 0 || wait(B_DQEMPTY, (g0 - 1) & 1)) && wait(B_DOFULL + so, (g0 / C::DOSTAGES) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_dp(so);
          mma_commit(BAR(B_DPFULL), leader);
        }
        for (int i = 0; i < n_it; ++i) {  // i: iteration; query tile i_begin + i; g: ring position
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          const int g = g0 + i;
          const int s = g % C::QSTAGES, so = g % C::DOSTAGES;
          const bool more = i + 1 < n_it;
          const int s1 = (g + 1) % C::QSTAGES, so1 = (g + 1) % C::DOSTAGES;
          const uint32_t ph1 = ((g + 1) / C::QSTAGES) & 1, pho1 = ((g + 1) / C::DOSTAGES) & 1;
          if (!wait(B_PTREADY, g & 1)) { ok = false; break; }
          // the first dV (and dK) product of a later item overwrites the
          // accumulators once the dQ warps have written the previous item's
          // (softmax-warp epilogue: their pt_ready arrivals follow it)
          if (EPI_DQ && i == 0 && ui > 0 && !wait(B_ACCEMPTY, (ui - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_dv(so, i > 0);
          mma_commit(BAR(B_DOEMPTY + so), leader);  // dO_i: last use was dV
          if (more) {
            if (!wait(B_QFULL + s1, ph1)) { ok = false; break; }
            tc_fence_after();
            issue_s(s1);  // overwrites P^T(i): ordered after the dV products that read it
            mma_commit(BAR(B_SFULL), leader);
          }
          if (!wait(B_DSREADY, g & 1)) { ok = false; break; }
          tc_fence_after();
          issue_dq();  // the dP^T columns: dP^T(i) was consumed before ds_ready
          mma_commit(BAR(B_DQFULL), leader);
          if (!more) mma_commit(BAR(B_KVEMPTY), leader);  // K, V: last uses were dQ and dP^T of this tile
          issue_dk(s, i > 0);
          mma_commit(BAR(B_QEMPTY + s), leader);  // Q_i: last use was dK
          mma_commit(BAR(B_DSEMPTY), leader);     // dS^T(i): last use was dQ/dK
          if (more) {
            // dP^T(i+1) reuses the dQ columns once the dQ warps have read dQ(i)
            if (!wait(B_DQEMPTY, g & 1) ||
                !wait(B_DOFULL + so1, pho1)) { ok = false; break; }
            tc_fence_after();
            issue_dp(so1);
            mma_commit(BAR(B_DPFULL), leader);
          }
        }
        if (!ok) break;
        mma_commit(BAR(B_ACC), leader);  // the item's dV and dK are complete
        g0 += n_it;
        ++ui;
        release_item(n);
      }
      if (!ok && lane == 0) *abort_flag = 1;
      mma_commit(BAR(B_DRAIN), leader);
      wait(B_DRAIN, 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax: P^T, dS^T
    // Two warpgroups; warpgroup g handles query columns [64g, 64g + 64) of
    // every key row (thread = key row = TMEM lane).
    const int g = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row within the tile == TMEM lane
    const int qc0 = 64 * g;  // first query column of this group
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    const uint64_t c22 = f2_pack(a.scale_log2, a.scale_log2);
    uint8_t* dsrow = smem + C::OFF_DS + g * C::ROW_CHUNK + r * 128;  // this group's dS^T chunk
    bool ok = true;
    int ui = 0, g0 = 0;  // items and query tiles before this item
    for (int n = 0; ok; ++n) {
      int n_it, diag_i;
      bool key_live;
      {
        BwdItem it;
        const int got = get_item(n, it);
        if (got < 0) { ok = false; break; }
        if (got == 1) break;
        if (got == 2) continue;
        n_it = it.n_it;
        diag_i = causal ? it.kb - it.i_begin : -1;  // iteration of the diagonal tile
        key_live = it.kb * C::BK + r < it.sv.len;
      }
      for (int i = 0; i < n_it; ++i) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        const int gt = g0 + i;  // ring position of the tile
        const int st = gt % C::STATSTAGES;
        // On the causal diagonal, P = 0 in the columns q < r (key r after query
        // q): column 32h + 4k4 + e of this group is masked when it is below
        // r - 64g. (Queries past the sequence have -LSE*log2e = -inf: P = 0.)
        const bool diag = i == diag_i;
        const int r_rel = r - qc0;
        bool w_ok = mbar_wait(BAR(B_SFULL), gt & 1, a.status, a.wait_limit_ns) &&
                    mbar_wait(BAR(B_STFULL + st), (gt / C::STATSTAGES) & 1, a.status, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        tc_fence_after();
        const float* lse2 = stat_smem + st * (C::STAT_BYTES / 4) + 64 * g;
        const float* drow = stat_smem + st * (C::STAT_BYTES / 4) + C::BQ + 64 * g;
        // phase 1: P^T = 2^(S^T * scale*log2e - LSE*log2e), bf16, written over
        // this group's S^T columns (64 queries -> packed columns 64g..64g+31)
        // for the dV products; phase 2 takes the fp32 values, kept in
        // registers (no unpacking, and dS from P before its rounding)
        uint64_t pf[32];  // P of the 64 query columns as fp32 pairs
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t sr[32];
          tmem_ld32(lane_addr + C::COL_S + 64 * g + 32 * h, sr);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            // nl = -LSE*log2e of four query columns
            const float4 nl = *reinterpret_cast<const float4*>(lse2 + 32 * h + 4 * k4);
            const float2 xa = f2_unpack(ffma2(f2_pack(__uint_as_float(sr[4 * k4]), __uint_as_float(sr[4 * k4 + 1])), c22, f2_pack(nl.x, nl.y)));
            const float2 xb = f2_unpack(ffma2(f2_pack(__uint_as_float(sr[4 * k4 + 2]), __uint_as_float(sr[4 * k4 + 3])), c22, f2_pack(nl.z, nl.w)));
            float p0 = ex2_approx(xa.x), p1 = ex2_approx(xa.y), p2 = ex2_approx(xb.x), p3 = ex2_approx(xb.y);
            if (!key_live) p0 = p1 = p2 = p3 = 0.f;
            if (diag) {
              const int c = 32 * h + 4 * k4;
              p0 = c < r_rel ? 0.f : p0;
              p1 = c + 1 < r_rel ? 0.f : p1;
              p2 = c + 2 < r_rel ? 0.f : p2;
              p3 = c + 3 < r_rel ? 0.f : p3;
            }
            pf[16 * h + 2 * k4] = f2_pack(p0, p1);
            pf[16 * h + 2 * k4 + 1] = f2_pack(p2, p3);
            pk[2 * k4] = pack_bf16x2(p0, p1);
            pk[2 * k4 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st16(lane_addr + C::COL_S + 64 * g + 16 * h, pk);
        }
        // P^T of this group's 64 queries goes to the first 32 of its own S^T
        // columns (64g .. 64g+31), so neither group overwrites scores the
        // other has not read yet; the dV products take their A slices there.
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_PTREADY));
        // phase 2: dS'^T = P^T o (dP^T - D), bf16, into this group's swizzled
        // [128 keys][64 queries] chunk of the dS^T tile (16-byte unit c of row r
        // lands at unit c ^ (r & 7))
        w_ok = mbar_wait(BAR(B_DPFULL), gt & 1, a.status, a.wait_limit_ns) &&
               mbar_wait(BAR(B_DSEMPTY), (gt & 1) ^ 1, a.status, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dr[32];
          tmem_ld32(lane_addr + C::COL_DP + 64 * g + 32 * h, dr);
          tmem_ld_wait();
          uint32_t dk[16];
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            // nd = -D of four query columns; dS' = P * (dP - D). The softmax
            // scale of dS is applied once to dK (epilogue) and dQ (convert).
            const float4 nd = *reinterpret_cast<const float4*>(drow + 32 * h + 4 * k4);
            const uint64_t ta = fadd2(f2_pack(__uint_as_float(dr[4 * k4]), __uint_as_float(dr[4 * k4 + 1])), f2_pack(nd.x, nd.y));
            const uint64_t tb = fadd2(f2_pack(__uint_as_float(dr[4 * k4 + 2]), __uint_as_float(dr[4 * k4 + 3])), f2_pack(nd.z, nd.w));
            const float2 ga = f2_unpack(fmul2(pf[16 * h + 2 * k4], ta));
            const float2 gb = f2_unpack(fmul2(pf[16 * h + 2 * k4 + 1], tb));
            dk[2 * k4] = pack_bf16x2(ga.x, ga.y);
            dk[2 * k4 + 1] = pack_bf16x2(gb.x, gb.y);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = h * 4 + u;
            *reinterpret_cast<uint4*>(dsrow + ((c ^ (r & 7)) * 16)) =
                make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(B_DSREADY));
          mbar_arrive(BAR(B_STEMPTY + st));  // this tile's LSE/D are no longer read
        }
      }
      if (!ok) break;
      if constexpr (!EPI_DQ) {
        // epilogue: group 0 writes dV, group 1 writes dK (which carries the
        // softmax scale of dS); a query range of a split unit leaves its fp32
        // partial sums (dK unscaled) for the dQ-convert stage to add up. The
        // next item's first dV (dK) product overwrites these columns only
        // after this warp's next pt_ready (ds_ready) arrival.
        {
          const bool w_ok = mbar_wait(BAR(B_ACC), ui & 1, a.status, a.wait_limit_ns);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
        }
        tc_fence_after();
        BwdItem it;  // read again: keeps the tile loop's registers free
        reload_item(n, it);
        const int k0 = it.kb * C::BK;
        const uint32_t col = g == 0 ? C::COL_DV : C::COL_DK;
        if (it.tail_unit >= 0) {
          float* prow = a.dKVpart + ((size_t)(it.tail_unit * a.splits + it.part) * 2 + g) * (size_t)C::BK * D +
                        (size_t)r * D;
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_addr + col + 32 * q, v);
            tmem_ld_wait();
            if (key_live) {
              float4* d4 = reinterpret_cast<float4*>(prow + 32 * q);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                d4[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            }
          }
        } else {
          // The warp stages its 32 rows, 64 columns (128 bytes of bf16) at a
          // time, in its own rows of the group's dS^T chunk (free here: the
          // item's dK and dQ products, its readers, are complete, and the
          // group writes it again only in its next phase 2), in the 128-byte
          // swizzle. Fixed length: one TMA tensor store of the 32 x 64 box
          // (rows past N are clipped); packed batches read the rows back so
          // that each store instruction writes 4 whole 128-byte rows of this
          // sequence instead of 16 bytes of 32 rows.
          const bool tma_out = a.seq.cu_seqlens == nullptr;
          const float f = g == 0 ? 1.f : a.scale;
          __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(g == 0 ? a.dV : a.dK);
          uint8_t* stg = smem + C::OFF_DS + g * C::ROW_CHUNK + wq * 32 * 128;  // [32 rows][128 B]
          const int rsub = lane >> 3, unit = lane & 7;  // read-back: row 4j + rsub, 16-byte unit
#pragma unroll 1
          for (int hc = 0; hc < D / 64; ++hc) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t v[32];
              tmem_ld32(lane_addr + col + 64 * hc + 32 * hh, v);
              tmem_ld_wait();
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(dsrow + (((4 * hh + u) ^ (lane & 7)) << 4)) =
                    make_uint4(pack_bf16x2(f * __uint_as_float(v[8 * u]), f * __uint_as_float(v[8 * u + 1])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 2]), f * __uint_as_float(v[8 * u + 3])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 4]), f * __uint_as_float(v[8 * u + 5])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 6]), f * __uint_as_float(v[8 * u + 7])));
            }
            if (tma_out) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(g == 0 ? &a.tmdV : &a.tmdK, smem_u32(stg), 64 * hc, it.sv.start + k0 + wq * 32,
                             it.sv.plane);
                bulk_commit_group();
                bulk_wait_group_read<0>();  // the rows are read before the next pass (or phase 2) writes them
              }
              __syncwarp();
            } else {
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int rr = 4 * j + rsub;  // row within the warp's 32
                const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((unit ^ (rr & 7)) << 4));
                const int key = k0 + wq * 32 + rr;
                if (key < it.sv.len)
                  *reinterpret_cast<uint4*>(base + seq_row_offset(a.seq, it.sv, key) + 64 * hc + 8 * unit) = x;
              }
              __syncwarp();  // the rows are read before the next pass (or phase 2) writes them
            }
          }
        }
      }
      ++ui;
      g0 += n_it;
      release_item(n);
    }
    if (!ok) *abort_flag = 1;
    if (lane == 0) bulk_wait_group_all();  // the epilogue's tensor stores have completed
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ reduction
    const int wq = warp & 3;  // TMEM lanes 32wq..32wq+31: d indices (dQ^T) or query rows (dQ)
    const uint32_t lane_addr = tmem + ((uint32_t)(wq * 32) << 16);
    constexpr int NCOL = C::DQ_T ? C::BQ : D;  // columns of the dQ tile
    constexpr int HALF = NCOL / 2;             // read in two halves (register budget)
    uint8_t* wstage = smem + C::OFF_DQS + wq * 2 * C::DQ_BLOCK_BYTES;
    int nblk = 0;  // staging blocks issued so far by this warp
    int ui = 0, g0 = 0;  // items and query tiles before this item
    bool ok = true;
    for (int n = 0; ok; ++n) {
      size_t row_first;  // workspace row of the item's first query tile
      int n_it;
      {
        BwdItem it;
        const int got = get_item(n, it);
        if (got < 0) { ok = false; break; }
        if (got == 1) break;
        if (got == 2) continue;
        row_first = (size_t)it.sv.plane * a.ws_rows + (size_t)it.sv.start + (size_t)it.i_begin * C::BQ;
        n_it = it.n_it;
      }
      for (int i = 0; i < n_it; ++i) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        const bool w_ok = mbar_wait(BAR(B_DQFULL), (g0 + i) & 1, a.status, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { *abort_flag = 1; ok = false; break; }
        tc_fence_after();
        // rows past the sequence receive exact zeros (their P is 0)
        const size_t row0 = row_first + (size_t)i * C::BQ;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[HALF];
#pragma unroll
          for (int q = 0; q < HALF / 32; ++q)
            tmem_ld32(lane_addr + C::COL_DP + HALF * hh + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * q]));
          tmem_ld_wait();
          if (hh == 1) {
            // all of dQ(i) is in registers: the MMA warp may reuse the columns
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_DQEMPTY));
          }
          if (C::DQ_T) {
            // lane t holds dQ[row0 + q][t] for this half's queries. Each warp
            // stages its 32 d-columns of 32 query rows at a time ([row][32 d]
            // fp32, 4 KB) and lets the TMA engine add the block into the
            // accumulator; two buffers per warp, tracked by the warp's lane 0.
#pragma unroll
            for (int c = 0; c < HALF / C::DQ_ROWS; ++c, ++nblk) {
              const int buf = nblk & 1;
              if (lane == 0) bulk_wait_group_read<1>();  // the reduction that last read buf is done
              __syncwarp();
              float* stage = reinterpret_cast<float*>(wstage + buf * C::DQ_BLOCK_BYTES);
#pragma unroll
              for (int q = 0; q < C::DQ_ROWS; ++q) stage[q * 32 + lane] = __uint_as_float(v[C::DQ_ROWS * c + q]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_reduce_add_2d(&a.tmDQacc, smem_u32(stage), wq * 32,
                                  (int)(row0 + (size_t)HALF * hh + (size_t)C::DQ_ROWS * c));
                bulk_commit_group();
              }
            }
          } else {
            // lane t holds this half (32 columns) of the dQ row of query
            // row0 + t. The warp stages its 32 rows x 32 columns as [row][32]
            // fp32 in the TMA 128-byte swizzle (16-byte unit k of row r at unit
            // k ^ (r % 8): the float4 stores of the 32 lanes hit every bank
            // equally) and lets the TMA engine add the block into the
            // accumulator; two buffers per warp, tracked by the warp's lane 0.
            const int buf = nblk & 1;
            if (lane == 0) bulk_wait_group_read<1>();  // the reduction that last read buf is done
            __syncwarp();
            uint8_t* stage = wstage + buf * C::DQ_BLOCK_BYTES;
#pragma unroll
            for (int k = 0; k < HALF / 4; ++k)
              *reinterpret_cast<float4*>(stage + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                  make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                              __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&a.tmDQacc, smem_u32(stage), HALF * hh, (int)(row0 + (size_t)wq * 32));
              bulk_commit_group();
            }
            ++nblk;
          }
        }
      }
      if (!ok) break;
      if constexpr (EPI_DQ) {
      // epilogue of the item: dV, then dK (which carries the softmax scale
      // of dS), one key row per thread (TMEM lane 32wq + lane); a query
      // range of a split unit leaves its fp32 partial sums (dK unscaled) for
      // the dQ-convert stage to add up
      {
        const bool w_ok = mbar_wait(BAR(B_ACC), ui & 1, a.status, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, w_ok)) { *abort_flag = 1; ok = false; break; }
      }
      tc_fence_after();
      BwdItem it;  // read again: keeps the tile loop's registers free
      reload_item(n, it);
      const int r = wq * 32 + lane;
      const int k0 = it.kb * C::BK;
      if (it.tail_unit >= 0) {
        const bool key_live = k0 + r < it.sv.len;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          float* prow = a.dKVpart + ((size_t)(it.tail_unit * a.splits + it.part) * 2 + g) * (size_t)C::BK * D +
                        (size_t)r * D;
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            tmem_ld32(lane_addr + (g == 0 ? C::COL_DV : C::COL_DK) + 32 * q, v);
            tmem_ld_wait();
            if (key_live) {
              float4* d4 = reinterpret_cast<float4*>(prow + 32 * q);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                d4[u] = make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
            }
          }
        }
      } else {
        // The warp stages its 32 rows, 64 columns (128 bytes of bf16) at a
        // time, in its dQ staging buffers (free once its reductions have read
        // them; dV in the first, dK in the second) in the 128-byte swizzle.
        // Fixed length: one TMA tensor store per 32 x 64 box (rows past N
        // are clipped); packed batches read the rows back so that each store
        // instruction writes 4 whole 128-byte rows of this sequence instead
        // of 16 bytes of 32 rows.
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        const bool tma_out = a.seq.cu_seqlens == nullptr;
        const int rsub = lane >> 3, unit = lane & 7;  // read-back: row 4j + rsub, 16-byte unit
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint8_t* stg = wstage + g * C::DQ_BLOCK_BYTES;  // [32 rows][128 B]
          const uint32_t col = g == 0 ? C::COL_DV : C::COL_DK;
          const float f = g == 0 ? 1.f : a.scale;
          __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(g == 0 ? a.dV : a.dK);
#pragma unroll 1
          for (int hc = 0; hc < D / 64; ++hc) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t v[32];
              tmem_ld32(lane_addr + col + 64 * hc + 32 * hh, v);
              tmem_ld_wait();
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(stg + lane * 128 + (((4 * hh + u) ^ (lane & 7)) << 4)) =
                    make_uint4(pack_bf16x2(f * __uint_as_float(v[8 * u]), f * __uint_as_float(v[8 * u + 1])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 2]), f * __uint_as_float(v[8 * u + 3])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 4]), f * __uint_as_float(v[8 * u + 5])),
                               pack_bf16x2(f * __uint_as_float(v[8 * u + 6]), f * __uint_as_float(v[8 * u + 7])));
            }
            if (tma_out) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(g == 0 ? &a.tmdV : &a.tmdK, smem_u32(stg), 64 * hc, it.sv.start + k0 + wq * 32,
                             it.sv.plane);
                bulk_commit_group();
                if (hc + 1 < D / 64) bulk_wait_group_read<0>();  // the buffer takes the next pass
              }
              __syncwarp();
            } else {
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int rr = 4 * j + rsub;  // row within the warp's 32
                const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((unit ^ (rr & 7)) << 4));
                const int key = k0 + wq * 32 + rr;
                if (key < it.sv.len)
                  *reinterpret_cast<uint4*>(base + seq_row_offset(a.seq, it.sv, key) + 64 * hc + 8 * unit) = x;
              }
              __syncwarp();  // the rows are read before the next pass writes them
            }
          }
        }
        // the staging buffers take dQ blocks again only after these stores read them
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      }
      // dV and dK have left TMEM: the next item may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_ACCEMPTY));
      }
      ++ui;
      g0 += n_it;
      release_item(n);
    }
    // every bulk reduction must have read its staging block before the CTA
    // exits; the additions land before the kernel ends
    if (lane == 0) bulk_wait_group_read<0>();
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
  cudaError_t e = cudaSuccess;
  if (stages & kStagePre) {
    constexpr int RPW = 32 / (D / 8);
    const long long rows = (long long)a.planes * a.ws_rows;
    const long long warps = (rows + RPW - 1) / RPW;
    const long long blocks = (warps * 32 + 255) / 256 + (a.nseq > 0 ? 1 : 0);  // + the schedule block
    bwd_pre_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kStageMain) {
    const bool dyn = a.items > 0 && (a.seq.causal || a.seq.cu_seqlens != nullptr);
    e = cudaFuncSetAttribute(dyn ? bwd_main_kernel<D, true> : bwd_main_kernel<D, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const unsigned kblocks = (unsigned)((a.seq.N + C::BK - 1) / C::BK);
    dim3 grid(kblocks, (unsigned)BH);
    if (a.items > 0) {
      // persistent grid over the item list: one CTA per SM (each holds all of
      // TMEM and most of shared memory)
      if (a.item_counter == nullptr) return cudaErrorInvalidValue;
      if (a.seq.cu_seqlens) {
        if (a.nseq < 1 || a.splits != 1 || (long long)a.items != (long long)BH * kblocks)
          return cudaErrorInvalidValue;
      } else if (a.seq.causal) {
        const int hpg = causal_heads_per_group(BH, 8ll * a.seq.N * D, 48ll << 20);
        if (a.splits != 1 || a.causal_hpg != hpg ||
            (long long)a.items != (long long)hpg * kblocks * ((BH + hpg - 1) / hpg))
          return cudaErrorInvalidValue;
      } else if (a.splits < 1 || a.n_tail < 0 || (long long)a.n_full + a.n_tail != (long long)kblocks * BH ||
                 (long long)a.items != (long long)a.n_full + (long long)a.n_tail * a.splits ||
                 (a.splits > 1 && (a.dKVpart == nullptr || a.n_tail < 1))) {
        return cudaErrorInvalidValue;
      }
      const int sms = fwd_slots();
      grid = dim3((unsigned)(sms > 0 && sms < a.items ? sms : a.items));
    } else if (a.splits > 1) {
      return cudaErrorInvalidValue;  // a split tail runs only as an item list
    } else if (a.seq.causal) {
      // every CTA of a head streams the head's Q and dO and adds into its dQ accumulator
      const int hpg = causal_heads_per_group(BH, 8ll * a.seq.N * D, 48ll << 20);
      grid = dim3((unsigned)hpg, kblocks, (unsigned)((BH + hpg - 1) / hpg));
    }
    if (dyn) bwd_main_kernel<D, true><<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(a);
    else bwd_main_kernel<D, false><<<grid, C::THREADS, C::SMEM_ALLOC, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kStageConvert) {
    const long long groups = (long long)a.planes * a.seq.total * (D / 8);
    const unsigned conv_blocks = (unsigned)((groups + 255) / 256);
    // plus one warp per key row of a split unit (8 rows per block)
    const unsigned merge_blocks = a.splits > 1 ? (unsigned)(((long long)a.n_tail * 128 + 7) / 8) : 0u;
    dq_convert_kernel<D><<<conv_blocks + merge_blocks, 256, 0, st>>>(a, conv_blocks);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

BwdTailPlan plan_bwd_tail(long long units, int n_q, int slots) {
  BwdTailPlan p{(int)units, 0, 1};
  if (units < 1 || slots < 1 || n_q < 1) return p;
  const long long rem = units % slots;
  if (units < slots || rem == 0) return p;  // no whole wave before the tail, or no tail
  long long sp = slots / rem;
  if (sp > 4) sp = 4;
  if (sp > n_q / 4) sp = n_q / 4;
  if (sp < 2) return p;
  p.n_full = (int)(units - rem);
  p.n_tail = (int)rem;
  p.splits = (int)sp;
  return p;
}

size_t bwd_tail_part_bytes(const BwdTailPlan& p, int d) {
  if (p.splits <= 1 || p.n_tail <= 0) return 0;
  return ((size_t)p.n_tail * p.splits * 2 * 128 * d * 4 + 255) & ~(size_t)255;
}

cudaError_t launch_bwd_bf16(const BwdArgs& a, int BH, int d, unsigned stages, cudaStream_t st) {
  if (d == 128) return launch_bwd_d<128>(a, BH, stages, st);
  if (d == 64) return launch_bwd_d<64>(a, BH, stages, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
