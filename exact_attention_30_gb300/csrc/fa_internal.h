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

// Where the rows of each (batch, head) live and which keys a query row sees.
//  * fixed length (cu_seqlens == nullptr): a [B, H, N, d] tensor; (b, h) is
//    plane b*H + h with rows 0..N-1 (row_stride = d, plane_stride = N*d,
//    statistics [B*H, N]: stat_plane = N).
//  * variable length: a packed [total, H, d] tensor; sequence b holds rows
//    cu_seqlens[b] .. cu_seqlens[b+1]-1 of plane h (row_stride = H*d,
//    plane_stride = d, statistics [H, total]: stat_plane = total).
// causal: query row r of a sequence sees keys c <= r of the same sequence.
struct SeqArgs {
  const int* cu_seqlens;  // device [B+1] or nullptr
  int H;
  int N;                  // fixed length, or the longest sequence (the grid covers it)
  int total;              // rows per plane of the tensors (fixed: N)
  int causal;
  long long row_stride, plane_stride;  // elements
  long long stat_plane;                // elements between planes of LSE / statistics
};

// ---- fp32 CUDA-core path (attn_f32.cu) ----
cudaError_t launch_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                           const SeqArgs& sq, int* status, int BH, int d, float scale,
                           cudaStream_t st);
// Backward stage bits: preprocess, main, dQ convert.
enum : unsigned { kStagePre = 1u, kStageMain = 2u, kStageConvert = 4u, kStageAll = 7u };
// Dws: D per row, [planes, total] floats.
cudaError_t launch_bwd_f32(const float* Q, const float* K, const float* V, const float* O,
                           const float* dO, const float* LSE, float* dQ, float* dK, float* dV,
                           float* Dws, const SeqArgs& sq, int* status, int BH, int d, float scale,
                           unsigned stages, cudaStream_t st);

// ---- bf16 tcgen05 path ----
// Tensor maps view a bf16 tensor of the SeqArgs layout as 3-D (d, rows,
// planes) with 64-element x {128, 64}-row boxes and 128-byte swizzle.
struct FwdArgs {
  CUtensorMap tmQ, tmK, tmV;  // 3-D (d, rows, planes) views of the SeqArgs layout
  CUtensorMap tmO;            // the same view of O (epilogue tensor stores)
  void* O;      // bf16, SeqArgs layout
  float* LSE;   // SeqArgs statistics layout
  SeqArgs seq;
  int BH;       // batch * heads
  float scale_log2;  // scale * log2(e)
  int* status;
  unsigned long long wait_limit_ns;
  // Tail split (fixed length, non-causal): units (head, 256-row block)
  // 0..n_full-1 run whole; the n_tail units after them run as `splits` key
  // ranges each, and a second kernel merges the partial results. splits = 1
  // and n_full = every unit when nothing is split.
  int n_full, n_tail, splits;
  float* Opart;        // fp32 [n_tail][splits][256][d]: normalised partial O
  float* Lpart;        // fp32 [n_tail][splits][256]: base-2 log-sum-exp of each part
  CUtensorMap tmOpart;  // Opart as 2-D (d, rows), 32 x 128 boxes, 128-byte swizzle
  // Test hook (fa_debug_fwd_skip_load): the producer issues neither the load
  // nor the expected-bytes arrival of this key tile (index within the CTA's
  // range), so the consumers' bounded waits run out. -1: load everything.
  int debug_skip_kv;
};
cudaError_t launch_fwd_bf16(const FwdArgs& a, int BH, int d, cudaStream_t st);
// The d = 64 forward with four 128-row query tiles per CTA and 64-key K/V
// tiles (attn_fwd_bf16_q4.cu): fixed-length, non-causal, unsplit problems;
// tmK / tmV must have 64-row boxes.
cudaError_t launch_fwd_bf16_q4(const FwdArgs& a, int BH, cudaStream_t st);
constexpr int kFwdQ4KeyTile = 64;

// The tail split of the bf16 forward for `units` units of n_kv key tiles on
// a GPU that runs `slots` forward CTAs at once: the units of the last,
// partly filled wave are split when that shortens the makespan (whole waves
// + 1/splits instead of + 1).
struct FwdTailPlan {
  int n_full, n_tail, splits;
};
FwdTailPlan plan_fwd_tail(long long units, int n_kv, int slots);
// Scratch for a plan: partial O, partial LSE (256-byte aligned parts).
size_t fwd_tail_workspace_bytes(const FwdTailPlan& p, int d);
// Forward CTAs resident at once on the current device (one per SM).
int fwd_slots();

struct BwdArgs {
  CUtensorMap tmQ, tmK, tmV, tmdO;  // 3-D (d, rows, planes) views of the SeqArgs layout
  CUtensorMap tmdK, tmdV;           // the same views of dK, dV; 32-row boxes (epilogue stores)
  CUtensorMap tmDQacc;  // fp32 [planes*ws_rows, d], 32 x 32 boxes; 128-byte swizzle at d = 64
  const void* O;     // bf16, SeqArgs layout (as Q, K, V, dO, dQ, dK, dV)
  const void* dO;
  const float* LSE;  // SeqArgs statistics layout
  void* dQ;
  void* dK;
  void* dV;
  float* dQacc;      // fp32 [planes, ws_rows, d]
  float* lse2;       // fp32 [planes, ws_rows]  -LSE * log2(e); -inf past the rows
  float* Drow;       // fp32 [planes, ws_rows]  -rowsum(dO o O); 0 past the rows
  SeqArgs seq;
  int planes;        // B*H (fixed) or H (variable length)
  int BH;            // batch * heads
  int ws_rows;       // workspace rows per plane, a multiple of 128: roundup(N, 128)
                     // (fixed length) or roundup(total, 128) + 128 (variable length)
  float scale;
  float scale_log2;
  int* status;
  unsigned long long wait_limit_ns;
  // Test hook (fa_debug_bwd_skip_load): the producer issues neither the load
  // nor the expected-bytes arrival of the Q tile of this iteration, so the
  // consumers' bounded waits run out. -1: load everything.
  int debug_skip_q;
  // Tail split (fixed length, non-causal, splits > 1): units (batch*head,
  // 128-key tile), key tile fastest, 0..n_full-1 run whole; the n_tail units
  // after them run as `splits` ranges of query tiles each, one item per range,
  // leaving fp32 partial dV and dK (unscaled) in dKVpart; the dQ-convert
  // stage adds the ranges up. splits = 1: every unit runs whole.
  int n_full, n_tail, splits;
  float* dKVpart;  // fp32 [n_tail][splits][2 (dV, dK)][128][d]
  // Items of the main kernel's persistent grid (fixed length): non-causal
  // n_full + n_tail * splits, taken by min(items, SM count) CTAs with stride
  // gridDim.x; causal causal_hpg * key tiles * head groups (heads past BH
  // skipped), the first by block index, the rest from *item_counter (zeroed
  // by the preprocess stage); packed batches (an upper bound here; the total
  // is in the schedule the preprocess writes) sequences longest first, then
  // heads, then key tiles, from the counter as well. 0: one unit per CTA of
  // the 2-D/3-D grids.
  int items;
  int causal_hpg;     // heads per group of the causal item order
  int* item_counter;  // in the workspace: the schedule ints (counter first)
  int nseq;           // packed batches: sequences (their schedule follows the counter); else 0
};
cudaError_t launch_bwd_bf16(const BwdArgs& a, int BH, int d, unsigned stages, cudaStream_t st);
// The backward's tail split for `units` (batch*head, key tile) units with n_q
// query tiles each on a GPU running `slots` backward CTAs at once (one per
// SM): the units of a last wave that fills at most half the GPU run as
// splits = min(slots / (units mod slots), 4, n_q / 4) >= 2 query ranges.
struct BwdTailPlan {
  int n_full, n_tail, splits;
};
BwdTailPlan plan_bwd_tail(long long units, int n_q, int slots);
// fp32 partial dV/dK bytes of a plan (0 when nothing is split).
size_t bwd_tail_part_bytes(const BwdTailPlan& p, int d);
// Row padding used by the bf16 backward workspace: ws_rows = roundup(total, 128)
// (+128 with variable lengths, where a sequence's last tile may start anywhere).
constexpr int kBwdRowPad = 128;
// Query rows per streamed tile of the bf16 backward kernel (its Q/dO TMA box
// height); must match BwdCfg<d>::BQ.
constexpr int bwd_query_tile(int d) { return d > 0 ? 128 : 128; }

// Fused row softmax (softmax_rows.cu): rows x cols, fp32 or bf16, cols <= 32768.
constexpr int kSoftmaxMaxCols = 32768;
cudaError_t launch_softmax_rows(const void* X, void* Y, int rows, int cols, float scale, bool bf16,
                                cudaStream_t st);

// ---- KV-cache decode (decode_splitkv.cu) ----
constexpr int kDecodeMaxQueries = 16;
constexpr int kDecodeMaxSplits = 256;
struct DecodeArgs {
  CUtensorMap tmK, tmV;  // [BH, Nk, d] bf16 as 3-D (d, Nk, BH), 64 x decode_tile_keys(Nq) boxes, 128-byte swizzle
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
// The same choice for a given number of resident CTAs on the GPU, with key
// ranges in multiples of `tile` keys.
DecodePlan plan_decode_for_slots(int BH, int Nk, int slots, int tile);
// Keys per tile of the decode kernel used for Nq queries per head (64 on CUDA
// cores for one query, 128 on tensor cores for more).
int decode_tile_keys(int Nq);
cudaError_t launch_decode_bf16(const DecodeArgs& a, int d, cudaStream_t st);

// Causal grids: (heads of a group, blocks, groups). Within a group of heads
// the CTAs run longest first; groups run one after the other, each small
// enough that what its heads' CTAs all stream stays in L2 (bytes_per_head;
// the backward: Q, dO and the dQ accumulator). Groups are of equal size, so
// that the last one is not a short tail of heavy CTAs.
inline int causal_heads_per_group(int BH, long long bytes_per_head, long long budget) {
  long long g = bytes_per_head > 0 ? budget / bytes_per_head : BH;
  if (g < 1) g = 1;
  if (g >= BH) return BH;
  const long long groups = (BH + g - 1) / g;
  return (int)((BH + groups - 1) / groups);
}

// Bounded-wait probe (fa_debug_timeout_probe).
cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t st);

}  // namespace fa
