// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// TMA tensor-map encoding, the device status word and kernel dispatch.
// Host code only, apart from the bounded-wait probe kernel at the bottom.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

// One status word per device that loads the library; kernels record bounded
// wait expiry here, fa_check_device_status reads and clears it.
__device__ int g_fa_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool get_encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return true;
}

// A bf16 tensor of the SeqArgs layout viewed as 3-D (d, rows, planes); box
// 64 x box_rows x 1, 128-byte swizzle. Rows past `total` read as zero.
bool encode_seq_bf16(CUtensorMap* m, const void* ptr, const SeqArgs& sq, int planes, int d,
                     int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)sq.total, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)sq.row_stride * 2, (cuuint64_t)sq.plane_stride * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [BH, N, d] bf16 (the fixed-length layout).
bool encode_bhnd_bf16(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows) {
  SeqArgs sq{};
  sq.total = N;
  sq.row_stride = d;
  sq.plane_stride = (long long)N * d;
  return encode_seq_bf16(m, ptr, sq, BH, d, box_rows);
}

// fp32 [rows, d] accumulator as 2-D (d, rows); 32 x 32 boxes.
bool encode_acc_f32(CUtensorMap* m, void* ptr, long long rows, int d) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  // d = 128 stages [query][32 d] blocks written one d column per lane (no
  // swizzle needed); d = 64 stages one query row per lane, in the 128-byte
  // swizzle that keeps those shared-memory stores free of bank conflicts.
  const CUtensorMapSwizzle sw = d == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Partial O of the forward's split units: fp32 [rows, d] as 2-D (d, rows),
// boxes of 32 columns (128 bytes) x 128 rows in the 128-byte swizzle.
bool encode_part_f32(CUtensorMap* m, void* ptr, long long rows, int d) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status check_dtype_d(int d, fa_dtype dt) {
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  if (dt == FA_BF16 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dt == FA_F32 && d > 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_shape(int B, int H, int N, int d, float scale, fa_dtype dt) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  if (BH > 65535) return FA_ERR_UNSUPPORTED;  // a grid dimension
  if (BH * (long long)N * d >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  return check_dtype_d(d, dt);
}

fa_status check_varlen(const int* cu_seqlens, int B, int H, int total, int max_seqlen, int d,
                       float scale, fa_dtype dt) {
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || total < 1 || max_seqlen < 1 || max_seqlen > total || d < 1)
    return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
  if ((long long)total * H * d >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  return check_dtype_d(d, dt);
}

SeqArgs fixed_seq(int H, int N, int d, bool causal) {
  SeqArgs sq{};
  sq.cu_seqlens = nullptr;
  sq.H = H;
  sq.N = N;
  sq.total = N;
  sq.causal = causal ? 1 : 0;
  sq.row_stride = d;
  sq.plane_stride = (long long)N * d;
  sq.stat_plane = N;
  return sq;
}

SeqArgs varlen_seq(const int* cu_seqlens, int H, int total, int max_seqlen, int d, bool causal) {
  SeqArgs sq{};
  sq.cu_seqlens = cu_seqlens;
  sq.H = H;
  sq.N = max_seqlen;
  sq.total = total;
  sq.causal = causal ? 1 : 0;
  sq.row_stride = (long long)H * d;
  sq.plane_stride = d;
  sq.stat_plane = total;
  return sq;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct BwdWorkspaceLayout {
  size_t dqacc, lse2, drow, part, sched, total;
  int planes, ws_rows;
  BwdTailPlan plan;
};
// fp32: D per row ([planes, total]). bf16: fp32 dQ accumulator
// [planes, ws_rows, d], two per-row statistics [planes, ws_rows] and, when the
// schedule splits its tail (fixed length, non-causal, on the current device),
// the split units' fp32 partial dV and dK, and the main kernel's item counter.
BwdWorkspaceLayout bwd_layout(const SeqArgs& sq, int B, int d, fa_dtype dt) {
  BwdWorkspaceLayout L{};
  L.plan = BwdTailPlan{0, 0, 1};
  L.planes = sq.cu_seqlens ? sq.H : B * sq.H;
  const size_t P = (size_t)L.planes;
  if (dt == FA_F32) {
    L.ws_rows = sq.total;
    L.drow = 0;
    L.total = align_up(P * sq.total * sizeof(float), 256);
    return L;
  }
  L.ws_rows = (sq.total + kBwdRowPad - 1) / kBwdRowPad * kBwdRowPad + (sq.cu_seqlens ? kBwdRowPad : 0);
  L.dqacc = 0;
  L.lse2 = align_up(P * L.ws_rows * d * sizeof(float), 256);
  L.drow = L.lse2 + align_up(P * L.ws_rows * sizeof(float), 256);
  L.part = L.drow + align_up(P * L.ws_rows * sizeof(float), 256);
  if (!sq.causal && sq.cu_seqlens == nullptr)
    L.plan = plan_bwd_tail((long long)B * sq.H * ((sq.N + 127) / 128), (sq.N + 127) / 128, fwd_slots());
  L.sched = L.part + bwd_tail_part_bytes(L.plan, d);
  // the main kernel's schedule: item counter, item total and, for a packed
  // batch, the sequence order and the B + 1 unit prefix sums
  L.total = L.sched + align_up(sizeof(int) * (2 + (sq.cu_seqlens ? 2 * (size_t)B + 1 : 0)), 256);
  return L;
}

unsigned flag_stages(int flags) {
  const unsigned m = ((unsigned)flags >> 8) & 7u;
  return m == 0 ? kStageAll : m;
}

}  // namespace

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

// ---------------------------------------------------------------------------
// bounded-wait probe: one block waits on a barrier nobody arrives at
// ---------------------------------------------------------------------------
__global__ void timeout_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(b, 0, status, limit_ns);  // gives up, records a timeout
  __syncthreads();
}

cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

namespace {

// Bounded-wait limit of the test hooks, clamped to [1 us, 2 s].
unsigned long long clamp_limit(long long limit_ns) {
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 2000000000ll) limit_ns = 2000000000ll;
  return (unsigned long long)limit_ns;
}

// The bf16 forward at d = 64 runs on the four-query-tile kernel (one CTA per
// batch*head and 512-row block) when the problem is fixed-length (causal or
// not) and its grid fills at least three quarters of the GPU's resident CTAs
// (fewer CTAs leave too many SMs idle; the two-tile kernel's grid, twice as
// large and split at its tail, then finishes first). Everything else runs on
// the two-tile kernel. `slots`: forward CTAs resident at once (the SM count).
bool fwd_uses_q4(const SeqArgs& sq, int BH, int d, fa_dtype dt, int slots) {
  if (dt != FA_BF16 || d != 64 || sq.cu_seqlens != nullptr) return false;
  const long long ctas = (long long)BH * ((sq.N + 511) / 512);
  return 4 * ctas >= 3ll * slots;
}

// Tail split of the bf16 forward for this problem on the current device (only
// fixed-length, non-causal problems of the two-tile kernel are split; the
// others: one plain plan).
FwdTailPlan fwd_tail_plan(const SeqArgs& sq, int BH, int d, fa_dtype dt) {
  const long long qblocks = ((long long)sq.N + 255) / 256;
  const long long units = qblocks * BH;
  if (dt != FA_BF16 || sq.causal || sq.cu_seqlens || fwd_uses_q4(sq, BH, d, dt, fwd_slots()))
    return FwdTailPlan{(int)units, 0, 1};
  return plan_fwd_tail(units, (sq.N + 127) / 128, fwd_slots());
}

fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   const SeqArgs& sq, int B, int d, float scale, fa_dtype dt, void* stream,
                   void* workspace = nullptr, size_t workspace_bytes = 0, int debug_skip = -1,
                   unsigned long long wait_limit_ns = kDefaultWaitLimitNs) {
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  const size_t al = dt == FA_BF16 ? 16 : 4;
  if (!aligned(Q, al) || !aligned(K, al) || !aligned(V, al) || !aligned(O, al) || !aligned(LSE, 4))
    return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * sq.H;
  const int planes = sq.cu_seqlens ? sq.H : BH;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  if (dt == FA_F32) {
    return launch_fwd_f32(static_cast<const float*>(Q), static_cast<const float*>(K),
                          static_cast<const float*>(V), static_cast<float*>(O), LSE, sq, status, BH,
                          d, scale, st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  if (!get_encode_fn()) return FA_ERR_CUDA;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool q4 = fwd_uses_q4(sq, BH, d, dt, fwd_slots());
  const int kv_rows = q4 ? kFwdQ4KeyTile : 128;  // TMA box height of the K/V tiles
  if (!encode_seq_bf16(&a.tmQ, Q, sq, planes, d, 128) || !encode_seq_bf16(&a.tmK, K, sq, planes, d, kv_rows) ||
      !encode_seq_bf16(&a.tmV, V, sq, planes, d, kv_rows) || !encode_seq_bf16(&a.tmO, O, sq, planes, d, 128))
    return FA_ERR_CUDA;
  a.O = O;
  a.LSE = LSE;
  a.seq = sq;
  a.BH = BH;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.debug_skip_kv = debug_skip;
  FwdTailPlan plan = fwd_tail_plan(sq, BH, d, dt);
  const size_t need = fwd_tail_workspace_bytes(plan, d);
  if (workspace != nullptr && need > 0) {
    if (!aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    const size_t rows = (size_t)plan.n_tail * plan.splits * 256;
    const size_t o_bytes = (rows * d * 4 + 255) & ~(size_t)255;
    char* ws = static_cast<char*>(workspace);
    a.Opart = reinterpret_cast<float*>(ws);
    a.Lpart = reinterpret_cast<float*>(ws + o_bytes);
    if (!encode_part_f32(&a.tmOpart, a.Opart, (long long)rows, d)) return FA_ERR_CUDA;
  } else {
    plan = FwdTailPlan{plan.n_full + plan.n_tail, 0, 1};  // no scratch: every unit runs whole
  }
  a.n_full = plan.n_full;
  a.n_tail = plan.n_tail;
  a.splits = plan.splits;
  if (q4) return launch_fwd_bf16_q4(a, BH, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  return launch_fwd_bf16(a, BH, d, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status bwd_impl(unsigned stages, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                   void* workspace, size_t workspace_bytes, const SeqArgs& sq, int B, int d,
                   float scale, fa_dtype dt, void* stream, int debug_skip = -1,
                   unsigned long long wait_limit_ns = kDefaultWaitLimitNs) {
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
    return FA_ERR_INVALID_ARG;
  const size_t al = dt == FA_BF16 ? 16 : 4;
  if (!aligned(Q, al) || !aligned(K, al) || !aligned(V, al) || !aligned(O, al) ||
      !aligned(dO, al) || !aligned(dQ, al) || !aligned(dK, al) || !aligned(dV, al) ||
      !aligned(LSE, 4) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const BwdWorkspaceLayout L = bwd_layout(sq, B, d, dt);
  if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * sq.H;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  if (dt == FA_F32) {
    return launch_bwd_f32(static_cast<const float*>(Q), static_cast<const float*>(K),
                          static_cast<const float*>(V), static_cast<const float*>(O),
                          static_cast<const float*>(dO), LSE, static_cast<float*>(dQ),
                          static_cast<float*>(dK), static_cast<float*>(dV),
                          static_cast<float*>(workspace), sq, status, BH, d, scale, stages,
                          st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  if (!get_encode_fn()) return FA_ERR_CUDA;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  // query-side tiles (Q, dO) are bwd_query_tile(d) rows, key-side tiles 128 rows
  const int qrows = bwd_query_tile(d);
  if (!encode_seq_bf16(&a.tmQ, Q, sq, L.planes, d, qrows) ||
      !encode_seq_bf16(&a.tmK, K, sq, L.planes, d, 128) ||
      !encode_seq_bf16(&a.tmV, V, sq, L.planes, d, 128) ||
      !encode_seq_bf16(&a.tmdO, dO, sq, L.planes, d, qrows) ||
      !encode_seq_bf16(&a.tmdK, dK, sq, L.planes, d, 32) ||
      !encode_seq_bf16(&a.tmdV, dV, sq, L.planes, d, 32))
    return FA_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  a.O = O;
  a.dO = dO;
  a.LSE = LSE;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.dQacc = reinterpret_cast<float*>(ws + L.dqacc);
  if (!encode_acc_f32(&a.tmDQacc, a.dQacc, (long long)L.planes * L.ws_rows, d)) return FA_ERR_CUDA;
  a.lse2 = reinterpret_cast<float*>(ws + L.lse2);
  a.Drow = reinterpret_cast<float*>(ws + L.drow);
  a.seq = sq;
  a.planes = L.planes;
  a.BH = BH;
  a.ws_rows = L.ws_rows;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.debug_skip_q = debug_skip;
  a.n_full = L.plan.n_full;
  a.n_tail = L.plan.n_tail;
  a.splits = L.plan.splits;
  a.dKVpart = L.plan.splits > 1 ? reinterpret_cast<float*>(ws + L.part) : nullptr;
  a.item_counter = reinterpret_cast<int*>(ws + L.sched);
  if (sq.cu_seqlens != nullptr) {
    // packed batch: every (sequence, head, key tile) unit, at most
    // B * H * ceil(max_seqlen / 128); the preprocess writes the exact total
    const long long bound = (long long)BH * ((sq.N + 127) / 128);
    if (bound <= (1ll << 30)) {  // else one CTA per unit of the 2-D grid
      a.nseq = B;
      a.items = (int)bound;
    }
  } else {
    // fixed length: the persistent grid's item list
    const int kblocks = (sq.N + 127) / 128;
    if (sq.causal) {
      a.causal_hpg = causal_heads_per_group(BH, 8ll * sq.N * d, 48ll << 20);
      a.items = a.causal_hpg * kblocks * ((BH + a.causal_hpg - 1) / a.causal_hpg);
    } else {
      a.items = L.plan.n_full + L.plan.n_tail * L.plan.splits;
    }
  }
  return launch_bwd_bf16(a, BH, d, stages, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported configuration";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime or launch error";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel abandoned a bounded wait";
    default: return "unknown fa_status";
  }
}

fa_status fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                    int N, int d, float scale, int flags, fa_dtype dt, void* stream) {
  const fa_status s = check_shape(B, H, N, d, scale, dt);
  if (s != FA_OK) return s;
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, fixed_seq(H, N, d, flags & FA_CAUSAL), B, d, scale, dt, stream);
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int N, int d, float scale, fa_dtype dt, void* stream) {
  return fa_fwd_ex(Q, K, V, O, LSE, B, H, N, d, scale, 0, dt, stream);
}

size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int flags, fa_dtype dt) {
  if (check_shape(B, H, N, d, 1.f, dt) != FA_OK || (flags & ~FA_CAUSAL)) return 0;
  const SeqArgs sq = fixed_seq(H, N, d, flags & FA_CAUSAL);
  return fwd_tail_workspace_bytes(fwd_tail_plan(sq, B * H, d, dt), d);
}

fa_status fa_fwd_plan(int B, int H, int N, int d, int flags, fa_dtype dt, int resident_ctas,
                      int* n_full, int* n_tail, int* splits) {
  if (!n_full || !n_tail || !splits || resident_ctas < 0) return FA_ERR_INVALID_ARG;
  const fa_status s = check_shape(B, H, N, d, 1.f, dt);
  if (s != FA_OK) return s;
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  const SeqArgs sq = fixed_seq(H, N, d, flags & FA_CAUSAL);
  const long long units = ((long long)N + 255) / 256 * B * H;
  FwdTailPlan p{(int)units, 0, 1};
  if (resident_ctas == 0)
    p = fwd_tail_plan(sq, B * H, d, dt);
  else if (dt == FA_BF16 && !(flags & FA_CAUSAL) && !fwd_uses_q4(sq, B * H, d, dt, resident_ctas))
    p = plan_fwd_tail(units, (N + 127) / 128, resident_ctas);
  *n_full = p.n_full;
  *n_tail = p.n_tail;
  *splits = p.splits;
  return FA_OK;
}

fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                    float scale, int flags, fa_dtype dt, void* stream) {
  const fa_status s = check_shape(B, H, N, d, scale, dt);
  if (s != FA_OK) return s;
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, fixed_seq(H, N, d, flags & FA_CAUSAL), B, d, scale, dt, stream,
                  workspace, workspace_bytes);
}

fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const int* cu_seqlens, int B, int H, int total, int max_seqlen, int d,
                        float scale, int flags, fa_dtype dt, void* stream) {
  const fa_status s = check_varlen(cu_seqlens, B, H, total, max_seqlen, d, scale, dt);
  if (s != FA_OK) return s;
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, varlen_seq(cu_seqlens, H, total, max_seqlen, d, flags & FA_CAUSAL),
                  B, d, scale, dt, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d, fa_dtype dt) {
  if (check_shape(B, H, N, d, 1.0f, dt) != FA_OK) return 0;
  return bwd_layout(fixed_seq(H, N, d, false), B, d, dt).total;
}

fa_status fa_bwd_plan(int B, int H, int N, int d, int flags, fa_dtype dt, int resident_ctas,
                      int* n_full, int* n_tail, int* splits) {
  if (!n_full || !n_tail || !splits || resident_ctas < 0) return FA_ERR_INVALID_ARG;
  const fa_status s = check_shape(B, H, N, d, 1.f, dt);
  if (s != FA_OK) return s;
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  const long long units = (long long)B * H * ((N + 127) / 128);
  BwdTailPlan p{(int)units, 0, 1};
  if (dt == FA_BF16 && !(flags & FA_CAUSAL)) {
    if (resident_ctas == 0)
      p = bwd_layout(fixed_seq(H, N, d, false), B, d, dt).plan;
    else
      p = plan_bwd_tail(units, (N + 127) / 128, resident_ctas);
  }
  *n_full = p.n_full;
  *n_tail = p.n_tail;
  *splits = p.splits;
  return FA_OK;
}

size_t fa_bwd_varlen_workspace_bytes(int B, int H, int total, int max_seqlen, int d, fa_dtype dt) {
  static const int kDummy[2] = {0, 0};  // only the sizes are checked here
  if (check_varlen(kDummy, B, H, total, max_seqlen, d, 1.0f, dt) != FA_OK) return 0;
  return bwd_layout(varlen_seq(kDummy, H, total, max_seqlen, d, false), B, d, dt).total;
}

fa_status fa_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                    size_t workspace_bytes, int B, int H, int N, int d, float scale, int flags,
                    fa_dtype dt, void* stream) {
  const fa_status s = check_shape(B, H, N, d, scale, dt);
  if (s != FA_OK) return s;
  if (flags & ~(FA_CAUSAL | FA_STAGE_MASK)) return FA_ERR_INVALID_ARG;
  return bwd_impl(flag_stages(flags), Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes,
                  fixed_seq(H, N, d, flags & FA_CAUSAL), B, d, scale, dt, stream);
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float scale, fa_dtype dt,
                 void* stream) {
  return fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale,
                   0, dt, stream);
}

fa_status fa_bwd_stage(int stage, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, fa_dtype dt, void* stream) {
  int bits;
  switch (stage) {
    case FA_BWD_PREPROCESS: bits = FA_STAGE_PREPROCESS; break;
    case FA_BWD_MAIN: bits = FA_STAGE_MAIN; break;
    case FA_BWD_DQ_CONVERT: bits = FA_STAGE_DQ_CONVERT; break;
    default: return FA_ERR_INVALID_ARG;
  }
  return fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d, scale,
                   bits, dt, stream);
}

fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV, const int* cu_seqlens,
                        void* workspace, size_t workspace_bytes, int B, int H, int total,
                        int max_seqlen, int d, float scale, int flags, fa_dtype dt, void* stream) {
  const fa_status s = check_varlen(cu_seqlens, B, H, total, max_seqlen, d, scale, dt);
  if (s != FA_OK) return s;
  if (flags & ~(FA_CAUSAL | FA_STAGE_MASK)) return FA_ERR_INVALID_ARG;
  return bwd_impl(flag_stages(flags), Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes,
                  varlen_seq(cu_seqlens, H, total, max_seqlen, d, flags & FA_CAUSAL), B, d, scale,
                  dt, stream);
}

fa_status fa_softmax_rows(const void* X, void* Y, int rows, int cols, float scale, fa_dtype dt,
                          void* stream) {
  if (!X || !Y || rows < 1 || cols < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  const size_t es = dt == FA_BF16 ? 2 : 4;
  if (!aligned(X, es) || !aligned(Y, es)) return FA_ERR_INVALID_ARG;
  if (cols > kSoftmaxMaxCols) return FA_ERR_UNSUPPORTED;
  if ((long long)rows * cols >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  return launch_softmax_rows(X, Y, rows, cols, scale, dt == FA_BF16,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"

namespace {
fa_status check_decode(int B, int H, int Nq, int Nk, int d, fa_dtype dt) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  if (dt != FA_BF16 || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  if (Nq > kDecodeMaxQueries || Nk > (1 << 30)) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

struct DecodeLayout {
  DecodePlan plan;
  size_t opart, lsepart, total;
};
DecodeLayout decode_layout(int B, int H, int Nq, int Nk, int d) {
  DecodeLayout L{};
  L.plan = plan_decode(B * H, Nq, Nk, d);
  if (L.plan.splits < 1) return L;
  const size_t rows = (size_t)B * H * Nq;
  L.opart = 0;
  L.lsepart = align_up((size_t)L.plan.splits * rows * d * sizeof(float), 256);
  L.total = L.lsepart + align_up((size_t)L.plan.splits * rows * sizeof(float), 256);
  return L;
}
}  // namespace

extern "C" {

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d, fa_dtype dt) {
  if (check_decode(B, H, Nq, Nk, d, dt) != FA_OK) return 0;
  return decode_layout(B, H, Nq, Nk, d).total;
}

fa_status fa_decode_plan(int B, int H, int Nq, int Nk, int d, int resident_ctas, int* splits,
                         int* keys_per_split) {
  if (!splits || !keys_per_split || resident_ctas < 0) return FA_ERR_INVALID_ARG;
  const fa_status s = check_decode(B, H, Nq, Nk, d, FA_BF16);
  if (s != FA_OK) return s;
  const DecodePlan p = resident_ctas > 0
                           ? plan_decode_for_slots(B * H, Nk, resident_ctas, decode_tile_keys(Nq))
                           : plan_decode(B * H, Nq, Nk, d);
  if (p.splits < 1) return FA_ERR_CUDA;
  *splits = p.splits;
  *keys_per_split = p.keys_per_split;
  return FA_OK;
}

fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int H, int Nq, int Nk, int d,
                    float scale, fa_dtype dt, void* stream) {
  fa_status s = check_decode(B, H, Nq, Nk, d, dt);
  if (s != FA_OK) return s;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !LSE || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
      !aligned(LSE, 4) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(B, H, Nq, Nk, d);
  if (L.plan.splits < 1) return FA_ERR_CUDA;
  if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
  if (!get_encode_fn()) return FA_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  const int BH = B * H;
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  // TMA boxes are the decode kernel's key tile (64 or 128 rows)
  const int box_rows = decode_tile_keys(Nq);
  if (!encode_bhnd_bf16(&a.tmK, K, BH, Nk, d, box_rows) ||
      !encode_bhnd_bf16(&a.tmV, V, BH, Nk, d, box_rows))
    return FA_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  a.Q = Q;
  a.O = O;
  a.LSE = LSE;
  a.Opart = reinterpret_cast<float*>(ws + L.opart);
  a.LSEpart = reinterpret_cast<float*>(ws + L.lsepart);
  a.BH = BH;
  a.Nq = Nq;
  a.Nk = Nk;
  a.splits = L.plan.splits;
  a.keys_per_split = L.plan.keys_per_split;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.wait_limit_ns = kDefaultWaitLimitNs;
  return launch_decode_bf16(a, d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                     : FA_ERR_CUDA;
}

fa_status fa_check_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  int* p = device_status_ptr();
  if (!p) return FA_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0 && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_CUDA;
  if (v == 0) return FA_OK;
  if (v == kStatusTimeout) return FA_ERR_TIMEOUT;
  if (v == kStatusBadSeqlens) return FA_ERR_INVALID_ARG;
  return FA_ERR_CUDA;
}

fa_status fa_debug_fwd_skip_load(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int N, int d, float scale, int skip_tile,
                                 long long limit_ns, void* stream) {
  const fa_status s = check_shape(B, H, N, d, scale, FA_BF16);
  if (s != FA_OK) return s;
  if (skip_tile < 1 || skip_tile >= (N + 127) / 128) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, fixed_seq(H, N, d, false), B, d, scale, FA_BF16, stream, nullptr,
                  0, skip_tile, clamp_limit(limit_ns));
}

fa_status fa_debug_bwd_skip_load(const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                 void* workspace, size_t workspace_bytes, int B, int H, int N,
                                 int d, float scale, int skip_tile, long long limit_ns,
                                 void* stream) {
  const fa_status s = check_shape(B, H, N, d, scale, FA_BF16);
  if (s != FA_OK) return s;
  if (skip_tile < 1 || skip_tile >= (N + bwd_query_tile(d) - 1) / bwd_query_tile(d))
    return FA_ERR_INVALID_ARG;
  return bwd_impl(kStageAll, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes,
                  fixed_seq(H, N, d, false), B, d, scale, FA_BF16, stream, skip_tile,
                  clamp_limit(limit_ns));
}

fa_status fa_debug_bwd_skip_load_ex(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* LSE, void* dQ, void* dK,
                                    void* dV, void* workspace, size_t workspace_bytes, int B,
                                    int H, int N, int d, float scale, int flags, int skip_tile,
                                    long long limit_ns, void* stream) {
  if (flags & ~FA_CAUSAL) return FA_ERR_INVALID_ARG;
  const fa_status s = check_shape(B, H, N, d, scale, FA_BF16);
  if (s != FA_OK) return s;
  if (skip_tile < 1 || skip_tile >= (N + bwd_query_tile(d) - 1) / bwd_query_tile(d))
    return FA_ERR_INVALID_ARG;
  return bwd_impl(kStageAll, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes,
                  fixed_seq(H, N, d, (flags & FA_CAUSAL) != 0), B, d, scale, FA_BF16, stream,
                  skip_tile, clamp_limit(limit_ns));
}

fa_status fa_debug_timeout_probe(long long limit_ns, void* stream) {
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return launch_timeout_probe(status, clamp_limit(limit_ns),
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"
