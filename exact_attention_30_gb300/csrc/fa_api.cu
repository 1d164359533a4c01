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

// [BH, N, d] bf16 viewed as 3-D (d, N, BH); box 64 x box_rows x 1, 128-byte
// swizzle. Rows past N within a head read as zero.
bool encode_bhnd_bf16(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 [rows, d] accumulator as 2-D (d, rows); 32 x 32 boxes, no swizzle.
bool encode_acc_f32(CUtensorMap* m, void* ptr, long long rows, int d) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status check_shape(int B, int H, int N, int d, float scale, fa_dtype dt) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (dt != FA_F32 && dt != FA_BF16) return FA_ERR_INVALID_ARG;
  const long long BH = (long long)B * H;
  if (BH > 65535) return FA_ERR_UNSUPPORTED;  // grid.y
  if (BH * (long long)N * d >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  if (dt == FA_BF16 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dt == FA_F32 && d > 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct BwdWorkspaceLayout {
  size_t dqacc, lse2, drow, total;
  int Npad;
};
BwdWorkspaceLayout bwd_layout(int B, int H, int N, int d, fa_dtype dt) {
  BwdWorkspaceLayout L{};
  const size_t BH = (size_t)B * H;
  if (dt == FA_F32) {
    L.Npad = N;
    L.drow = 0;
    L.total = align_up(BH * N * sizeof(float), 256);
    return L;
  }
  L.Npad = (N + kBwdRowPad - 1) / kBwdRowPad * kBwdRowPad;
  L.dqacc = 0;
  L.lse2 = align_up(BH * L.Npad * d * sizeof(float), 256);
  L.drow = L.lse2 + align_up(BH * L.Npad * sizeof(float), 256);
  L.total = L.drow + align_up(BH * L.Npad * sizeof(float), 256);
  return L;
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

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int N, int d, float scale, fa_dtype dt, void* stream) {
  fa_status s = check_shape(B, H, N, d, scale, dt);
  if (s != FA_OK) return s;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  const size_t al = dt == FA_BF16 ? 16 : 4;
  if (!aligned(Q, al) || !aligned(K, al) || !aligned(V, al) || !aligned(O, al) || !aligned(LSE, 4))
    return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  if (dt == FA_F32) {
    return launch_fwd_f32(static_cast<const float*>(Q), static_cast<const float*>(K),
                          static_cast<const float*>(V), static_cast<float*>(O), LSE, BH, N, d,
                          scale, st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  if (!get_encode_fn()) return FA_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  if (!encode_bhnd_bf16(&a.tmQ, Q, BH, N, d, 128) || !encode_bhnd_bf16(&a.tmK, K, BH, N, d, 128) ||
      !encode_bhnd_bf16(&a.tmV, V, BH, N, d, 128))
    return FA_ERR_CUDA;
  a.O = O;
  a.LSE = LSE;
  a.N = N;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.wait_limit_ns = kDefaultWaitLimitNs;
  return launch_fwd_bf16(a, BH, d, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d, fa_dtype dt) {
  if (check_shape(B, H, N, d, 1.0f, dt) != FA_OK) return 0;
  return bwd_layout(B, H, N, d, dt).total;
}

}  // extern "C"

namespace {
fa_status bwd_impl(unsigned stages, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                   void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                   float scale, fa_dtype dt, void* stream) {
  fa_status s = check_shape(B, H, N, d, scale, dt);
  if (s != FA_OK) return s;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
    return FA_ERR_INVALID_ARG;
  const size_t al = dt == FA_BF16 ? 16 : 4;
  if (!aligned(Q, al) || !aligned(K, al) || !aligned(V, al) || !aligned(O, al) ||
      !aligned(dO, al) || !aligned(dQ, al) || !aligned(dK, al) || !aligned(dV, al) ||
      !aligned(LSE, 4) || !aligned(workspace, 256))
    return FA_ERR_INVALID_ARG;
  const BwdWorkspaceLayout L = bwd_layout(B, H, N, d, dt);
  if (workspace_bytes < L.total) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  if (dt == FA_F32) {
    return launch_bwd_f32(static_cast<const float*>(Q), static_cast<const float*>(K),
                          static_cast<const float*>(V), static_cast<const float*>(O),
                          static_cast<const float*>(dO), LSE, static_cast<float*>(dQ),
                          static_cast<float*>(dK), static_cast<float*>(dV),
                          static_cast<float*>(workspace), BH, N, d, scale, stages, st) == cudaSuccess
               ? FA_OK
               : FA_ERR_CUDA;
  }
  if (!get_encode_fn()) return FA_ERR_CUDA;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  // query-side tiles (Q, dO) are bwd_query_tile(d) rows, key-side tiles 128 rows
  const int qrows = bwd_query_tile(d);
  if (!encode_bhnd_bf16(&a.tmQ, Q, BH, N, d, qrows) || !encode_bhnd_bf16(&a.tmK, K, BH, N, d, 128) ||
      !encode_bhnd_bf16(&a.tmV, V, BH, N, d, 128) || !encode_bhnd_bf16(&a.tmdO, dO, BH, N, d, qrows))
    return FA_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  a.O = O;
  a.dO = dO;
  a.LSE = LSE;
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.dQacc = reinterpret_cast<float*>(ws + L.dqacc);
  if (!encode_acc_f32(&a.tmDQacc, a.dQacc, (long long)BH * L.Npad, d)) return FA_ERR_CUDA;
  a.lse2 = reinterpret_cast<float*>(ws + L.lse2);
  a.Drow = reinterpret_cast<float*>(ws + L.drow);
  a.N = N;
  a.Npad = L.Npad;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.wait_limit_ns = kDefaultWaitLimitNs;
  return launch_bwd_bf16(a, BH, d, stages, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

extern "C" {

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int N, int d, float scale, fa_dtype dt,
                 void* stream) {
  return bwd_impl(kStageAll, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H,
                  N, d, scale, dt, stream);
}

fa_status fa_bwd_stage(int stage, const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                       void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                       float scale, fa_dtype dt, void* stream) {
  unsigned bits;
  switch (stage) {
    case FA_BWD_PREPROCESS: bits = kStagePre; break;
    case FA_BWD_MAIN: bits = kStageMain; break;
    case FA_BWD_DQ_CONVERT: bits = kStageConvert; break;
    default: return FA_ERR_INVALID_ARG;
  }
  return bwd_impl(bits, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, N, d,
                  scale, dt, stream);
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
  const DecodePlan p = resident_ctas > 0 ? plan_decode_for_slots(B * H, Nk, resident_ctas)
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
  if (!encode_bhnd_bf16(&a.tmK, K, BH, Nk, d, 64) || !encode_bhnd_bf16(&a.tmV, V, BH, Nk, d, 64))
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
  return v == 0 ? FA_OK : (v == kStatusTimeout ? FA_ERR_TIMEOUT : FA_ERR_CUDA);
}

fa_status fa_debug_timeout_probe(long long limit_ns, void* stream) {
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 2000000000ll) limit_ns = 2000000000ll;
  int* status = device_status_ptr();
  if (!status) return FA_ERR_CUDA;
  return launch_timeout_probe(status, (unsigned long long)limit_ns,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // extern "C"
