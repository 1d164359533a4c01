// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// fa_bwd needs a caller-provided scratch buffer (the fp32 dQ accumulator and
// two per-row statistics). Some callers cannot provide one: code that runs
// inside a host application which owns every byte of device memory through its
// own pool or arena and forbids allocations behind its back, or serving loops
// where a cudaMalloc (which may synchronise the device and can fail under
// memory pressure) is not allowed on the request path. For them this file
// keeps one fixed scratch array in device memory, defined at file scope, and
// passes it to fa_bwd as the workspace.
//
// Properties a caller must know:
//  * The array is FA_BWD_NOALLOC_MAX_WORKSPACE_BYTES (32 MiB) on every device
//    that loads the library, held until the process exits.
//  * Problems whose workspace (fa_bwd_workspace_bytes) exceeds it are rejected
//    with FA_ERR_UNSUPPORTED before anything is launched.
//  * Every call on a device shares the one array. The backward's first stage
//    rewrites everything it reads later (it zeroes the dQ accumulator and
//    writes both statistics), so stale contents from an earlier call do not
//    matter; but two calls whose kernels overlap on the GPU (different
//    streams, no ordering between them) race on the array and give wrong
//    results. Order such calls on one stream or with events.
//  * The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress with that device current) and caches it; make that
//    first call before any stream capture begins.
//  * Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocBytes = FA_BWD_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDev = 64;

// The scratch itself. In host code this name is only a host-side stand-in for
// the device symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device (nullptr on error).
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* LSE, void* dQ, void* dK,
                                    void* dV, int B, int H, int N, int d, float scale,
                                    fa_dtype dt, void* stream) {
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d, dt);
  if (need == 0) {
    // invalid or unsupported shape: let fa_bwd's validation name the error
    return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, nullptr, 0, B, H, N, d, scale, dt, stream);
  }
  if (need > fa::kNoallocBytes) return FA_ERR_UNSUPPORTED;
  void* ws = fa::noalloc_scratch();
  if (!ws) return FA_ERR_CUDA;
  return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, ws, fa::kNoallocBytes, B, H, N, d, scale, dt,
                stream);
}
