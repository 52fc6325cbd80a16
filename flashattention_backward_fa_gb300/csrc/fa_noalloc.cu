// fa_bwd_noalloc: the deterministic backward without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code running inside a pre-planned memory arena that forbids new
// allocations, runtimes that record work before any allocator exists, or
// embedding environments that hand over only the tensors themselves. For them
// this entry point takes the scratch it needs (the per-row D and L*log2(e)
// vectors of the deterministic backward and four unit counters of its
// persistent kernels) from one fixed device array that is
// part of this library's module, so the call allocates nothing.
//
// Limits and sharing:
//  * The array holds kNoAllocScratchBytes (8 MiB + 256 bytes): B*H*roundup(N,128) must not
//    exceed 1,048,576 rows. Larger problems are rejected with FA_ERR_WORKSPACE
//    before anything is launched; use fa_bwd with a workspace for them.
//  * Every GPU that loads the library holds the array until the process exits.
//  * All calls on a device share the one array and it keeps the last call's
//    contents. Each call overwrites every entry it reads (including the row
//    padding) in its first kernel, so nothing needs clearing between calls.
//    Calls whose kernels overlap on the GPU (different streams without
//    ordering between them) race on the array: order them.
//  * The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current). Make
//    that first call before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_host.h"
#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (8u << 20) + 256u;
constexpr int kMaxDevicesNoAlloc = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevicesNoAlloc] = {};

// Device address of the scratch array on the current device (looked up once per device).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoAlloc) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                              fa_strides strides, fa_dtype dtype, float scale, int causal, int window,
                              float dropout_p, uint64_t seed, uint64_t offset, void* stream) {
  // The same size, dtype and stride checks as fa_bwd first, so that both entry
  // points return the same code for the same bad argument; then the scratch limit.
  int rc = fa::check_bwd_args(B, H, N, d, strides, dtype, scale, window, dropout_p);
  if (rc) return rc;
  const size_t need = fa_bwd_workspace_size(B, H, N, d, dtype, FA_DQ_RECOMPUTE);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  // Single stream: this entry point creates nothing, not even the side stream.
  return fa::bwd_run(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, strides, dtype, scale, causal, window,
                     dropout_p, seed, offset, fa::Extras{}, FA_DQ_RECOMPUTE, scratch, kNoAllocScratchBytes, stream,
                     false);
}
