// noalloc.cu -- the low-rank head for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a serving runtime
// that fixes its device-memory budget at start-up and forbids allocations once
// requests flow, plugin code hosted inside another framework that exposes no
// device allocator, or a latency-critical loop that cannot afford the
// device-wide synchronisation cudaMalloc may imply.  For them,
// slimspec_head_forward_noalloc runs exactly the kernels of
// slimspec_head_forward with its scratch in a fixed array owned by this
// library instead of a caller workspace.
//
// The array lives in device memory of every GPU that loads the library and
// stays there until the process exits.  Host code cannot use its name as a
// device address, so the address is fetched with cudaGetSymbolAddress (with
// the device current) the first time a device is used, and again whenever
// that device's current context has changed since (a cudaDeviceReset makes
// the runtime load the library's module anew, and the array may move); the
// address is passed to the kernels.  All calls share the one array: calls
// that overlap on the GPU race on it.
#include <cuda.h>  // CUcontext; cuCtxGetCurrent is fetched at run time

#include <mutex>

#include "../../include/slimspec.h"
#include "ss_internal.h"

namespace ss {

// Scratch of slimspec_head_forward_noalloc (SS_NOALLOC_SCRATCH_BYTES bytes).
static __device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// A driver entry point, fetched through the runtime (nullptr if absent).
static void* driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return p;
}

// Process-unique id of the current context (cuCtxGetId: a context created
// after a reset gets a new id even where its handle value is reused), or 0
// when no context is current.  False on a driver error.
static bool current_ctx_id(unsigned long long* id) {
  static const auto get = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
  static const auto get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  CUcontext ctx = nullptr;
  *id = 0;
  if (get == nullptr || get_id == nullptr || get(&ctx) != CUDA_SUCCESS) return false;
  return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call per device and again after the device's context changed (the
// cached address belongs to the context it was looked up in).  Returns
// nullptr (and a status) on error.
static void* noalloc_scratch(int* status) {
  static std::mutex mu;
  static void* cached[64] = {nullptr};
  static unsigned long long cached_ctx[64] = {0};
  int dev = 0;
  unsigned long long ctx = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || !current_ctx_id(&ctx)) {
    *status = SS_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (ctx == 0 || cached[dev] == nullptr || cached_ctx[dev] != ctx) {
    // the lookup also makes the device's primary context current if no
    // context was yet
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr || !current_ctx_id(&ctx) || ctx == 0) {
      *status = SS_ERR_CUDA;
      return nullptr;
    }
    cached[dev] = p;
    cached_ctx[dev] = ctx;
  }
  return cached[dev];
}

}  // namespace ss

extern "C" int slimspec_head_forward_noalloc(const void* hidden, const void* w_down,
                                             const void* w_up, int M, int d, int r, int V,
                                             int dtype, float temperature, uint64_t seed,
                                             uint64_t offset, const float* uniforms,
                                             int32_t* out_tokens, float* out_logprob,
                                             float* out_row_max, float* out_row_lse, void* out_z,
                                             float* out_logits, cudaStream_t stream) {
  const size_t need = slimspec_head_workspace_size(M, d, r, V, dtype);
  if (need == 0)  // argument errors (reported by the regular call) or an empty batch
    return slimspec_head_forward(hidden, w_down, w_up, M, d, r, V, dtype, temperature, seed,
                                 offset, uniforms, out_tokens, out_logprob, out_row_max,
                                 out_row_lse, out_z, out_logits, nullptr, 0, stream);
  if (need > (size_t)SS_NOALLOC_SCRATCH_BYTES) return SS_ERR_WORKSPACE;
  int status = SS_OK;
  void* scratch = ss::noalloc_scratch(&status);
  if (scratch == nullptr) return status;
  // Nothing in the scratch has to start at zero: the call clears the counters
  // it uses and overwrites everything else it reads.
  return slimspec_head_forward(hidden, w_down, w_up, M, d, r, V, dtype, temperature, seed, offset,
                               uniforms, out_tokens, out_logprob, out_row_max, out_row_lse, out_z,
                               out_logits, scratch, (size_t)SS_NOALLOC_SCRATCH_BYTES, stream);
}
