// swa_attend_noalloc: the attention of swa_attend, with its split-KV scratch in
// a fixed array that the library owns, so that the caller never allocates.
//
// Some callers cannot call cudaMalloc: a plugin that a host program hands only
// its input and output buffers, a serving engine whose device memory is all
// reserved up front by its own allocator, or a latency-critical loop that must
// not take the device-wide synchronisation an allocation can cause. For them
// the scratch (the per-split partial records and the valid-split counts) lives
// in the file-scope array below, which every GPU that loads this library holds
// until the process exits.
#include "swa_internal.cuh"

#include <cuda.h>

#include <mutex>

namespace swa {
namespace {

constexpr size_t kScratchBytes = SWA_NOALLOC_SCRATCH_BYTES;

// The scratch itself. In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current CUDA context, 0 when there is
// none or the driver cannot say. The driver functions are taken from the
// runtime, so the library needs no link against the driver library.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q{};
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_scratch on the current device, looked up (with that
// device current) on the first call and again whenever the device's context
// has changed since: after cudaDeviceReset the module is loaded anew and the
// array may sit at another address.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return SWA_E_SHAPE;
  std::lock_guard<std::mutex> lock(g_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (!p) return SWA_E_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();   // the lookup made the device's context current
  }
  *out = g_scratch_ptr[dev];
  return SWA_OK;
}

}  // namespace
}  // namespace swa

extern "C" int swa_attend_noalloc(const swa_attend_args* args, cudaStream_t stream) {
  // the checks of swa_attend first, in its order, so both report the same error
  const int rc0 = swa::attend_args_status(args);
  if (rc0 != SWA_OK) return rc0;
  // Sizes whose partial records would not fit the fixed scratch are refused
  // before anything is enqueued (the split-once operand blocks of the tensor-core
  // prompt kernel are used when they fit as well, skipped otherwise).
  const size_t need = swa_attend_workspace_min(args);
  if (need == 0) return SWA_E_SHAPE;
  if (need > swa::kScratchBytes) return SWA_E_WORKSPACE;
  void* scratch = nullptr;
  const int rc = swa::scratch_address(&scratch);
  if (rc != SWA_OK) return rc;
  swa_attend_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = swa::kScratchBytes;
  return swa_attend(&a, stream);
}
