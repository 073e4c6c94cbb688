// tv_noalloc.cu -- tv_verify_attn_noalloc: the CUDA-core attention with its split-KV
// scratch taken from a fixed device array inside the library instead of a caller
// workspace.
//
// Why: some callers cannot hand the library a workspace.  A plugin loaded into a host
// program that owns every byte of device memory has no allocator to call; a serving loop
// that must never stall cannot call cudaMalloc/cudaFree, which may synchronise the whole
// device; a caller with a fixed, pre-planned memory budget may not grow it at run time.
// For them the scratch lives in `g_noalloc_scratch` below, reserved when the library is
// loaded on a device and held by that device until the process exits.
//
// The scratch holds the per-split partial outputs and log-sum-exps of the split-KV
// decomposition.  Every split writes its partial for every row before the combine kernel
// reads it, so nothing in the array has to start at zero and stale contents from an
// earlier call are never read.  Calls share the one array: two calls whose kernels can
// overlap on the GPU (different streams without ordering, or different host threads)
// race on it and must be serialised by the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "tv.h"
#include "tv_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)TV_NOALLOC_SCRATCH_BYTES;

// One copy per device that loads the library.  In host code this name is only a host
// stand-in for the symbol, never a device address: the address is looked up per device
// with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// The address is cached per device together with the CUDA context it was looked up in: a
// new context on the device (after cudaDeviceReset, or a context the caller made current)
// loads the module again, possibly elsewhere, so the lookup is then repeated.
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  CUcontext c = nullptr;
  if (!g_ctx_current || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

void set_error(const char* what, cudaError_t e) {
  char buf[256];
  snprintf(buf, sizeof(buf), "tv_verify_attn_noalloc: %s failed: %s", what, cudaGetErrorString(e));
  tv::set_last_error(buf);
}

// Device address of the scratch array in the current device's current context.  The first
// call on a device (and the first after that device's context changed) looks it up with
// cudaGetSymbolAddress, which may load the library's device code; make that call before
// any stream capture.  Returns nullptr and sets the error text on failure.
void* scratch_for_current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error("cudaGetDevice", e);
    return nullptr;
  }
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev] || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      set_error("cudaGetSymbolAddress", e);
      g_scratch_ptr[dev] = nullptr;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
    // the look-up makes the runtime's context current if there was none yet
    g_scratch_ctx[dev] = ctx ? ctx : current_context();
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t tv_noalloc_scratch_bytes(void) { return kScratchBytes; }

int tv_verify_attn_noalloc(const tv_attn_args* a, void* stream) {
  // Validation shared with tv_verify_attn (sets the error text on failure).
  const int path = tv_verify_attn_path(a);
  if (path < 0) return path;
  if (a->path == TV_PATH_TCGEN05) {
    tv::set_last_error("tv_verify_attn_noalloc: runs the CUDA-core kernel only");
    return TV_ERR_UNSUPPORTED;
  }
  if (!tv::simt_supported(a)) {
    tv::set_last_error("tv_verify_attn_noalloc: shape not supported by the CUDA-core kernel");
    return TV_ERR_UNSUPPORTED;
  }
  if (a->B == 0) return TV_OK;
  const tv::SimtPlan plan = tv::simt_plan(a, tv::current_sm_count());
  const size_t need = tv::simt_workspace(a, plan);
  if (need > kScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "tv_verify_attn_noalloc: needs %zu bytes of scratch, the fixed array holds %zu; "
             "use tv_verify_attn with a workspace, or fewer splits",
             need, kScratchBytes);
    tv::set_last_error(buf);
    return TV_ERR_WORKSPACE;
  }
  // The address is resolved on every call, also when this request needs no scratch, so
  // that the first call on a device always does the one-time look-up.
  void* scratch = scratch_for_current_device();
  if (!scratch) return TV_ERR_CUDA;
  void* ws = need > 0 ? scratch : nullptr;
  cudaError_t e = tv::launch_attn_simt(a, plan, ws, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    char buf[256];
    snprintf(buf, sizeof(buf), "tv_verify_attn_noalloc: %s", cudaGetErrorString(e));
    tv::set_last_error(buf);
    return TV_ERR_CUDA;
  }
  tv::set_last_error("");
  return TV_OK;
}

}  // extern "C"
