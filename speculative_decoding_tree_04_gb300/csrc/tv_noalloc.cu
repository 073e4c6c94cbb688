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
#include <cuda_runtime.h>

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
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up once per device
// (the first call on a device does it, so that call should come before any stream
// capture).  Returns nullptr and sets the error text on failure.
void* scratch_for_current_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char buf[256];
    snprintf(buf, sizeof(buf), "tv_verify_attn_noalloc: cudaGetDevice failed: %s",
             cudaGetErrorString(e));
    tv::set_last_error(buf);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      snprintf(buf, sizeof(buf), "tv_verify_attn_noalloc: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      tv::set_last_error(buf);
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
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
  void* ws = nullptr;
  if (need > 0) {
    ws = scratch_for_current_device();
    if (!ws) return TV_ERR_CUDA;
  }
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
