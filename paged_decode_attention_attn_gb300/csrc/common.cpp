// Error reporting and small device queries shared by every entry point.
#include "common.h"

#include <cuda.h>

#include <cstdio>
#include <mutex>

namespace pa {

namespace {
thread_local char g_message[1024] = "";
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_message, sizeof(g_message), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_message[0] = '\0'; }

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
}  // namespace

bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(ptr);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace pa

extern "C" const char* kv_last_error(void) { return pa::g_message; }

#define PA_STR2(x) #x
#define PA_STR(x) PA_STR2(x)

extern "C" const char* pa_version(void) {
  return "libpagedattn 0.1 (sm_103a, CUDA runtime " PA_STR(CUDART_VERSION) ")";
}

// Pinned host memory for the caller's history and compact store ("GPU memory
// management", section "A host pool that explains its own size": the host
// pool that owns every history is pinned and sized explicitly).
extern "C" int kv_host_alloc(size_t bytes, void** out) {
  pa::clear_error();
  if (!out || bytes == 0) return pa::fail(PA_ERR_INVALID, "bytes must be > 0 and out non-null");
  *out = nullptr;
  const cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocDefault);
  if (e != cudaSuccess) {
    *out = nullptr;
    return pa::fail(PA_ERR_CUDA, "cudaHostAlloc of %zu bytes failed: %s", bytes,
                    cudaGetErrorString(e));
  }
  return PA_OK;
}

extern "C" int kv_host_free(void* p) {
  pa::clear_error();
  if (!p) return PA_OK;
  const cudaError_t e = cudaFreeHost(p);
  return e == cudaSuccess ? PA_OK
                          : pa::fail(PA_ERR_CUDA, "cudaFreeHost failed: %s", cudaGetErrorString(e));
}
