// Shared host-side helpers of libpagedattn: error reporting and device queries.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "pagedattn.h"

namespace pa {

// Sets the thread-local message returned by kv_last_error() and returns code.
int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Id of the CUDA context current on this thread (unique for the process's
// lifetime, so a context destroyed and made again gets a new one); false if
// no context is current or the driver cannot say.
bool current_context_id(unsigned long long* id);

// A per-context setting (a kernel attribute, say): apply(set) runs `set`
// (returning cudaError_t) unless it already succeeded in the context now
// current on this thread's device, so a device reset, or a primary context
// released and made again, gets the setting anew.  When the driver cannot
// name the context, every call runs `set`.
class PerContext {
 public:
  template <typename F>
  cudaError_t apply(F set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevices) return set();
    unsigned long long id = 0;
    const bool have = current_context_id(&id);
    std::lock_guard<std::mutex> lock(mu_);
    if (have && done_[dev] && ctx_[dev] == id) return cudaSuccess;
    e = set();
    if (e != cudaSuccess) return e;
    // `set` makes the device's primary context current if none was.
    done_[dev] = current_context_id(&ctx_[dev]);
    return cudaSuccess;
  }

 private:
  static constexpr int kDevices = 64;
  std::mutex mu_;
  bool done_[kDevices] = {};
  unsigned long long ctx_[kDevices] = {};
};

// Launches a kernel that may start while the previous kernel in the stream is
// still running (programmatic dependent launch).  The kernel must execute
// griddepcontrol.wait before it reads anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace pa

#define PA_CHECK_CUDA(call)                                                    \
  do {                                                                         \
    cudaError_t pa_err_ = (call);                                              \
    if (pa_err_ != cudaSuccess)                                                \
      return ::pa::fail(PA_ERR_CUDA, "%s failed: %s", #call,                   \
                        cudaGetErrorString(pa_err_));                          \
  } while (0)

#define PA_REQUIRE(cond, ...)                                                  \
  do {                                                                         \
    if (!(cond)) return ::pa::fail(PA_ERR_INVALID, __VA_ARGS__);               \
  } while (0)
