// Shared host-side helpers of libpagedattn: error reporting and device queries.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cuda_runtime.h>

#include "pagedattn.h"

namespace pa {

// Sets the thread-local message returned by kv_last_error() and returns code.
int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void clear_error();

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

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
