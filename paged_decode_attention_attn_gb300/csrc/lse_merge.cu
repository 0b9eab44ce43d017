// FP32 log-sum-exp merge of per-tile partials, and the device tail-row write.
//
// Merge rule ("KV-cache engineering", section "Exact recent pages, compact
// older pages"): weight each partial by exp(LSE_i - max LSE), sum the weighted
// outputs, divide by the summed weights, and return max + log(sum) as the
// merged LSE.  Each output column sums its partials in increasing order so
// the result is deterministic (and equal to the decode kernel's fused merge),
// and the division by the summed weights (not a multiply by its reciprocal)
// returns a single partial bit for bit.  The merge reads H*(D+1)*4 bytes per
// partial once; with up to 64 partials per request the time is set by the
// longest rows, whose partials are streamed through shared memory several
// at a time.
#include <cuda_runtime.h>

#include <cmath>

#include "common.h"
#include "ptx.cuh"

namespace pa {
namespace merge {

// One block per (request, head) row; thread t owns float4 column t of each
// kCols-column pass.  The row's partials stream through kStages shared-memory
// stages of kStageParts partials each, filled by cp.async (16 bytes of a
// partial's output row and 4 bytes of its LSE per copy), so the loads in
// flight hold no registers.  Two stages of 12 partials (24.6 KB per block,
// nine blocks per SM) measured best on the merge-stress shape (64 requests x
// 24 heads x 256, 1..64 partials; per launch, back to back on inputs larger
// than L2): 8 x 2 13.4 us, 10 x 2 12.4, 12 x 2 12.0, 14 x 2 13.2, 16 x 2 12.8,
// 20 x 2 12.6, 8 x 3 12.7, 12 x 3 13.5.  Every column sums its partials in
// increasing order with the same expressions as the decode kernel's fused
// merge (mergerow::merge_cols), so the bits are the same.
constexpr int kCols = 64;
constexpr int kStageParts = 12;
constexpr int kStages = 2;
static_assert(kStages >= 1 && kStages <= 4, "the stage waits below cover up to four stages");

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_addr(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(ptx::smem_addr(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kCols)
    lse_merge_kernel(const float* __restrict__ out_parts, const float* __restrict__ lse_parts,
                     const int32_t* __restrict__ offsets, int B, int H, int D,
                     float* __restrict__ out, float* __restrict__ lse) {
  __shared__ __align__(16) float4 sbuf[kStages][kStageParts][kCols];
  __shared__ float slse[kStages][kStageParts];
  __shared__ float red_m[kCols / 32];
  __shared__ int red_nan[kCols / 32];
  ptx::launch_dependents();
  ptx::grid_dependency_wait();  // the partials come from the previous kernel
  const int t = threadIdx.x;
  const int lane = t & 31;
  const long long row = blockIdx.x;
  const int b = static_cast<int>(row / H);
  const int h = static_cast<int>(row - (long long)b * H);
  const int p0 = offsets[b];
  const int n = offsets[b + 1] - p0;

  const int D4 = D / 4;
  const int n_stages = (n + kStageParts - 1) / kStageParts;
  // Stage s of the pass at column c0: partials [s kStageParts, +kStageParts)
  // into buffer s % kStages, one commit group per stage.
  auto issue = [&](int c0, int s) {
    const int c = c0 + t;
    const int i0 = s * kStageParts;
    const int cn = min(kStageParts, n - i0);
    if (c < D4) {
      for (int k = 0; k < cn; ++k)
        cp_async16(&sbuf[s % kStages][k][t],
                   out_parts + ((size_t)(p0 + i0 + k) * H + h) * D + 4 * (size_t)c);
    }
    if (t < cn) cp_async4(&slse[s % kStages][t], lse_parts + (size_t)(p0 + i0 + t) * H + h);
    cp_async_commit();
  };
  // The first pass's first stages need no statistics: they go out before
  // the LSE maximum, whose round trip they overlap.
  for (int s = 0; s < min(kStages, n_stages); ++s) issue(0, s);

  float big_m = -INFINITY;
  int nan = 0;
  for (int i = t; i < n; i += kCols) {
    const float x = lse_parts[(size_t)(p0 + i) * H + h];
    nan |= (x != x);
    big_m = fmaxf(big_m, x);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, off));
    nan |= __shfl_xor_sync(0xffffffffu, nan, off);
  }
  if (lane == 0) {
    red_m[t >> 5] = big_m;
    red_nan[t >> 5] = nan;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kCols / 32; ++w) {
    big_m = fmaxf(big_m, red_m[w]);
    nan |= red_nan[w];
  }
  float4* orow = reinterpret_cast<float4*>(out + (size_t)row * D);
  if (nan || n <= 0 || big_m == -INFINITY) {
    cp_async_wait<0>();   // no copy into this block's shared memory outlives it
    const float fill = nan ? __int_as_float(0x7fc00000) : 0.f;
    for (int c = t; c < D4; c += kCols) orow[c] = make_float4(fill, fill, fill, fill);
    if (t == 0) lse[row] = nan ? fill : -INFINITY;
    return;
  }
  for (int c0 = 0; c0 < D4; c0 += kCols) {
    const int c = c0 + t;
    const bool live = c < D4;
    if (c0 > 0)
      for (int s = 0; s < min(kStages, n_stages); ++s) issue(c0, s);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float ws = 0.f;
    for (int s = 0; s < n_stages; ++s) {
      // Groups committed after stage s's may stay in flight.
      const int ahead = min(n_stages, s + kStages) - s - 1;
      if (ahead >= 3) cp_async_wait<3>();
      else if (ahead == 2) cp_async_wait<2>();
      else if (ahead == 1) cp_async_wait<1>();
      else cp_async_wait<0>();
      __syncthreads();
      const int cn = min(kStageParts, n - s * kStageParts);
      for (int k = 0; k < cn; ++k) {
        const float w = expf(slse[s % kStages][k] - big_m);
        ws += w;
        if (live) {
          const float4 x = sbuf[s % kStages][k][t];
          acc.x = fmaf(w, x.x, acc.x);
          acc.y = fmaf(w, x.y, acc.y);
          acc.z = fmaf(w, x.z, acc.z);
          acc.w = fmaf(w, x.w, acc.w);
        }
      }
      __syncthreads();   // buffer s % kStages is read before it is refilled
      if (s + kStages < n_stages) issue(c0, s + kStages);
    }
    if (live) orow[c] = make_float4(acc.x / ws, acc.y / ws, acc.z / ws, acc.w / ws);
    // ws lies in [1, n] (the largest partial weighs 1): one rounding of
    // big_m + ln(ws), as in the fused merge.
    if (c0 == 0 && t == 0) lse[row] = big_m + logf(ws);
  }
}

// One warp per row: copy rows[b] into the pool row of token positions[b].
__global__ void append_rows_kernel(uint8_t* __restrict__ pool, long long pool_pages,
                                   const int32_t* __restrict__ page_table, int max_pages,
                                   const int32_t* __restrict__ positions,
                                   const uint8_t* __restrict__ rows, int B, int row_bytes,
                                   int32_t* status) {
  ptx::launch_dependents();
  ptx::grid_dependency_wait();  // earlier kernels may still read this row's page
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int pos = positions[b];
  const int lp = pos / PA_PAGE_TOKENS;
  bool bad = pos < 0 || lp >= max_pages;
  long long page = 0;
  if (!bad) {
    page = page_table[(size_t)b * max_pages + lp];
    bad = page < 0 || page >= pool_pages;
  }
  if (bad) {
    if (lane == 0 && status) atomicOr(status, PA_STATUS_BAD_ROW);
    return;
  }
  uint8_t* dst = pool + ((size_t)page * PA_PAGE_TOKENS + pos % PA_PAGE_TOKENS) * row_bytes;
  const uint8_t* src = rows + (size_t)b * row_bytes;
  for (int c = lane; c < row_bytes / 16; c += 32)
    reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
}

}  // namespace merge
}  // namespace pa

extern "C" int lse_merge(const float* out_parts, const float* lse_parts,
                         const int32_t* part_offsets, int B, int H, int D, float* out,
                         float* lse, cudaStream_t stream) {
  pa::clear_error();
  PA_REQUIRE(B >= 0 && H >= 0 && D >= 0, "negative size");
  if ((long long)B * H == 0) return PA_OK;
  // The partial arrays are required even when every request may turn out to
  // have none: the offsets live on the device, so the host cannot tell.
  PA_REQUIRE(out_parts && lse_parts && part_offsets && out && lse, "null pointer argument");
  PA_REQUIRE(D > 0 && D % 4 == 0, "D (%d) must be a positive multiple of 4", D);
  PA_REQUIRE(reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(out_parts) % 16 == 0,
             "out and out_parts must be 16-byte aligned");
  const long long rows = (long long)B * H;
  PA_REQUIRE(rows < (1ll << 31), "too many (request, head) pairs");
  // Many 24.7 KB blocks per SM: ask for the largest shared-memory carveout
  // (once per context).
  static pa::PerContext carveout;
  PA_CHECK_CUDA(carveout.apply([] {
    return cudaFuncSetAttribute(pa::merge::lse_merge_kernel,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  }));
  PA_CHECK_CUDA(pa::launch_dependent(pa::merge::lse_merge_kernel, dim3((unsigned)rows),
                                     dim3(pa::merge::kCols), 0, stream, out_parts, lse_parts,
                                     part_offsets, B, H, D, out, lse));
  PA_CHECK_CUDA(cudaGetLastError());
  return PA_OK;
}

extern "C" int kv_append_rows(void* pool, int64_t pool_pages, const int32_t* page_table,
                              int max_pages, const int32_t* positions, const void* rows, int B,
                              int row_bytes, int32_t* status, cudaStream_t stream) {
  pa::clear_error();
  PA_REQUIRE(B >= 0, "negative B");
  if (B == 0) return PA_OK;
  PA_REQUIRE(pool && page_table && positions && rows, "null pointer argument");
  PA_REQUIRE(row_bytes > 0 && row_bytes % 16 == 0, "row_bytes must be a positive multiple of 16");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(pool) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(rows) % 16 == 0,
             "pool and rows must be 16-byte aligned");
  const int warps_per_block = 4;
  const int blocks = (B + warps_per_block - 1) / warps_per_block;
  PA_CHECK_CUDA(pa::launch_dependent(pa::merge::append_rows_kernel, dim3(blocks),
                                     dim3(warps_per_block * 32), 0, stream,
                                     static_cast<uint8_t*>(pool), pool_pages, page_table,
                                     max_pages, positions, static_cast<const uint8_t*>(rows), B,
                                     row_bytes, status));
  PA_CHECK_CUDA(cudaGetLastError());
  return PA_OK;
}
