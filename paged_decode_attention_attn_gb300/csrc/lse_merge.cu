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
// longest rows, so each row is spread over several warps and each warp keeps
// several partials' loads in flight.
#include <cuda_runtime.h>

#include <cmath>

#include "common.h"
#include "merge_row.cuh"
#include "ptx.cuh"

namespace pa {
namespace merge {

constexpr int kWarpsPerBlock = 8;
constexpr int kLoadBatch = 8;  // partials loaded ahead of their arithmetic per warp
constexpr int kVec = 1;        // float4 columns per lane: a warp takes 128 columns of a row
constexpr int kChunkCols = 32 * kVec;

// One warp per (request, head, 128-column chunk): a row with many partials is
// read by D/128 warps at once.  The chunk-0 warp writes the row's LSE.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    lse_merge_kernel(const float* __restrict__ out_parts, const float* __restrict__ lse_parts,
                     const int32_t* __restrict__ offsets, int B, int H, int D, int n_chunks,
                     float* __restrict__ out, float* __restrict__ lse) {
  ptx::launch_dependents();
  ptx::grid_dependency_wait();  // the partials come from the previous kernel
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (wid >= (long long)B * H * n_chunks) return;
  const long long row = wid / n_chunks;
  const int chunk = static_cast<int>(wid - row * n_chunks);
  const int b = static_cast<int>(row / H);
  const int h = static_cast<int>(row - (long long)b * H);
  const int p0 = offsets[b];
  const int n = offsets[b + 1] - p0;
  const int c_lo = chunk * kChunkCols;
  const int c_hi = min(D / 4, c_lo + kChunkCols);
  mergerow::merge_cols<false, kLoadBatch, kVec>(out_parts, lse_parts, p0, n, H, h, D, c_lo, c_hi,
                                                out + (size_t)row * D,
                                                chunk == 0 ? lse + row : nullptr, lane);
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
  PA_REQUIRE(part_offsets && out && lse, "null pointer argument");
  PA_REQUIRE(D > 0 && D % 4 == 0, "D (%d) must be a positive multiple of 4", D);
  PA_REQUIRE(reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
                 reinterpret_cast<uintptr_t>(out_parts) % 16 == 0,
             "out and out_parts must be 16-byte aligned");
  const int n_chunks = (D / 4 + pa::merge::kChunkCols - 1) / pa::merge::kChunkCols;
  const long long warps = (long long)B * H * n_chunks;
  const long long blocks = (warps + pa::merge::kWarpsPerBlock - 1) / pa::merge::kWarpsPerBlock;
  PA_REQUIRE(blocks < (1ll << 31), "too many (request, head) pairs");
  PA_CHECK_CUDA(pa::launch_dependent(pa::merge::lse_merge_kernel, dim3((unsigned)blocks),
                                     dim3(pa::merge::kWarpsPerBlock * 32), 0, stream, out_parts,
                                     lse_parts, part_offsets, B, H, D, n_chunks, out, lse));
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
