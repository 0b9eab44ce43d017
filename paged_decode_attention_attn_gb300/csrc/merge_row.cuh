// The FP32 log-sum-exp merge of one (request, head) row, used by the decode
// kernel's fused cross-tile merge.  The standalone merge kernel (lse_merge.cu)
// computes every column with the same expressions in the same partial order,
// so both give the same bits.
//
// Merge rule ("KV-cache engineering", section "Exact recent pages, compact
// older pages"): weight each partial by exp(LSE_i - max LSE), sum the weighted
// outputs, divide by the summed weights, and return max + log(sum) as the
// merged LSE.  One warp per row; partials are read in increasing order so the
// result is deterministic, and the division by the summed weights (not a
// multiply by its reciprocal) returns a single partial bit for bit.
#pragma once

#include <cuda_runtime.h>

#include <cmath>

namespace pa {
namespace mergerow {

constexpr int kVecPerLane = 2;  // float4 chunks of the output row per lane per pass

// kL2: read through L2 only (partials written by other CTAs of the running
// kernel); otherwise plain loads (partials from an earlier kernel).
template <bool kL2>
__device__ __forceinline__ float load1(const float* p) {
  if constexpr (kL2) return __ldcg(p);
  else return *p;
}
template <bool kL2>
__device__ __forceinline__ float4 load4(const float4* p) {
  if constexpr (kL2) return __ldcg(p);
  else return *p;
}

// Partial i of the row is out_parts[((p0 + i) * H + h) * D ...] with LSE
// lse_parts[(p0 + i) * H + h], i < n.  Writes the float4 columns [c_lo, c_hi)
// of orow and, when lse_out is not null, *lse_out.  D is a multiple of 4 and
// the rows 16-byte aligned.  Called by all 32 lanes of a warp; several warps
// may share a row by taking disjoint column ranges.
//   kBatch  partials whose loads are issued before their arithmetic (bytes in
//           flight per warp);
//   kVec    float4 columns per lane per pass.
// Every column's arithmetic runs in partial order whatever kBatch, kVec and
// the column split, so the result bits depend on none of them.
template <bool kL2, int kBatch, int kVec>
__device__ __forceinline__ void merge_cols(const float* out_parts, const float* lse_parts, int p0,
                                           int n, int H, int h, int D, int c_lo, int c_hi,
                                           float* orow, float* lse_out, int lane) {
  float big_m = -INFINITY;
  int nan = 0;
  for (int i = lane; i < n; i += 32) {
    const float x = load1<kL2>(lse_parts + (size_t)(p0 + i) * H + h);
    nan |= (x != x);
    big_m = fmaxf(big_m, x);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, off));
    nan |= __shfl_xor_sync(0xffffffffu, nan, off);
  }
  if (nan || n <= 0 || big_m == -INFINITY) {
    const float fill = nan ? __int_as_float(0x7fc00000) : 0.f;
    for (int c = c_lo + lane; c < c_hi; c += 32)
      reinterpret_cast<float4*>(orow)[c] = make_float4(fill, fill, fill, fill);
    if (lane == 0 && lse_out) *lse_out = nan ? fill : -INFINITY;
    return;
  }
  float wsum = 0.f;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32 * kVec) {
    float4 acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float ws = 0.f;
    for (int i0 = 0; i0 < n; i0 += kBatch) {
      float lx[kBatch];
      float4 xs[kBatch][kVec];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j;
        if (i < n) {
          lx[j] = load1<kL2>(lse_parts + (size_t)(p0 + i) * H + h);
          const float4* src =
              reinterpret_cast<const float4*>(out_parts + ((size_t)(p0 + i) * H + h) * D);
#pragma unroll
          for (int v = 0; v < kVec; ++v) {
            const int c = c0 + v * 32 + lane;
            if (c < c_hi) xs[j][v] = load4<kL2>(src + c);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (i0 + j < n) {
          const float w = expf(lx[j] - big_m);
          ws += w;
#pragma unroll
          for (int v = 0; v < kVec; ++v) {
            const int c = c0 + v * 32 + lane;
            if (c < c_hi) {
              acc[v].x = fmaf(w, xs[j][v].x, acc[v].x);
              acc[v].y = fmaf(w, xs[j][v].y, acc[v].y);
              acc[v].z = fmaf(w, xs[j][v].z, acc[v].z);
              acc[v].w = fmaf(w, xs[j][v].w, acc[v].w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const int c = c0 + v * 32 + lane;
      if (c < c_hi)
        reinterpret_cast<float4*>(orow)[c] =
            make_float4(acc[v].x / ws, acc[v].y / ws, acc[v].z / ws, acc[v].w / ws);
    }
    wsum = ws;
  }
  // wsum is in [1, n] (the largest partial weighs 1): one fp32 rounding of
  // big_m + ln(wsum); a single partial gives big_m exactly.  It is the same
  // sum on every pass and in every warp of the row.
  if (lane == 0 && lse_out) *lse_out = big_m + logf(wsum);
}

// The whole row (all D columns and the LSE) by one warp, loads one partial
// at a time: the decode kernel's fused cross-tile merge.
template <bool kL2>
__device__ __forceinline__ void merge_row(const float* out_parts, const float* lse_parts, int p0,
                                          int n, int H, int h, int D, float* orow, float* lse_out,
                                          int lane) {
  merge_cols<kL2, 1, kVecPerLane>(out_parts, lse_parts, p0, n, H, h, D, 0, D / 4, orow, lse_out,
                                  lane);
}

}  // namespace mergerow
}  // namespace pa
