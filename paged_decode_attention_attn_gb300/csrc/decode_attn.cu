// Split-KV paged GQA decode attention with a per-tile log-sum-exp, for sm_103a.
//
// What it computes ("KV-cache engineering", section "Exact recent pages,
// compact older pages"): for every tile of a request's history and every
// query head, the softmax-normalised output over the tile's keys and the
// tile's log-sum-exp, so that tiles can later be merged exactly.  The history
// is read once per call ("Costing the bus before changing anything": the exact
// path re-reads every byte of history for every generated token), so the
// kernel is bound by HBM bandwidth and is built around keeping HBM busy:
//
//  * Work = (tile, kv head) units, each a run of 64-token pages.  All units'
//    pages are laid end to end and cut into one contiguous page range per CTA
//    (persistent grid, one CTA per SM; 90% of the SMs for launches of many
//    pages per SM), so every CTA streams the same number of pages whatever the
//    mix of lengths.  A unit that spans several CTAs leaves one partial (max,
//    sum, unnormalised output) per CTA; once the last of them has arrived, the
//    unit's CTAs merge the partials in slices of the output, each slice with a
//    fixed summation order, so the result does not depend on timing, on which
//    CTA merges which slice, or on where pages sit physically.
//  * One producer warp streams pages with TMA: per page the K slice and the V
//    slice of one kv head (64 rows x 512 B each, row stride 4 KiB) as eight
//    64x64 boxes with the 128-byte swizzle, into a 3-stage mbarrier ring
//    (64 KiB per stage).
//  * Eight consumer warps: each 16-token group of a page is taken by two
//    warps that compute the same grouped scores and split the 256 output
//    dims, so every SM sub-partition interleaves two consumer warps.  All
//    G <= 8 query heads of the GQA group share the page, so the grouped
//    scores are a 16 x 8 x 256 product per warp (tensor-core mma.sync
//    m16n8k16, heads as rows, bf16 in, fp32 accumulate).  Online softmax runs
//    in the log2 domain against a reference kept on multiples of 8, so it
//    moves (an exact power-of-two rescale) only when the max crosses the next
//    multiple.  P enters the PV product as a hi + lo pair of bf16 values
//    packed into the otherwise idle rows 8..15 of the A tile (~16 significant
//    bits of every probability at no extra MMA cost); each page's PV product
//    starts from zero and is added to the running output with fp32
//    round-to-nearest adds.
//  * A CUDA-core variant (FP32 FMAs, one lane per 8 dims) runs the same
//    pipeline; it exists to measure the tensor-core choice against.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.h"
#include "merge_row.cuh"
#include "ptx.cuh"

namespace pa {
namespace decode {

constexpr int kPage = PA_PAGE_TOKENS;                    // tokens per page
constexpr int kD = 256;                                  // head_dim
constexpr int kMaxG = 8;                                 // query heads per kv head
constexpr int kStages = 3;
constexpr int kGroups = 4;                               // 16-token groups per page
constexpr int kBoxCols = 64;                             // 128 B swizzle span
constexpr int kBoxBytes = kPage * kBoxCols * 2;          // 8 KiB
constexpr int kHalfBytes = kBoxBytes * (kD / kBoxCols);  // K (or V) slice: 32 KiB
constexpr int kStageBytes = 2 * kHalfBytes;              // 64 KiB
constexpr int kXRow = kD + 8;                            // padded exchange row
constexpr int kXOBytes = kGroups * kMaxG * kXRow * 4;
constexpr int kXMLBytes = kGroups * kMaxG * 2 * 4;  // >= 3 * kMaxG floats for the merge
constexpr int kSmemXO = kStages * kStageBytes;
constexpr int kSmemXML = kSmemXO + kXOBytes;
constexpr int kSmemBar = kSmemXML + kXMLBytes;
constexpr int kSmemMisc = kSmemBar + 2 * kStages * 8;
constexpr int kSmemUsed = kSmemMisc + 64;
constexpr int kSmemAlloc = kSmemUsed + 1024;             // slack to align to 1 KiB
constexpr int kMaxUnitsLarge = 1024;
constexpr int kMaxUnitsSmall = 64;
constexpr int kWidePages = 32;     // pages per SM from which a launch leaves SMs idle
constexpr int kWideGridPct = 90;   // share of the SMs such a launch runs on
constexpr int kSegmentCharge = 6;  // pages charged per segment when CTAs' shares are cut (measured: 3-8 best)
constexpr uint64_t kWaitLimitNs = 2000000000ull;         // 2 s per wait
// A split unit's merge reads up to kMaxPartsPerLane partials per lane of a
// 32-lane team, which bounds the CTAs a unit may span and so the grid.
constexpr int kMaxPartsPerLane = 5;
constexpr int kMaxGrid = 32 * kMaxPartsPerLane;
// How long a CTA that has stored its partial waits without seeing another
// CTA of the unit arrive before it leaves its share of the merge to the
// unit's last CTA.  The CTAs of a launch finish within ~25 us of each other
// (per-SM streaming speeds differ by up to ~10% over a long launch), with
// arrivals every few hundred ns; the limit matters only when some of them
// cannot be resident at the same time (other work holds SMs), where waiting
// longer would only delay them.
constexpr uint64_t kSliceWaitNs = 50000ull;
constexpr size_t kStatusBytes = 256;
// A split unit's outputs are merged in at most this many slices, one per
// waiting CTA: enough to spread the partials' loads, few enough that most of
// a widely split unit's CTAs leave at once (their SMs then take the next
// launch's first page loads).
constexpr int kMaxSlices = 16;
// Per unit: a 64-bit arrival word (count | leavers << 16 | generation << 32).
constexpr size_t kCounterBytes = 8 * kMaxUnitsLarge;
constexpr size_t kPartOBytes = size_t(kMaxG) * kD * 4;   // per partial slot
constexpr size_t kPartMLBytes = size_t(kMaxG) * 2 * 4;
constexpr float kLn2Hi = 0.693145751953125f;        // ln 2, high bits (exact products)
constexpr float kLn2Lo = 1.428606765330187045e-06f; // ln 2 - kLn2Hi
constexpr float kLog2e = 1.44269504088896341f;
// The running softmax reference is kept on multiples of kRefStep (log2 units):
// rescales and the weights between partials are then exact powers of two, and
// every probability is the same number (up to an exact power of two) however
// the tokens are split into tiles, chunks and warps.
constexpr float kRefStep = 8.0f;

static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kMaxSlices <= kMaxGrid - 1, "slices per split unit");

struct Unit {
  int32_t bt_g;        // (b * T + t) * Hkv + g
  int32_t tok_start;
  int32_t tok_end;
  int32_t page_first;  // flattened index of the unit's first page in this launch
  int32_t part_base;   // first partial slot (units covered by several CTAs)
  int32_t n_parts;     // CTAs covering the unit
  int32_t pair_total;  // completions the (request, kv head) tile counter reaches (fused merge)
};

template <int kMaxUnits>
struct Params {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  float* out;
  float* lse;
  int32_t* status;
  unsigned long long* arrivals;  // [unit] split units: CTAs arrived, leavers, generation
  int32_t* req_counters;  // [B][Hkv] tiles finished (fused merge)
  float* part_o;   // [slot][kMaxG][kD]
  float* part_ml;  // [slot][kMaxG][2]
  long long pool_pages;
  long long total_pages;
  int max_pages;
  int T;
  int Hq;
  int Hkv;
  int G;
  int n_units;
  int grid;
  float scale_log2;
  // Optional new-token rows: row new_rows[b] is written to the pool at token
  // positions[b] of request b, and attention uses it for that token.
  __nv_bfloat16* pool;
  const __nv_bfloat16* new_rows;
  const int32_t* positions;
  int n_requests;
  int row_elems;
  // The page table and the pool rows read are final before the kernel that
  // precedes this one in the stream runs: the producer may issue its first
  // kStages page loads before the grid dependency wait.
  int kv_ready;
  // Bounded device waits give up after wait_limit_ns (PA_STATUS_TIMEOUT).
  // stall_iteration >= 0 (test hook only): CTA 0's producer leaves that
  // stage unarmed, so its consumers' wait runs out.
  unsigned long long wait_limit_ns;
  int stall_iteration;
  // How long a split unit's CTA waits without a new arrival before it
  // leaves its merge slice to the unit's last CTA (kSliceWaitNs; a test hook
  // can shorten it to exercise that path).
  unsigned long long slice_wait_ns;
  // Optional fused cross-tile merge: merged [B][Hq][kD] and [B][Hq].
  float* m_out;
  float* m_lse;
  Unit units[kMaxUnits];
};
// Kernel parameters travel in the 32 KiB parameter space.
static_assert(sizeof(Params<kMaxUnitsLarge>) <= 32764, "kernel parameters too large");

// Slices a unit split over n >= 2 CTAs is merged in: half its CTAs wait and
// merge, the other half leave at once (their SMs take the next launch's first
// page loads).  Measured per launch against n - 1 slices (both capped at 16),
// one box: 4 x 31,744 tokens (n ~ 9) 77.76 -> 77.05 us, 2 x 32,768 (n ~ 19)
// 44.18 -> 43.37 us, 1 x 32,768 (n ~ 38) and 1 x 262,144 unchanged; a third
// of them cost 1 x 32,768 0.3 us, two thirds gained half as much.
__host__ __device__ __forceinline__ int split_slices(int n) {
  return n / 2 < kMaxSlices ? n / 2 : kMaxSlices;
}

__host__ __device__ __forceinline__ int unit_pages(int tok_start, int tok_end) {
  return tok_end > tok_start ? (tok_end + kPage - 1) / kPage - tok_start / kPage : 0;
}

// CTAs of a launch of `total` flattened pages on a device of `sms` SMs.  A
// launch of at least kWidePages pages per SM runs on kWideGridPct percent of
// the SMs: with HBM saturated, fewer, longer streams finish sooner.  Measured
// per launch on one box (grids 152 / 144 / 136 / 128): 4 x 31,744 tokens 78.6
// / 77.9 / 78.1 / 78.1 us, 1 x 262,144 in 8 tiles 157.5 / 155.7 / 154.8 /
// 155.6 us, the ragged window workload 462.4 / 459.8 / 459.2 / 460.3 us;
// smaller launches keep every SM (1 x 32,768: 25.4 us on 152, 25.7 on 136;
// 2 x 32,768 within 0.1% from 120 to 152).  Of the other launches above the
// threshold measured, 3 x 32,768, 8 x 16,384 and 64 x 2,048 gain 0.2-1.6% and
// 16 x 8,192 loses 0.6%.
// The grid is rounded down to a multiple of the kv-head count (when it holds
// at least one CTA per kv head), so the CTAs at the same offset of each kv
// head's block of units stream the same pages at the same time: with 4 kv
// heads, 129 CTAs took the bench workload to 80.6 us against 77.1 on 136 and
// 77.1 on 144; with 6 kv heads, 150 CTAs instead of 152 took 1 x 32,768
// tokens from 34.95 to 34.05 us and 2 x 16,384 from 34.64 to 33.94 us.
__host__ __forceinline__ int launch_grid(long long total, int sms, int n_kv_heads) {
  if (total <= 0) return 1;
  int grid = total >= (long long)kWidePages * sms ? std::max(1, sms * kWideGridPct / 100)
                                                  : (int)std::min<long long>(sms, total);
  if (grid >= n_kv_heads) grid -= grid % n_kv_heads;
  return grid;
}

// CTA whose page range [k P / grid, (k+1) P / grid) holds flattened page p.
__host__ __device__ __forceinline__ int cta_of(long long p, long long total, int grid) {
  return static_cast<int>(((p + 1) * grid - 1) / total);
}

template <int N>
__device__ __forceinline__ int first_unit(const Params<N>& p, long long start) {
  int lo = 0, hi = p.n_units - 1, ans = 0;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (p.units[mid].page_first <= start) {
      ans = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  return ans;
}

// ln-domain LSE of a reference m (log2 units, a multiple of kRefStep) and a
// sum l > 0: (m + e) ln 2 + ln f with l = f 2^e, f in [0.5, 1).  m + e is an
// exact small integer, its product with the high part of ln 2 (a Cody-Waite
// split) is exact, and the small terms go into the last addition, so the
// result carries about one fp32 rounding, as a double evaluation rounded to
// fp32 would -- without FP64 arithmetic, which is slow on this part (a double
// log per row had cost microseconds of every launch's tail).
__device__ __forceinline__ float lse_of(float m, float l) {
  if (m == -INFINITY || !(l > 0.f)) return m * kLn2Hi + logf(l);   // -inf / degenerate
  int e;
  const float f = frexpf(l, &e);
  const float t = m + static_cast<float>(e);
  return t * kLn2Hi + fmaf(t, kLn2Lo, logf(f));
}

__device__ __forceinline__ float ref_ceil(float x) {
  return ceilf(x * (1.0f / kRefStep)) * kRefStep;
}

// Weight of a partial whose reference is m relative to the common reference
// big_m >= m (both multiples of kRefStep): exactly 2^(m - big_m), 0 for -inf.
__device__ __forceinline__ float ref_weight(float m, float big_m) {
  return (m == -INFINITY) ? 0.f : ptx::pow2i(static_cast<int>(m - big_m));
}

struct Shared {
  uint8_t* stages;
  float* xo;       // [token group][kMaxG][kXRow]
  float* xml;      // [token group][kMaxG][2]
  uint32_t full_bar;
  uint32_t empty_bar;
  volatile int* poison;  // [kStages]
  volatile int* abort_flag;
  volatile int* fin_flag;
  volatile int* merge_info;  // split-unit merge: mode, leavers, finisher
};

__device__ __forceinline__ Shared carve(uint8_t* raw) {
  Shared s;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.stages = base;
  s.xo = reinterpret_cast<float*>(base + kSmemXO);
  s.xml = reinterpret_cast<float*>(base + kSmemXML);
  s.full_bar = ptx::smem_addr(base + kSmemBar);
  s.empty_bar = s.full_bar + kStages * 8;
  int* misc = reinterpret_cast<int*>(base + kSmemMisc);
  s.poison = misc;
  s.abort_flag = misc + kStages;
  s.fin_flag = misc + kStages + 2;
  s.merge_info = misc + 8;
  return s;
}

// Writes `count` 16-byte chunks of a new row's K (or V) slice into row r of
// a swizzled stage half (K at half_base, V at half_base + kHalfBytes): chunk
// c (8 dims) goes to box c / 8, 16-byte position (c % 8) ^ (r % 8).
__device__ __forceinline__ void put_row_chunk(uint32_t half_base, int r, int c, uint4 v) {
  const uint32_t a = half_base + (c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// Thread organisation.  Each page is split into kGroups groups of 16 tokens.
// Tensor-core variant: 8 consumer warps; warp w takes token group w % 4 and
// output dims [128 * (w / 4), +128): the two warps of a group compute the same
// grouped scores (QK) and each accumulates half of P V, so every SM
// sub-partition runs two consumer warps whose latencies overlap.
// CUDA-core variant: 4 consumer warps, one per token group, all dims.
// ---------------------------------------------------------------------------
template <bool kTensorCores>
struct Shape {
  static constexpr int kConsumerWarps = kTensorCores ? 8 : 4;
  static constexpr int kConsumers = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumers + 32;  // + one producer warp
};
constexpr int kDimHalves = 2;
constexpr int kHalfD = kD / kDimHalves;

// Tensor-core accumulators of one warp: o[n][0..1] = head row (lane/4),
// dims 128*half + 8n + 2(lane%4) + {0,1}; each page adds its P_hi and P_lo
// products for those dims (mma rows lane/4 and lane/4 + 8).
struct MmaState {
  float o[kHalfD / 8][2];
  float m;  // reference of this lane's head row (log2 domain, multiple of 8)
  float l;  // this lane's share of the row sum (quad-reduced at the end)
};

struct FmaState {
  float o[kMaxG][8];  // head h, dims 8*lane .. 8*lane+7
  float m[kMaxG];
  float l[kMaxG];
};

// Called by every consumer thread once it has stored `done` parts of the
// tile outputs of (request b, kv head g): a whole unsplit (or empty) unit
// counts 1, a slice of a split unit 1.  With the fused merge, the CTA whose
// parts complete the pair's count (`total`, over its T tiles) merges the T
// tiles for the G query heads of g with the merge kernel's own row routine
// (same bits as lse_merge over those partials), then resets the counter for
// the next call.
template <int kMaxUnits, int kConsumers, int kConsumerWarps>
__device__ __forceinline__ void finish_unit(const Params<kMaxUnits>& p, const Shared& sh, int b,
                                            int g, int ct, int warp, int lane, int done,
                                            int total) {
  if (p.m_out == nullptr) return;
  ptx::named_barrier(1, kConsumers);       // this CTA's outputs are all stored
  if (ct == 0) {
    const int prev = ptx::atomic_add_acq_rel_gpu(p.req_counters + b * p.Hkv + g, done);
    *sh.fin_flag = (prev + done == total) ? 1 : 0;
  }
  ptx::named_barrier(1, kConsumers);
  if (*sh.fin_flag) {
    for (int r = warp; r < p.G; r += kConsumerWarps) {
      const int h = g * p.G + r;
      mergerow::merge_row<true>(p.out, p.lse, b * p.T, p.T, p.Hq, h, kD,
                                p.m_out + ((size_t)b * p.Hq + h) * kD,
                                p.m_lse + (size_t)b * p.Hq + h, lane);
    }
    if (ct == 0) p.req_counters[b * p.Hkv + g] = 0;
  }
  ptx::named_barrier(1, kConsumers);
}

// Merges output float4s [o_lo, o_hi) of a split unit (o = row * kD/4 + float4
// column) from its n partials (slots part_base ..): the unit's tile output and,
// at column 0, its LSE.  The same merge rule as the tile merge: common
// reference = max partial reference, weights exactly 2^(m_c - max), output =
// weighted sum / summed weights.  Each output is taken by a team of t lanes
// (t a power of two, as large as one pass over the outputs allows); lane j
// adds partials j, j + t, ... in that order, and the team adds its lanes'
// sums by a butterfly.  The arithmetic depends only on n and the range, never
// on which CTA runs it, so slices merged by different CTAs, or twice, give
// the same bits.  All of a lane's loads are issued before its arithmetic.
template <int kMaxUnits, int kConsumers>
__device__ __forceinline__ void merge_split_slice(const Params<kMaxUnits>& p, int part_base, int n,
                                                  int o_lo, int o_hi, size_t orow0, int ct) {
  constexpr int kVec = kD / 4;
  const int len = o_hi - o_lo;
  int t = 32;
  while (t > 1 && kConsumers / t < len && (n + t / 2 - 1) / (t / 2) <= kMaxPartsPerLane) t >>= 1;
  const int n_teams = kConsumers / t;
  const int j = ct & (t - 1);
  const int team = ct / t;
  const float2* pml = reinterpret_cast<const float2*>(p.part_ml) + (size_t)part_base * kMaxG;
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + (size_t)part_base * kMaxG * kVec;
  for (int base = o_lo; base < o_hi; base += n_teams) {
    const int o = base + team;
    const bool have = o < o_hi;
    const int row = have ? o / kVec : 0;
    const int dv = have ? o - row * kVec : 0;
    float2 ml[kMaxPartsPerLane];
    float4 v[kMaxPartsPerLane];
#pragma unroll
    for (int k = 0; k < kMaxPartsPerLane; ++k) {
      const int c = j + k * t;
      if (have && c < n) {
        ml[k] = __ldcg(pml + (size_t)c * kMaxG + row);
        v[k] = __ldcg(po + ((size_t)c * kMaxG + row) * kVec + dv);
      } else {
        ml[k] = make_float2(-INFINITY, 0.f);
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float big_m = -INFINITY;
    int nan = 0;
#pragma unroll
    for (int k = 0; k < kMaxPartsPerLane; ++k) {
      big_m = fmaxf(big_m, ml[k].x);
      nan |= (ml[k].x != ml[k].x);
    }
    for (int off = t >> 1; off > 0; off >>= 1) {
      big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, off));
      nan |= __shfl_xor_sync(0xffffffffu, nan, off);
    }
    float l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kMaxPartsPerLane; ++k) {
      const float a = ref_weight(ml[k].x, big_m);
      l = fmaf(a, ml[k].y, l);
      acc.x = fmaf(a, v[k].x, acc.x);
      acc.y = fmaf(a, v[k].y, acc.y);
      acc.z = fmaf(a, v[k].z, acc.z);
      acc.w = fmaf(a, v[k].w, acc.w);
    }
    for (int off = t >> 1; off > 0; off >>= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if (have && j == 0) {
      const size_t orow = orow0 + row;
      const float qnan = __int_as_float(0x7fc00000);
      reinterpret_cast<float4*>(p.out + orow * kD)[dv] =
          nan ? make_float4(qnan, qnan, qnan, qnan)
              : make_float4(acc.x / l, acc.y / l, acc.z / l, acc.w / l);
      if (dv == 0) p.lse[orow] = nan ? qnan : lse_of(big_m, l);
    }
  }
}

// Thread 0 of a CTA that has arrived at split unit `arrival` in generation
// `gen`, with this unit's segment as its last: waits until every CTA of the
// unit has arrived (the count reaches n, or the last CTA has already opened
// the next generation), so every partial is stored and visible.  If no other
// CTA of the unit arrives for slice_wait_ns while some have not, it records
// itself as a leaver (the last CTA then merges every slice) and returns false.
__device__ __forceinline__ bool wait_unit_complete(unsigned long long* arrival, unsigned gen,
                                                   int n, uint64_t slice_wait_ns,
                                                   uint64_t wait_limit_ns, int32_t* status) {
  const uint64_t t0 = ptx::globaltimer_ns();
  uint64_t t_seen = t0;
  int seen = -1;
  while (true) {
    // Acquire polls: the one that sees every arrival synchronises with all
    // of them (each arrival is an acquire-release add, and the opening add
    // is in the release sequence of each).  Measured against relaxed polls
    // followed by a fence: 25.33 -> 24.96 us per launch at 1 x 32,768 tokens,
    // 78.17 -> 77.84 us with 4 x 31,744.
    const unsigned long long v = ptx::load_acquire_gpu(arrival);
    const int count = (int)(v & 0xffffu);
    if ((unsigned)(v >> 32) != gen || count == n) return true;
    const uint64_t now = ptx::globaltimer_ns();
    if (count != seen) {
      seen = count;
      t_seen = now;
    }
    if (now - t_seen > slice_wait_ns && ptx::atomic_cas_gpu(arrival, v, v + (1ull << 16)) == v)
      return false;
    if (now - t0 > wait_limit_ns) {
      atomicOr(status, PA_STATUS_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int kMaxUnits, bool kTensorCores>
__global__ void __launch_bounds__(Shape<kTensorCores>::kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap,
                        const __grid_constant__ Params<kMaxUnits> p) {
  constexpr int kConsumerWarps = Shape<kTensorCores>::kConsumerWarps;
  constexpr int kConsumers = Shape<kTensorCores>::kConsumers;
  extern __shared__ uint8_t smem_raw[];
  const Shared sh = carve(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int Hkv = p.Hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(sh.full_bar + 8 * s, 1);
      ptx::mbar_init(sh.empty_bar + 8 * s, kConsumerWarps);
      sh.poison[s] = 0;
    }
    *sh.abort_flag = 0;
    ptx::mbar_init_fence();
  }
  if (warp == kConsumerWarps && lane == 0) ptx::prefetch_tensormap(&tmap);
  __syncthreads();
  // Everything above touches only parameters and shared memory; from here on
  // the kernel reads what earlier kernels in the stream wrote.  With kv_ready
  // the producer warp defers this wait until its ring is full (below).
  const bool early_kv = p.kv_ready != 0 && warp == kConsumerWarps;
  if (!early_kv) ptx::grid_dependency_wait();

  // New-token rows: CTA b % grid stores request b's row into its page.  A CTA
  // of this launch may stream that page before or after the store, so every
  // consumer substitutes the row in shared memory instead of reading it from
  // the pool.  (Storing from the producer warp after its loads measured
  // slightly slower.)
  if (p.new_rows != nullptr && warp < kConsumerWarps) {
    for (int b = blockIdx.x; b < p.n_requests; b += p.grid) {
      const int pos = p.positions[b];
      const int lp = pos >= 0 ? pos / kPage : -1;
      const long long page = (lp >= 0 && lp < p.max_pages)
                                 ? (long long)p.page_table[(size_t)b * p.max_pages + lp] : -1;
      if (page < 0 || page >= p.pool_pages) {
        if (threadIdx.x == 0) atomicOr(p.status, PA_STATUS_BAD_ROW);
        continue;
      }
      const uint4* src = reinterpret_cast<const uint4*>(p.new_rows + (size_t)b * p.row_elems);
      uint4* dst = reinterpret_cast<uint4*>(p.pool + ((size_t)page * kPage + pos % kPage) *
                                                         (size_t)p.row_elems);
      for (int i = threadIdx.x; i < p.row_elems / 8; i += kConsumers) dst[i] = __ldg(src + i);
    }
  }


  // Flattened page range of this CTA (a launch holds fewer than 2^31 pages).
  const int cta_start = static_cast<int>((long long)blockIdx.x * p.total_pages / p.grid);
  const int cta_end = static_cast<int>((long long)(blockIdx.x + 1) * p.total_pages / p.grid);

  // ======================= producer warp =======================
  if (warp == kConsumerWarps) {
    int it = 0;
    bool ok = true;
    // Every page is read once: its lines go first when L2 needs room
    // (measured +2% on the bench step against the default policy).
    const uint64_t pol = ptx::policy_evict_first();
    for (int u = first_unit(p, cta_start); ok && u < p.n_units && p.units[u].page_first < cta_end;
         ++u) {
      const Unit U = p.units[u];
      const int np = unit_pages(U.tok_start, U.tok_end);
      if (np == 0) continue;
      const int pf = U.page_first;
      const int lo = max(cta_start, pf) - pf;
      const int hi = min(cta_end, pf + np) - pf;
      if (hi <= lo) continue;   // only the unit's segment charge falls in this range
      const int bt = U.bt_g / Hkv;
      const int g = U.bt_g - bt * Hkv;
      const int b = bt / p.T;
      const int32_t* prow = p.page_table + (size_t)b * p.max_pages + U.tok_start / kPage;
      const int xk = g * kD;
      const int xv = (Hkv + g) * kD;
      for (int base = lo; ok && base < hi; base += 32) {
        const int cnt = min(32, hi - base);
        const int my_pid = lane < cnt ? __ldg(prow + base + lane) : 0;
        for (int j = 0; j < cnt; ++j) {
          const int pid = __shfl_sync(0xffffffffu, my_pid, j);
          // Early loads only fill the ring: the producer waits for earlier
          // kernels before its first (bounded) wait on a consumer release,
          // which would otherwise count the consumers' own dependency wait.
          if (early_kv && it == kStages) ptx::grid_dependency_wait();
          int good = 1;
          if (lane == 0) {
            const int s = it % kStages;
            if (it >= kStages) {
              good = ptx::mbar_wait_bounded(sh.empty_bar + 8 * s, ((it / kStages) - 1) & 1,
                                            p.wait_limit_ns) ? 1 : 0;
            }
            if (good) {
              const bool bad = pid < 0 || (long long)pid >= p.pool_pages;
              if (bad) atomicOr(p.status, PA_STATUS_BAD_PAGE);
              sh.poison[s] = bad ? 1 : 0;
              const int y = (bad ? 0 : pid) * kPage;
              const uint32_t full = sh.full_bar + 8 * s;
              const uint32_t dst = ptx::smem_addr(sh.stages + s * kStageBytes);
              if (it != p.stall_iteration || blockIdx.x != 0) {
                ptx::mbar_arrive_expect_tx(full, kStageBytes);
#pragma unroll
                for (int c = 0; c < kD / kBoxCols; ++c) {
                  ptx::tma_load_2d_hint(dst + c * kBoxBytes, &tmap, xk + c * kBoxCols, y, full,
                                        pol);
                  ptx::tma_load_2d_hint(dst + kHalfBytes + c * kBoxBytes, &tmap,
                                        xv + c * kBoxCols, y, full, pol);
                }
              }
            } else {
              atomicOr(p.status, PA_STATUS_TIMEOUT);
              *sh.abort_flag = 1;
            }
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          ++it;
        }
      }
    }
    // Every page of this CTA is requested: the next kernel in the stream may
    // start its prologue (it waits for this grid before reading our output).
    if (lane == 0) ptx::launch_dependents();
    if (!ok && lane == 0) {
      // Let the copies already issued land before the CTA can exit.
      for (int k = max(0, it - kStages); k < it; ++k) {
        ptx::mbar_wait_bounded(sh.full_bar + 8 * (k % kStages), (k / kStages) & 1,
                               p.wait_limit_ns);
      }
    }
    return;
  }

  // ======================= consumer warps =======================
  const int ct = threadIdx.x;      // 0 .. kConsumers-1
  const int tg = warp % kGroups;   // token group of this warp
  const int dh = warp / kGroups;   // dim half (tensor-core variant)
  const int gr = lane >> 2;        // head row inside the group (tensor-core layout)
  const int tq = lane & 3;

  // Empty units: output 0, LSE -inf.
  for (int u = blockIdx.x; u < p.n_units; u += p.grid) {
    const Unit U = p.units[u];
    if (unit_pages(U.tok_start, U.tok_end) != 0) continue;
    const int bt = U.bt_g / Hkv;
    const int g = U.bt_g - bt * Hkv;
    for (int idx = ct; idx < G * kD; idx += kConsumers) {
      const int row = idx / kD;
      const int d = idx - row * kD;
      p.out[((size_t)bt * p.Hq + g * G + row) * kD + d] = 0.f;
      if (d == 0) p.lse[(size_t)bt * p.Hq + g * G + row] = -INFINITY;
    }
    finish_unit<kMaxUnits, kConsumers, kConsumerWarps>(p, sh, bt / p.T, g, ct, warp, lane, 1,
                                                       U.pair_total);
  }

  int it = 0;
  bool ok = true;
  for (int u = first_unit(p, cta_start); ok && u < p.n_units && p.units[u].page_first < cta_end;
       ++u) {
    const Unit U = p.units[u];
    const int np = unit_pages(U.tok_start, U.tok_end);
    if (np == 0) continue;
    const int pf = U.page_first;
    const int lo = max(cta_start, pf) - pf;
    const int hi = min(cta_end, pf + np) - pf;
    if (hi <= lo) continue;
    const int bt = U.bt_g / Hkv;
    const int g = U.bt_g - bt * Hkv;
    const int b = bt / p.T;
    const int first_page_tok = (U.tok_start / kPage) * kPage;
    int poisoned = 0;
    // The new token of this request, if it falls in this segment's pages:
    // its K slice (chunk `lane`) and V slice (chunk `lane`) of kv head g.
    // The position's load is issued before the Q loads below and the row's
    // loads go out with them, so neither adds a round trip to the segment's
    // start.
    const int pos = p.new_rows != nullptr ? __ldg(p.positions + b) : -1;
    int sub_pos = -1;
    uint4 sub_k = make_uint4(0u, 0u, 0u, 0u), sub_v = make_uint4(0u, 0u, 0u, 0u);
    auto load_new_row = [&]() {
      if (pos >= max(U.tok_start, first_page_tok + lo * kPage) &&
          pos < min(U.tok_end, first_page_tok + hi * kPage)) {
        sub_pos = pos;
        const uint4* row = reinterpret_cast<const uint4*>(p.new_rows + (size_t)b * p.row_elems);
        sub_k = __ldg(row + (g * kD) / 8 + lane);
        sub_v = __ldg(row + ((Hkv + g) * kD) / 8 + lane);
      }
    };


    if constexpr (kTensorCores) {
      // ---- Q fragments (A operand rows = heads; rows 8..15 stay zero) ----
      // Staged once per segment in the exchange area (free until the
      // publish below): qfrag[kk][lane] = {a0, a2} of k-step kk.
      uint2* qfrag = reinterpret_cast<uint2*>(sh.xo);
      {
        const bool live = gr < G;
        const __nv_bfloat16* qrow = p.q + ((size_t)b * p.Hq + g * G + (live ? gr : 0)) * kD;
#pragma unroll
        for (int j = 0; j < kD / 16 / kConsumerWarps; ++j) {
          const int kk = warp * (kD / 16 / kConsumerWarps) + j;
          uint2 v;
          v.x = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * tq)) : 0u;
          v.y = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * tq)) : 0u;
          qfrag[kk * 32 + lane] = v;
        }
      }
      // The new token's K and V slices (32 16-byte chunks each) go beside
      // the Q fragments, loaded with them whether or not the token falls in
      // this segment (its position arrives with them), so that neither the
      // segment's start nor the page loop's registers pay for them.
      uint4* xrow = reinterpret_cast<uint4*>(sh.xo) + kD / 16 * 32 / 2;
      if (p.new_rows != nullptr && ct < 64) {
        const uint4* row = reinterpret_cast<const uint4*>(p.new_rows + (size_t)b * p.row_elems);
        xrow[ct] = __ldg(row + ((ct < 32 ? g : Hkv + g) * kD) / 8 + (ct & 31));
      }
      if (pos >= max(U.tok_start, first_page_tok + lo * kPage) &&
          pos < min(U.tok_end, first_page_tok + hi * kPage))
        sub_pos = pos;
      ptx::named_barrier(1, kConsumers);
      MmaState st;
#pragma unroll
      for (int n = 0; n < kHalfD / 8; ++n) st.o[n][0] = st.o[n][1] = 0.f;
      st.m = -INFINITY;
      st.l = 0.f;

      const int r8 = lane & 7;
      const int mi = lane >> 3;
      const uint32_t k_lane = (16 * tg + (mi >> 1) * 8 + r8) * 128;
      const int sel_k = mi & 1;
      const uint32_t v_lane = kHalfBytes + (16 * tg + (mi & 1) * 8 + r8) * 128;
      const int sel_v = mi >> 1;

      for (int lp = lo; lp < hi; ++lp, ++it) {
        const int s = it % kStages;
        if (!ptx::mbar_wait_bounded(sh.full_bar + 8 * s, (it / kStages) & 1, p.wait_limit_ns)) {
          if (lane == 0) {
            atomicOr(p.status, PA_STATUS_TIMEOUT);
            *sh.abort_flag = 1;
          }
          ok = false;
          break;
        }
        poisoned |= sh.poison[s];
        const int page_tok = first_page_tok + lp * kPage;
        const int vlo = max(U.tok_start, page_tok);
        const int vhi = min(U.tok_end, page_tok + kPage);
        const int tb = page_tok + 16 * tg;
        const uint32_t stage = ptx::smem_addr(sh.stages + s * kStageBytes);
        if (sub_pos >= tb && sub_pos < tb + 16) {
          // The new token's row: both warps of the group write its K slice
          // (same bytes), each its own half of the V slice.
          const int r = sub_pos - page_tok;
          put_row_chunk(stage, r, lane, xrow[lane]);
          if ((lane >> 4) == dh) put_row_chunk(stage + kHalfBytes, r, lane, xrow[32 + lane]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
        }
        if (tb + 16 > vlo && tb < vhi) {
          if (tb < vlo || tb + 16 > vhi) {
            // Rows of this group outside the tile: zero this warp's half of
            // their V so that a non-finite value there cannot reach P V.
            for (int r = 0; r < 16; ++r) {
              const int tok = tb + r;
              if (tok >= vlo && tok < vhi) continue;
              if (lane < 16) {
                const uint32_t a = stage + kHalfBytes + (2 * dh + (lane >> 3)) * kBoxBytes +
                                   (16 * tg + r) * 128 + (lane & 7) * 16;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u)
                             : "memory");
              }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
          }
          // ---- S = Q K^T for the group's 16 tokens (two 8-token n-tiles) ----
          // Even and odd k-steps accumulate separately: four independent
          // MMA chains instead of two.
          float s0[4] = {0.f, 0.f, 0.f, 0.f}, s0o[4] = {0.f, 0.f, 0.f, 0.f};
          float s1[4] = {0.f, 0.f, 0.f, 0.f}, s1o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const int chunk = 2 * kk + sel_k;
            const uint32_t addr =
                stage + (chunk >> 3) * kBoxBytes + k_lane + (((chunk & 7) ^ r8) << 4);
            uint32_t b0, b1, b2, b3;
            ptx::ldmatrix_x4(addr, b0, b1, b2, b3);
            const uint2 qa = qfrag[kk * 32 + lane];
            if (kk & 1) {
              ptx::mma_bf16_16816(s0o, qa.x, 0u, qa.y, 0u, b0, b1);
              ptx::mma_bf16_16816(s1o, qa.x, 0u, qa.y, 0u, b2, b3);
            } else {
              ptx::mma_bf16_16816(s0, qa.x, 0u, qa.y, 0u, b0, b1);
              ptx::mma_bf16_16816(s1, qa.x, 0u, qa.y, 0u, b2, b3);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            s0[k] += s0o[k];
            s1[k] += s1o[k];
          }
          // ---- masked online softmax (log2 domain, reference on multiples of 8) ----
          const bool live = gr < G;
          const int j0 = tb + 2 * tq;
          float x[4];
          x[0] = (live && j0 >= vlo && j0 < vhi) ? s0[0] * p.scale_log2 : -INFINITY;
          x[1] = (live && j0 + 1 >= vlo && j0 + 1 < vhi) ? s0[1] * p.scale_log2 : -INFINITY;
          x[2] = (live && j0 + 8 >= vlo && j0 + 8 < vhi) ? s1[0] * p.scale_log2 : -INFINITY;
          x[3] = (live && j0 + 9 >= vlo && j0 + 9 < vhi) ? s1[1] * p.scale_log2 : -INFINITY;
          float bm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
          const bool need = bm > st.m;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(st.m, ref_ceil(bm));
            const float alpha = ref_weight(st.m, m_new);
#pragma unroll
            for (int n = 0; n < kHalfD / 8; ++n) {
              st.o[n][0] *= alpha;
              st.o[n][1] *= alpha;
            }
            st.l *= alpha;
            st.m = m_new;
          }
          const float mu = (st.m == -INFINITY) ? 0.f : st.m;
          float pr[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) pr[k] = ptx::ex2(x[k] - mu);
          st.l += (pr[0] + pr[1]) + (pr[2] + pr[3]);
          __nv_bfloat16 ph[4], pl[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ph[k] = __float2bfloat16_rn(pr[k]);
            pl[k] = __float2bfloat16_rn(pr[k] - __bfloat162float(ph[k]));
          }
          const uint32_t pa0 = ptx::pack_bf16x2(ph[0], ph[1]);
          const uint32_t pa1 = ptx::pack_bf16x2(pl[0], pl[1]);
          const uint32_t pa2 = ptx::pack_bf16x2(ph[2], ph[3]);
          const uint32_t pa3 = ptx::pack_bf16x2(pl[2], pl[3]);
          // ---- O += P V over this warp's dim half ----
          // Each page's product starts from a zero accumulator and is added
          // to O in fp32 with round-to-nearest, so the long running sum does
          // not inherit the tensor core's accumulation rounding.
#pragma unroll
          for (int nd2 = 0; nd2 < kHalfD / 16; ++nd2) {
            const int chunk = (kHalfD / 8) * dh + 2 * nd2 + sel_v;
            const uint32_t addr =
                stage + (chunk >> 3) * kBoxBytes + v_lane + (((chunk & 7) ^ r8) << 4);
            uint32_t b0, b1, b2, b3;
            ptx::ldmatrix_x4_trans(addr, b0, b1, b2, b3);
            float t0[4] = {0.f, 0.f, 0.f, 0.f};
            float t1[4] = {0.f, 0.f, 0.f, 0.f};
            ptx::mma_bf16_16816(t0, pa0, pa1, pa2, pa3, b0, b1);
            ptx::mma_bf16_16816(t1, pa0, pa1, pa2, pa3, b2, b3);
            // Rows 0..7 (P_hi) and 8..15 (P_lo) of the same head and dims
            // add up to the page's product with ~16-bit probabilities.
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              st.o[2 * nd2][k] += t0[k] + t0[k + 2];
              st.o[2 * nd2 + 1][k] += t1[k] + t1[k + 2];
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sh.empty_bar + 8 * s);
      }
      // ---- publish this warp's state for the CTA-level combine ----
      ptx::named_barrier(1, kConsumers);  // every warp is done with qfrag
      st.l += __shfl_xor_sync(0xffffffffu, st.l, 1);
      st.l += __shfl_xor_sync(0xffffffffu, st.l, 2);
      if (gr < G) {
        float* row = sh.xo + (tg * kMaxG + gr) * kXRow + kHalfD * dh;
#pragma unroll
        for (int n = 0; n < kHalfD / 8; ++n) {
          *reinterpret_cast<float2*>(row + 8 * n + 2 * tq) =
              make_float2(st.o[n][0], st.o[n][1]);
        }
        if (tq == 0 && dh == 0) {
          sh.xml[(tg * kMaxG + gr) * 2 + 0] = poisoned ? __int_as_float(0x7fc00000) : st.m;
          sh.xml[(tg * kMaxG + gr) * 2 + 1] = st.l;
        }
      }
    } else {
      // ---------------- CUDA-core variant ----------------
      load_new_row();
      FmaState st;
      float qf[kMaxG][8];
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
              p.q + ((size_t)b * p.Hq + g * G + h) * kD + 8 * lane));
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            qf[h][2 * i] = ptx::bf16_lo_to_f32(w4[i]);
            qf[h][2 * i + 1] = ptx::bf16_hi_to_f32(w4[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) qf[h][i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) st.o[h][i] = 0.f;
        st.m[h] = -INFINITY;
        st.l[h] = 0.f;
      }
      const uint32_t lane_box = (lane >> 3) * kBoxBytes;
      const int lane_chunk = lane & 7;
      for (int lp = lo; lp < hi; ++lp, ++it) {
        const int s = it % kStages;
        if (!ptx::mbar_wait_bounded(sh.full_bar + 8 * s, (it / kStages) & 1, p.wait_limit_ns)) {
          if (lane == 0) {
            atomicOr(p.status, PA_STATUS_TIMEOUT);
            *sh.abort_flag = 1;
          }
          ok = false;
          break;
        }
        poisoned |= sh.poison[s];
        const int page_tok = first_page_tok + lp * kPage;
        const int vlo = max(U.tok_start, page_tok);
        const int vhi = min(U.tok_end, page_tok + kPage);
        const int tb = page_tok + 16 * tg;
        const uint32_t stage = ptx::smem_addr(sh.stages + s * kStageBytes);
        if (sub_pos >= tb && sub_pos < tb + 16) {
          const int r = sub_pos - page_tok;
          put_row_chunk(stage, r, lane, sub_k);
          put_row_chunk(stage + kHalfBytes, r, lane, sub_v);
          ptx::fence_proxy_async_smem();
          __syncwarp();
        }
        const int r_lo = max(0, vlo - tb);
        const int r_hi = min(16, vhi - tb);
        for (int r = r_lo; r < r_hi; ++r) {
          const int row = 16 * tg + r;
          const uint32_t ka = stage + lane_box + row * 128 + ((lane_chunk ^ (row & 7)) << 4);
          uint32_t k4[4], v4[4];
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(k4[0]), "=r"(k4[1]), "=r"(k4[2]), "=r"(k4[3])
                       : "r"(ka));
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v4[0]), "=r"(v4[1]), "=r"(v4[2]), "=r"(v4[3])
                       : "r"(ka + kHalfBytes));
          float kf[8], vf[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            kf[2 * i] = ptx::bf16_lo_to_f32(k4[i]);
            kf[2 * i + 1] = ptx::bf16_hi_to_f32(k4[i]);
            vf[2 * i] = ptx::bf16_lo_to_f32(v4[i]);
            vf[2 * i + 1] = ptx::bf16_hi_to_f32(v4[i]);
          }
          float x[kMaxG];
#pragma unroll
          for (int h = 0; h < kMaxG; ++h) {
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaf(qf[h][i], kf[i], a);
            x[h] = a;
          }
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
            for (int h = 0; h < kMaxG; ++h) x[h] += __shfl_xor_sync(0xffffffffu, x[h], off);
          }
          bool need = false;
#pragma unroll
          for (int h = 0; h < kMaxG; ++h) {
            x[h] = h < G ? x[h] * p.scale_log2 : -INFINITY;
            need |= x[h] > st.m[h];
          }
          if (need) {  // uniform: every lane holds the same reduced scores
#pragma unroll
            for (int h = 0; h < kMaxG; ++h) {
              const float m_new = fmaxf(st.m[h], ref_ceil(x[h]));
              const float alpha = ref_weight(st.m[h], m_new);
#pragma unroll
              for (int i = 0; i < 8; ++i) st.o[h][i] *= alpha;
              st.l[h] *= alpha;
              st.m[h] = m_new;
            }
          }
#pragma unroll
          for (int h = 0; h < kMaxG; ++h) {
            const float pr = ptx::ex2(x[h] - (st.m[h] == -INFINITY ? 0.f : st.m[h]));
            st.l[h] += pr;
#pragma unroll
            for (int i = 0; i < 8; ++i) st.o[h][i] = fmaf(pr, vf[i], st.o[h][i]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sh.empty_bar + 8 * s);
      }
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h < G) {
          float* row = sh.xo + (tg * kMaxG + h) * kXRow + 8 * lane;
          *reinterpret_cast<float4*>(row) =
              make_float4(st.o[h][0], st.o[h][1], st.o[h][2], st.o[h][3]);
          *reinterpret_cast<float4*>(row + 4) =
              make_float4(st.o[h][4], st.o[h][5], st.o[h][6], st.o[h][7]);
          if (lane == 0) {
            sh.xml[(tg * kMaxG + h) * 2 + 0] = poisoned ? __int_as_float(0x7fc00000) : st.m[h];
            sh.xml[(tg * kMaxG + h) * 2 + 1] = st.l[h];
          }
        }
      }
    }

    // ============ CTA-level combine of the kGroups token groups ============
    ptx::named_barrier(1, kConsumers);
    if (!ok || *sh.abort_flag) {
      ok = false;
      break;
    }
    const bool single = U.n_parts == 1;
    int slot = 0;
    if (!single) slot = U.part_base + (int)blockIdx.x - cta_of(pf, p.total_pages, p.grid);
    // Four consecutive output dims per thread and step (float4 exchange
    // reads and stores): the combine sits on the critical path of the CTA
    // that finishes last.
    constexpr int kDimVec = kD / 4;
    for (int idx = ct; idx < G * kDimVec; idx += kConsumers) {
      const int row = idx / kDimVec;
      const int dv = idx - row * kDimVec;
      float mw[kGroups];
      float big_m = -INFINITY;
      bool nan = false;
#pragma unroll
      for (int w2 = 0; w2 < kGroups; ++w2) {
        mw[w2] = sh.xml[(w2 * kMaxG + row) * 2];
        nan |= (mw[w2] != mw[w2]);
        big_m = fmaxf(big_m, mw[w2]);
      }
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kGroups; ++w2) {
        const float a = ref_weight(mw[w2], big_m);
        const float4 x =
            *reinterpret_cast<const float4*>(sh.xo + (w2 * kMaxG + row) * kXRow + 4 * dv);
        o.x = fmaf(a, x.x, o.x);
        o.y = fmaf(a, x.y, o.y);
        o.z = fmaf(a, x.z, o.z);
        o.w = fmaf(a, x.w, o.w);
        l = fmaf(a, sh.xml[(w2 * kMaxG + row) * 2 + 1], l);
      }
      if (nan) big_m = __int_as_float(0x7fc00000);
      if (single) {
        const size_t orow = (size_t)bt * p.Hq + g * G + row;
        reinterpret_cast<float4*>(p.out + orow * kD)[dv] =
            nan ? make_float4(big_m, big_m, big_m, big_m)
                : make_float4(o.x / l, o.y / l, o.z / l, o.w / l);
        if (dv == 0) p.lse[orow] = nan ? big_m : lse_of(big_m, l);
      } else {
        reinterpret_cast<float4*>(p.part_o + ((size_t)slot * kMaxG + row) * kD)[dv] = o;
        if (dv == 0) {
          p.part_ml[((size_t)slot * kMaxG + row) * 2 + 0] = big_m;
          p.part_ml[((size_t)slot * kMaxG + row) * 2 + 1] = l;
        }
      }
    }
    if (!single) {
      // Split unit: CTAs k0 .. k1 each stored a partial.  The barrier orders
      // every thread's partial before thread 0's acquire-release arrival,
      // which publishes it at device scope.  CTAs k0 .. k0 + S - 1 (S <= n - 1:
      // their page ranges end inside this unit, so it is their last segment)
      // wait until all n have arrived and each merges one of S slices of the
      // unit's outputs, so the merge is spread over S SMs instead of loading
      // every partial into one; the last CTA to arrive resets the count and
      // opens the word's next generation for the next call.  A CTA that gave
      // up waiting leaves its slice to the last CTA, which then merges every
      // slice (a slice merged twice gets the same bits).  The other CTAs
      // leave at once.
      const int n = U.n_parts;
      const int S = split_slices(n);
      const int rank = (int)blockIdx.x - cta_of(pf, p.total_pages, p.grid);
      const bool participant = rank < S;
      unsigned long long* arrival = p.arrivals + u;
      ptx::named_barrier(1, kConsumers);
      if (ct == 0) {
        const unsigned long long prev = ptx::atomic_add_acq_rel_gpu(arrival, 1ull);
        const int arrived = (int)(prev & 0xffffu) + 1;
        int mode = 0;  // 0: no slice here, 1: this CTA's slice, 2: every slice
        int leavers = 0;
        if (arrived == n) {
          leavers = (int)((prev >> 16) & 0xffffu);
          // Count and leavers back to zero, generation + 1 (a plain add: a
          // waiting CTA that reads it still acquires every arrival, which
          // it follows in the word's order of modifications).
          ptx::red_add_relaxed_gpu(arrival, (1ull << 32) -
                                                ((unsigned long long)leavers << 16) -
                                                (unsigned long long)n);
          mode = leavers ? 2 : (participant ? 1 : 0);
          if (leavers) atomicAdd(p.status + 1, leavers);   // diagnostic count, not an error
        } else if (participant) {
          mode = wait_unit_complete(arrival, (unsigned)(prev >> 32), n, p.slice_wait_ns,
                                    p.wait_limit_ns, p.status) ? 1 : 0;
        }
        sh.merge_info[0] = mode;
        sh.merge_info[1] = leavers;
      }
      ptx::named_barrier(1, kConsumers);
      const int mode = sh.merge_info[0];
      if (mode != 0) {
        const int n_out = G * (kD / 4);
        for (int sl = mode == 2 ? 0 : rank; sl < (mode == 2 ? S : rank + 1); ++sl) {
          merge_split_slice<kMaxUnits, kConsumers>(
              p, U.part_base, n, (int)((long long)sl * n_out / S),
              (int)((long long)(sl + 1) * n_out / S), (size_t)bt * p.Hq + g * G, ct);
        }
        // Each slice counts once toward the pair's tile count (the slices
        // of leavers are counted by the last CTA, which merged them).
        const int done = mode == 2 ? sh.merge_info[1] + (participant ? 1 : 0) : 1;
        finish_unit<kMaxUnits, kConsumers, kConsumerWarps>(p, sh, b, g, ct, warp, lane, done,
                                                           U.pair_total);
      }
    } else {
      finish_unit<kMaxUnits, kConsumers, kConsumerWarps>(p, sh, b, g, ct, warp, lane, 1,
                                                         U.pair_total);
    }
    ptx::named_barrier(1, kConsumers);
  }
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Partial slots reserved: one per unit of a launch plus one per CTA (a CTA
// adds at most one split point), with room for grids up to 1,024 CTAs.
size_t part_slots(int B, int T, int Hkv) {
  const long long units = (long long)B * T * Hkv;
  return (size_t)std::min<long long>(units, kMaxUnitsLarge) + 1024;
}

// Per (request, kv head) counters of finished tiles for the fused merge.
size_t request_counter_bytes(int B, int Hkv) {
  return ((size_t)B * Hkv * 4 + 255) / 256 * 256;
}

size_t workspace_bytes(int B, int T, int Hkv) {
  return kStatusBytes + kCounterBytes + request_counter_bytes(B, Hkv) +
         part_slots(B, T, Hkv) * (kPartOBytes + kPartMLBytes);
}

template <int N, bool TC>
cudaError_t launch(const CUtensorMap& tmap, const Params<N>& prm, int grid, cudaStream_t stream) {
  static PerContext smem_limit;   // the attribute lives in the context
  cudaError_t e = smem_limit.apply([] {
    return cudaFuncSetAttribute(paged_decode_kernel<N, TC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  });
  if (e != cudaSuccess) return e;
  e = launch_dependent(paged_decode_kernel<N, TC>, dim3(grid), dim3(Shape<TC>::kThreads),
                       kSmemAlloc, stream, tmap, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int N, bool TC>
int launch_units(const CUtensorMap& tmap, const std::vector<Unit>& units, size_t u0, size_t n,
                 long long total_pages, int grid, const Params<kMaxUnitsSmall>& common,
                 cudaStream_t stream) {
  static_assert(N >= kMaxUnitsSmall, "");
  auto* prm = new Params<N>;
  std::memcpy(static_cast<void*>(prm), &common, offsetof(Params<kMaxUnitsSmall>, units));
  prm->n_units = static_cast<int>(n);
  prm->total_pages = total_pages;
  prm->grid = grid;
  std::memcpy(prm->units, units.data() + u0, n * sizeof(Unit));
  const cudaError_t e = launch<N, TC>(tmap, *prm, grid, stream);
  delete prm;
  if (e != cudaSuccess)
    return fail(PA_ERR_CUDA, "paged decode launch failed: %s", cudaGetErrorString(e));
  return PA_OK;
}

// Test hook state (paged_decode_attn_test_stall): consumed by the next run()
// on the calling thread.
thread_local int t_stall_iteration = -1;
thread_local unsigned long long t_wait_limit_ns = 0;
thread_local long long t_slice_wait_ns = -1;   // < 0: kSliceWaitNs

// Every host-side check of a decode call; enqueues nothing and touches no
// device state.  B * T == 0 passes (the call is then a no-op).
int check_args(const void* q, const void* pool, int64_t pool_pages, const int32_t* page_table,
               int max_pages, const int32_t* tiles, int B, int T, int n_q_heads,
               int n_kv_heads, int head_dim, float* out, float* lse, const void* workspace,
               size_t ws_bytes, const int32_t* positions, const void* new_rows, unsigned flags,
               const float* merged_out, const float* merged_lse) {
  PA_REQUIRE(B >= 0 && T >= 0, "B and T must be >= 0 (got %d, %d)", B, T);
  if ((long long)B * T == 0) return PA_OK;
  if (head_dim != kD)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d not built (supported: %d)", head_dim, kD);
  PA_REQUIRE(n_kv_heads >= 1 && n_q_heads >= n_kv_heads && n_q_heads % n_kv_heads == 0,
             "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)", n_q_heads,
             n_kv_heads);
  const int G = n_q_heads / n_kv_heads;
  if (G > kMaxG)
    return fail(PA_ERR_UNSUPPORTED, "group size %d above the supported %d", G, kMaxG);
  PA_REQUIRE(q && pool && page_table && tiles && out && lse && workspace,
             "null pointer argument");
  PA_REQUIRE(max_pages >= 1 && pool_pages >= 1, "max_pages and pool_pages must be >= 1");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(q) % 16 == 0, "q must be 16-byte aligned");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(pool) % 16 == 0, "pool must be 16-byte aligned");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(out) % 16 == 0, "out must be 16-byte aligned");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(workspace) % 256 == 0,
             "workspace must be 256-byte aligned");
  PA_REQUIRE(pool_pages * kPage < (1ll << 31), "pool too large for 32-bit row coordinates");
  PA_REQUIRE((long long)B * T * n_q_heads < (1ll << 31), "output too large");
  const size_t need = workspace_bytes(B, T, n_kv_heads);
  PA_REQUIRE(ws_bytes >= need, "workspace of %zu bytes is smaller than the %zu needed", ws_bytes,
             need);
  const long long max_tok = (long long)max_pages * kPage;
  for (long long i = 0; i < (long long)B * T; ++i) {
    const int s = tiles[2 * i], e = tiles[2 * i + 1];
    PA_REQUIRE(s >= 0 && s <= e && e <= max_tok,
               "tile %lld of request %lld is [%d, %d), outside [0, %lld]", i % T, i / T, s, e,
               max_tok);
  }
  PA_REQUIRE((flags & ~PA_DECODE_KV_READY) == 0, "unknown flags %#x", flags);
  PA_REQUIRE((merged_out == nullptr) == (merged_lse == nullptr),
             "merged_out and merged_lse go together");
  PA_REQUIRE(merged_out == nullptr || reinterpret_cast<uintptr_t>(merged_out) % 16 == 0,
             "merged_out must be 16-byte aligned");
  PA_REQUIRE((positions == nullptr) == (new_rows == nullptr),
             "positions and new_rows go together");
  PA_REQUIRE(new_rows == nullptr || reinterpret_cast<uintptr_t>(new_rows) % 16 == 0,
             "new_rows must be 16-byte aligned");
  return PA_OK;
}

int run(bool tensor_cores, const void* q, const void* pool, int64_t pool_pages,
        const int32_t* page_table, int max_pages, const int32_t* tiles, int B, int T,
        int n_q_heads, int n_kv_heads, int head_dim, float scale, float* out, float* lse,
        void* workspace, size_t ws_bytes, cudaStream_t stream,
        const int32_t* positions = nullptr, const void* new_rows = nullptr,
        unsigned flags = 0, float* merged_out = nullptr, float* merged_lse = nullptr) {
  clear_error();
  int rc0 = check_args(q, pool, pool_pages, page_table, max_pages, tiles, B, T, n_q_heads,
                       n_kv_heads, head_dim, out, lse, workspace, ws_bytes, positions, new_rows,
                       flags, merged_out, merged_lse);
  if (rc0 != PA_OK || (long long)B * T == 0) return rc0;
  const int G = n_q_heads / n_kv_heads;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");

  const int row_elems = 2 * n_kv_heads * kD;
  CUtensorMap tmap;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)pool_pages * kPage};
    const cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
    const cuuint32_t box[2] = {kBoxCols, kPage};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  }
  int sms = sm_count();
  if (sms <= 0) return fail(PA_ERR_CUDA, "cannot query the device's SM count");
  sms = std::min(sms, kMaxGrid);

  std::vector<Unit> units;
  units.reserve((size_t)B * T * n_kv_heads);
  // Kv-head-major order: the units of one kv head form a block of the page
  // sequence, and every block has the same unit sizes, so the CTAs at the
  // same offset of the n_kv_heads blocks stream the same physical pages (each
  // its head's slice of every row) at about the same time.
  for (int g = 0; g < n_kv_heads; ++g) {
    for (int bt = 0; bt < B * T; ++bt) {
      Unit u{};
      u.bt_g = bt * n_kv_heads + g;
      u.tok_start = tiles[2 * bt];
      u.tok_end = tiles[2 * bt + 1];
      units.push_back(u);
    }
  }

  Params<kMaxUnitsSmall> common{};
  common.q = static_cast<const __nv_bfloat16*>(q);
  common.page_table = page_table;
  common.out = out;
  common.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  common.status = reinterpret_cast<int32_t*>(ws);
  common.arrivals = reinterpret_cast<unsigned long long*>(ws + kStatusBytes);
  const size_t slots = part_slots(B, T, n_kv_heads);
  const size_t rc_bytes = request_counter_bytes(B, n_kv_heads);
  common.req_counters = reinterpret_cast<int32_t*>(ws + kStatusBytes + kCounterBytes);
  common.part_o = reinterpret_cast<float*>(ws + kStatusBytes + kCounterBytes + rc_bytes);
  common.part_ml = reinterpret_cast<float*>(ws + kStatusBytes + kCounterBytes + rc_bytes +
                                            slots * kPartOBytes);
  common.pool_pages = pool_pages;
  common.max_pages = max_pages;
  common.T = T;
  common.Hq = n_q_heads;
  common.Hkv = n_kv_heads;
  common.G = G;
  common.scale_log2 = scale * kLog2e;
  common.pool = static_cast<__nv_bfloat16*>(const_cast<void*>(pool));
  common.new_rows = static_cast<const __nv_bfloat16*>(new_rows);
  common.positions = positions;
  common.row_elems = row_elems;
  common.kv_ready = (flags & PA_DECODE_KV_READY) ? 1 : 0;
  common.m_out = merged_out;
  common.m_lse = merged_lse;
  common.wait_limit_ns = t_wait_limit_ns ? t_wait_limit_ns : kWaitLimitNs;
  common.stall_iteration = t_stall_iteration;
  common.slice_wait_ns = t_slice_wait_ns >= 0 ? (unsigned long long)t_slice_wait_ns : kSliceWaitNs;
  t_stall_iteration = -1;
  t_wait_limit_ns = 0;
  t_slice_wait_ns = -1;

  // Launches of at most kMaxUnitsLarge units each; every launch partitions its
  // own pages and reuses the workspace after the previous one (same stream).
  // All launches are laid out first: the fused merge's per-(request, kv
  // head) count spans every launch that holds a tile of the pair.
  struct Launch {
    size_t u0, n;
    long long total;
    int grid;
  };
  std::vector<Launch> launches;
  for (size_t u0 = 0; u0 < units.size(); u0 += kMaxUnitsLarge) {
    const size_t n = std::min<size_t>(kMaxUnitsLarge, units.size() - u0);
    // The CTAs' equal shares are cut from the units' pages laid end to end,
    // each unit preceded by kSegmentCharge pages that hold no data: a segment
    // (one unit's part on one CTA) costs a Q load, a combine and a partial
    // whatever its length, so a CTA whose range holds a unit start (one more
    // segment) gets that many fewer pages to stream.
    long long total = 0;
    for (size_t i = u0; i < u0 + n; ++i) {
      const int np = unit_pages(units[i].tok_start, units[i].tok_end);
      if (np > 0) total += kSegmentCharge;
      units[i].page_first = static_cast<int32_t>(total);
      total += np;
      PA_REQUIRE(total < (1ll << 31), "too many pages in one launch");
    }
    const int grid = launch_grid(total, sms, n_kv_heads);
    int part_cursor = 0;
    for (size_t i = u0; i < u0 + n; ++i) {
      const int np = unit_pages(units[i].tok_start, units[i].tok_end);
      if (np == 0) {
        units[i].n_parts = 0;
        continue;
      }
      const int k0 = cta_of(units[i].page_first, total, grid);
      const int k1 = cta_of(units[i].page_first + np - 1, total, grid);
      units[i].n_parts = k1 - k0 + 1;
      if (units[i].n_parts > 1) {
        units[i].part_base = part_cursor;
        part_cursor += units[i].n_parts;
      }
    }
    if ((size_t)part_cursor > slots)
      return fail(PA_ERR_INVALID, "internal: %d partial slots exceed the %zu reserved",
                  part_cursor, slots);
    launches.push_back({u0, n, total > 0 ? total : 1, grid});
  }
  // Completions each (request, kv head) pair's tile count reaches: one per
  // unsplit or empty unit, one per merge slice of a split unit.
  {
    std::vector<int32_t> pair_total((size_t)B * n_kv_heads, 0);
    auto pair_of = [&](const Unit& U) {
      const int bt = U.bt_g / n_kv_heads;
      return (size_t)(bt / T) * n_kv_heads + (U.bt_g - bt * n_kv_heads);
    };
    for (const Unit& U : units)
      pair_total[pair_of(U)] += U.n_parts > 1 ? split_slices(U.n_parts) : 1;
    for (Unit& U : units) U.pair_total = pair_total[pair_of(U)];
  }
  for (const Launch& L : launches) {
    common.n_requests = L.u0 == 0 ? B : 0;   // new rows are stored by the first launch
    int rc;
    if (L.n <= (size_t)kMaxUnitsSmall) {
      rc = tensor_cores ? launch_units<kMaxUnitsSmall, true>(tmap, units, L.u0, L.n, L.total,
                                                             L.grid, common, stream)
                        : launch_units<kMaxUnitsSmall, false>(tmap, units, L.u0, L.n, L.total,
                                                              L.grid, common, stream);
    } else {
      rc = tensor_cores ? launch_units<kMaxUnitsLarge, true>(tmap, units, L.u0, L.n, L.total,
                                                             L.grid, common, stream)
                        : launch_units<kMaxUnitsLarge, false>(tmap, units, L.u0, L.n, L.total,
                                                              L.grid, common, stream);
    }
    if (rc != PA_OK) return rc;
  }
  return PA_OK;
}

}  // namespace decode
}  // namespace pa

extern "C" size_t paged_decode_attn_lse_workspace_bytes(int B, int T, int n_q_heads,
                                                        int n_kv_heads, int head_dim) {
  if (B < 0 || T < 0 || head_dim != pa::decode::kD || n_kv_heads < 1 ||
      n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > pa::decode::kMaxG)
    return 0;
  return pa::decode::workspace_bytes(B, T, n_kv_heads);
}

extern "C" int paged_decode_attn_lse(const void* q, const void* pool, int64_t pool_pages,
                                     const int32_t* page_table, int max_pages,
                                     const int32_t* tiles, int B, int T, int n_q_heads,
                                     int n_kv_heads, int head_dim, float scale, float* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  return pa::decode::run(true, q, pool, pool_pages, page_table, max_pages, tiles, B, T,
                         n_q_heads, n_kv_heads, head_dim, scale, out, lse, workspace,
                         workspace_bytes, stream);
}

extern "C" int paged_decode_attn_lse_append(const void* q, void* pool, int64_t pool_pages,
                                            const int32_t* page_table, int max_pages,
                                            const int32_t* tiles, int B, int T, int n_q_heads,
                                            int n_kv_heads, int head_dim, float scale,
                                            const int32_t* positions, const void* new_rows,
                                            float* out, float* lse, float* merged_out,
                                            float* merged_lse, void* workspace,
                                            size_t workspace_bytes, unsigned flags,
                                            cudaStream_t stream) {
  pa::clear_error();
  if (!positions || !new_rows)
    return pa::fail(PA_ERR_INVALID, "positions and new_rows are required");
  return pa::decode::run(true, q, pool, pool_pages, page_table, max_pages, tiles, B, T,
                         n_q_heads, n_kv_heads, head_dim, scale, out, lse, workspace,
                         workspace_bytes, stream, positions, new_rows, flags, merged_out,
                         merged_lse);
}

extern "C" int paged_decode_attn_lse_cuda_core(const void* q, const void* pool,
                                               int64_t pool_pages, const int32_t* page_table,
                                               int max_pages, const int32_t* tiles, int B, int T,
                                               int n_q_heads, int n_kv_heads, int head_dim,
                                               float scale, float* out, float* lse,
                                               void* workspace, size_t workspace_bytes,
                                               cudaStream_t stream) {
  return pa::decode::run(false, q, pool, pool_pages, page_table, max_pages, tiles, B, T,
                         n_q_heads, n_kv_heads, head_dim, scale, out, lse, workspace,
                         workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers fix their device-memory budget before they start serving and
// forbid any allocation afterwards (so a long-running process cannot grow or
// fragment its footprint), and some cannot afford cudaMalloc in their hot
// loop because it can synchronise the whole device.  They cannot provide the
// workspace paged_decode_attn_lse asks for, so this entry point brings its
// own: a fixed array in this library's device globals, which every GPU that
// loads the library holds until the process exits.  The array is shared by
// every call on a device and keeps the previous call's contents; each call
// clears the part that must start at zero.  Calls that can overlap on the GPU
// (on different streams without ordering) race on the array.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchAddress {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};

std::mutex g_noalloc_mu;
ScratchAddress g_noalloc_addr[64];

// Device address of the scratch array in the current device's context.  The
// host-side name of the array is not a device address, and the address the
// runtime gives is valid only in the context it was looked up in (a device
// reset, or a primary context released and made again, loads the module
// anew, possibly elsewhere).  So the address is kept per device together
// with the id of the context it came from, and looked up again, with that
// device current, whenever the current context is another one.  If the
// driver cannot name the current context, every call looks it up.
int noalloc_scratch(void** out) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::fail(PA_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return pa::fail(PA_ERR_INVALID, "device index %d out of range", dev);
  unsigned long long id = 0;
  bool have_id = pa::current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  ScratchAddress& c = g_noalloc_addr[dev];
  if (!have_id || c.ptr == nullptr || c.ctx_id != id) {
    void* ptr = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (r != cudaSuccess || ptr == nullptr)
      return pa::fail(PA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed: %s",
                      cudaGetErrorString(r));
    // The lookup makes the device's primary context current if none was.
    if (!have_id) have_id = pa::current_context_id(&id);
    c.ptr = have_id ? ptr : nullptr;
    c.ctx_id = have_id ? id : 0;
    *out = ptr;
    return PA_OK;
  }
  *out = c.ptr;
  return PA_OK;
}

}  // namespace

extern "C" int paged_decode_attn_lse_noalloc(const void* q, const void* pool, int64_t pool_pages,
                                             const int32_t* page_table, int max_pages,
                                             const int32_t* tiles, int B, int T, int n_q_heads,
                                             int n_kv_heads, int head_dim, float scale,
                                             float* out, float* lse, int32_t* status,
                                             cudaStream_t stream) {
  pa::clear_error();
  if (B < 0 || T < 0) return pa::fail(PA_ERR_INVALID, "B and T must be >= 0 (got %d, %d)", B, T);
  if ((long long)B * T == 0) return PA_OK;
  const size_t need =
      paged_decode_attn_lse_workspace_bytes(B, T, n_q_heads, n_kv_heads, head_dim);
  if (need == 0) {
    // An unsupported geometry: let the checks below name it.
  } else if (need > kNoAllocScratchBytes)
    return pa::fail(PA_ERR_INVALID,
                    "this call needs %zu bytes of scratch, more than the %zu bytes the "
                    "no-allocation entry point holds; pass a workspace to "
                    "paged_decode_attn_lse instead",
                    need, kNoAllocScratchBytes);
  // Every argument is checked before the scratch is looked up or cleared,
  // so a refused call leaves the GPU and the array untouched.  The check
  // sees a stand-in workspace pointer (never dereferenced) of the array's size.
  int rc = pa::decode::check_args(q, pool, pool_pages, page_table, max_pages, tiles, B, T,
                                  n_q_heads, n_kv_heads, head_dim, out, lse,
                                  reinterpret_cast<const void*>(uintptr_t(256)),
                                  kNoAllocScratchBytes, nullptr, nullptr, 0, nullptr, nullptr);
  if (rc != PA_OK) return rc;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != PA_OK) return rc;
  // Status word and arrival counters must start at zero.
  const cudaError_t e = cudaMemsetAsync(scratch, 0, pa::decode::kStatusBytes + pa::decode::kCounterBytes,
                                        stream);
  if (e != cudaSuccess)
    return pa::fail(PA_ERR_CUDA, "clearing the scratch array failed: %s", cudaGetErrorString(e));
  rc = pa::decode::run(true, q, pool, pool_pages, page_table, max_pages, tiles, B, T, n_q_heads,
                       n_kv_heads, head_dim, scale, out, lse, scratch, kNoAllocScratchBytes,
                       stream);
  if (rc != PA_OK) return rc;
  if (status != nullptr) {
    const cudaError_t c =
        cudaMemcpyAsync(status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream);
    if (c != cudaSuccess)
      return pa::fail(PA_ERR_CUDA, "copying the status word failed: %s", cudaGetErrorString(c));
  }
  return PA_OK;
}

extern "C" int paged_decode_attn_test_slice_wait(int64_t slice_wait_ns) {
  pa::clear_error();
  if (slice_wait_ns < -1 || slice_wait_ns > (int64_t)pa::decode::kSliceWaitNs)
    return pa::fail(PA_ERR_INVALID, "slice_wait_ns must be -1 (clear) or in [0, %llu]",
                    (unsigned long long)pa::decode::kSliceWaitNs);
  pa::decode::t_slice_wait_ns = slice_wait_ns;
  return PA_OK;
}

extern "C" int paged_decode_attn_test_stall(int iteration, uint64_t wait_limit_ns) {
  pa::clear_error();
  if (iteration == -1 && wait_limit_ns == 0) {   // clear a pending setting
    pa::decode::t_stall_iteration = -1;
    pa::decode::t_wait_limit_ns = 0;
    return PA_OK;
  }
  if (iteration < 0 || wait_limit_ns == 0 || wait_limit_ns > pa::decode::kWaitLimitNs)
    return pa::fail(PA_ERR_INVALID,
                    "iteration must be >= 0 and wait_limit_ns in (0, %llu]",
                    (unsigned long long)pa::decode::kWaitLimitNs);
  pa::decode::t_stall_iteration = iteration;
  pa::decode::t_wait_limit_ns = wait_limit_ns;
  return PA_OK;
}
