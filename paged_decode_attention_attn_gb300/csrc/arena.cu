// Staging arena: pinned-host-owned KV history staged per layer into bounded
// device slots, ordered against attention and tail write-back by device events.
//
// Sources ("Staging without a stall", sections "Two copy queues and
// device-side ordering" and "Leases instead of buffers"; "KV-cache
// engineering", sections "Costing the bus before changing anything" and
// "Staging layers under a lease"):
//   * pinned host memory owns the history; the device holds a bounded set of
//     slots inside one explicitly sized allocation;
//   * the history copy runs on its own H2D stream and the compute stream waits
//     on an event recorded after it; the write-back runs on its own D2H stream
//     after an event recorded after attention; the host never blocks;
//   * a slot is reused only after the attention and the write-back that read
//     it: the next copy into the slot first waits on both events;
//   * only the new token's row goes back, and only to the owner the stage was
//     made for;
//   * any failure quarantines the arena; only a drain that establishes
//     completion releases it; destroy never waits, submits or drains.
//
// Two ways to drive an arena (one per arena):
//   * the stage calls (kv_stage_layer, kv_mark_attention_done,
//     kv_writeback_tail): a slot's next stage waits on the device for the
//     previous stage's attention and write-back events;
//   * leases ("Leases instead of buffers"; "Staging layers under a lease";
//     "GPU memory management", section "Staging as a lease"): every staged
//     layer is a transaction with a strictly increasing stage generation that
//     is begun, given its attention event and tail write-back, sealed with
//     exactly those events, and retired with host waits that produce a receipt.
//     Copy tickets pin the generation of the host pages a lease copies from, so
//     those pages cannot be recycled while a copy may still read them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cinttypes>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "common.h"

namespace pa {
namespace arena {

constexpr int kMaxRunsPerLaunch = 128;

struct TableRun {
  int32_t request;
  int32_t logical_page;
  int32_t n_pages;
  int32_t pad;
  long long first_page;
};

struct TableParams {
  int32_t* table;
  int max_pages;
  int n_runs;
  TableRun runs[kMaxRunsPerLaunch];
};

// Writes table[request][logical_page + i] = first_page + i for every run.
__global__ void fill_page_table_kernel(const __grid_constant__ TableParams p) {
  for (int r = blockIdx.x; r < p.n_runs; r += gridDim.x) {
    const TableRun run = p.runs[r];
    int32_t* row = p.table + (size_t)run.request * p.max_pages + run.logical_page;
    for (int i = threadIdx.x; i < run.n_pages; i += blockDim.x)
      row[i] = static_cast<int32_t>(run.first_page + i);
  }
}

struct ExpandRun {
  long long landing_off;  // bytes from the slot's landing area to the run's first compact page
  long long first_page;   // device page of the run's first page
  long long row_start;    // rows of the runs before this one in the launch
  int32_t n_pages;
  int32_t pad;
};

struct ExpandParams {
  const uint8_t* landing;   // the slot's landing area
  uint8_t* base;            // device_base
  long long page_bytes;     // bytes of a bf16 page
  long long cpage_bytes;    // bytes of a compact page
  long long total_rows;
  int row_elems;            // 2 * Hkv * head_dim
  int head_dim;
  int n_runs;
  ExpandRun runs[kMaxRunsPerLaunch];
};

// Rebuilds bf16 rows from compact pages: value = bf16_rne(float(code) * scale)
// with one binary32 scale per (row, K or V, kv head) slice.  One block per
// row (grid-stride); each thread turns 16 codes into 16 bf16 values.
__global__ void expand_compact_kernel(const __grid_constant__ ExpandParams p) {
  const int chunks = p.row_elems / 16;
  const int slices = p.row_elems / p.head_dim;
  for (long long row = blockIdx.x; row < p.total_rows; row += gridDim.x) {
    int r = 0;
    while (r + 1 < p.n_runs && p.runs[r + 1].row_start <= row) ++r;
    const ExpandRun run = p.runs[r];
    const long long rr = row - run.row_start;
    const long long page = rr / PA_PAGE_TOKENS;
    const int t = static_cast<int>(rr - page * PA_PAGE_TOKENS);
    const uint8_t* cpage = p.landing + run.landing_off + page * p.cpage_bytes;
    const int8_t* codes = reinterpret_cast<const int8_t*>(cpage) + (size_t)t * p.row_elems;
    const float* scales = reinterpret_cast<const float*>(
        cpage + (size_t)PA_PAGE_TOKENS * p.row_elems) + (size_t)t * slices;
    uint8_t* dst = p.base + (run.first_page + page) * p.page_bytes +
                   (size_t)t * p.row_elems * 2;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      const float s = scales[(c * 16) / p.head_dim];
      const uint4 raw = *reinterpret_cast<const uint4*>(codes + c * 16);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t out[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t word = w[k / 2];
        const int sh = (k % 2) * 16;
        const float lo = static_cast<float>(static_cast<int8_t>((word >> sh) & 0xFFu));
        const float hi = static_cast<float>(static_cast<int8_t>((word >> (sh + 8)) & 0xFFu));
        const __nv_bfloat16 blo = __float2bfloat16_rn(__fmul_rn(lo, s));
        const __nv_bfloat16 bhi = __float2bfloat16_rn(__fmul_rn(hi, s));
        out[k] = static_cast<uint32_t>(__bfloat16_as_ushort(blo)) |
                 (static_cast<uint32_t>(__bfloat16_as_ushort(bhi)) << 16);
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)c * 32);
      d4[0] = make_uint4(out[0], out[1], out[2], out[3]);
      d4[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
}

enum SlotState { kFree = 0, kStaged = 1, kAttended = 2 };

struct ReqRecord {
  int32_t request;
  uint64_t owner;
  std::vector<kv_page_run> runs;
  std::vector<int64_t> first_page;  // device page of each run's first page
};

struct Slot {
  SlotState state = kFree;
  int layer = -1;
  uint64_t generation = 0;
  bool written_back = false;
  bool retired = false;          // lease API: host confirmed completion of the last use
  uint64_t lease_id = 0;         // lease API: lease that last used the slot
  std::vector<ReqRecord> reqs;
};

enum LeaseState { kBegun = 0, kLeaseAttended = 1, kSealed = 2 };

struct Ticket {
  uint64_t owner;
  uint64_t host_generation;
  uint64_t bytes;
};

struct Lease {
  uint64_t id = 0;               // the stage generation
  int layer = 0;
  int64_t step = 0;
  int slot = 0;
  LeaseState state = kBegun;
  uint64_t attention_token = 0;
  uint64_t writeback_token = 0;  // 0 until a write-back is issued
  uint64_t staged_bytes = 0;
  uint64_t loaded_bytes = 0;      // kv_load_resident copies
  uint64_t written_back_bytes = 0;
  int32_t n_requests = 0;
  std::vector<Ticket> tickets;
};

struct HostOwner {
  uint64_t generation = 1;
  int64_t live_tickets = 0;
};

enum Mode { kModeUnset = 0, kModeStage = 1, kModeLease = 2 };

}  // namespace arena
}  // namespace pa

struct kv_arena {
  kv_arena_desc d{};
  bool record_only = false;
  bool quarantined = false;
  int64_t fail_after = -1;
  std::string log;
  std::vector<cudaEvent_t> ev_copy, ev_attn, ev_wb;
  cudaEvent_t ev_load = nullptr;  // recorded after each kv_load_resident's copies
  int last_attn_slot = -1;        // slot of the most recent attention event
  int last_wb_slot = -1;          // slot of the most recent write-back event
  std::vector<pa::arena::Slot> slots;
  std::map<int, int> layer_slot;
  uint64_t generation = 0;
  uint64_t staged_bytes = 0;
  uint64_t loaded_bytes = 0;      // kv_load_resident copies
  uint64_t written_back_bytes = 0;
  uint64_t slot_reuses = 0;
  int64_t page_bytes = 0;
  int64_t arena_pages = 0;
  int64_t cpage_bytes = 0;      // compact page bytes (0: no compact runs)
  pa::arena::Mode mode = pa::arena::kModeUnset;
  std::map<uint64_t, pa::arena::Lease> leases;      // begun, not yet retired
  std::map<uint64_t, pa::arena::HostOwner> owners;  // host page generations
  uint64_t last_lease = 0;                          // most recently begun lease
  uint64_t event_tokens = 0;
};

namespace pa {
namespace arena {

namespace {

int quarantine(kv_arena* a, const char* what, cudaError_t e) {
  a->quarantined = true;
  return fail(PA_ERR_CUDA, "%s failed (%s); arena quarantined", what,
              e == cudaSuccess ? "injected failure" : cudaGetErrorString(e));
}

// Gate every submission: honours the injected-failure countdown.
bool injected_failure(kv_arena* a) {
  if (a->fail_after < 0) return false;
  if (a->fail_after == 0) {
    a->fail_after = -1;
    return true;
  }
  --a->fail_after;
  return false;
}

void logf_(kv_arena* a, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
void logf_(kv_arena* a, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  a->log += buf;
  a->log += '\n';
}

const char* stream_name(kv_arena* a, cudaStream_t s) {
  if (s == a->d.h2d_stream) return "h2d";
  if (s == a->d.d2h_stream) return "d2h";
  if (s == a->d.compute_stream) return "compute";
  return "?";
}

int op_wait(kv_arena* a, cudaStream_t s, const char* ev_kind, int slot, cudaEvent_t ev) {
  if (injected_failure(a)) return quarantine(a, "cudaStreamWaitEvent", cudaSuccess);
  if (a->record_only) {
    logf_(a, "%s wait %s[%d]", stream_name(a, s), ev_kind, slot);
    return PA_OK;
  }
  const cudaError_t e = cudaStreamWaitEvent(s, ev, 0);
  return e == cudaSuccess ? PA_OK : quarantine(a, "cudaStreamWaitEvent", e);
}

int op_record(kv_arena* a, cudaStream_t s, const char* ev_kind, int slot, cudaEvent_t ev) {
  if (injected_failure(a)) return quarantine(a, "cudaEventRecord", cudaSuccess);
  if (a->record_only) {
    logf_(a, "%s record %s[%d]", stream_name(a, s), ev_kind, slot);
    return PA_OK;
  }
  const cudaError_t e = cudaEventRecord(ev, s);
  return e == cudaSuccess ? PA_OK : quarantine(a, "cudaEventRecord", e);
}

// Host wait on an event (lease retirement); a failure quarantines.
int op_host_wait(kv_arena* a, const char* ev_kind, int slot, cudaEvent_t ev) {
  if (injected_failure(a)) return quarantine(a, "cudaEventSynchronize", cudaSuccess);
  if (a->record_only) {
    logf_(a, "host wait %s[%d]", ev_kind, slot);
    return PA_OK;
  }
  const cudaError_t e = cudaEventSynchronize(ev);
  return e == cudaSuccess ? PA_OK : quarantine(a, "cudaEventSynchronize", e);
}

int op_copy(kv_arena* a, cudaStream_t s, void* dst, const void* src, size_t bytes,
            cudaMemcpyKind kind, long long dev_page, long long row) {
  if (injected_failure(a)) return quarantine(a, "cudaMemcpyAsync", cudaSuccess);
  if (a->record_only) {
    logf_(a, "%s copy %s bytes=%zu page=%lld row=%lld", stream_name(a, s),
          kind == cudaMemcpyHostToDevice ? "h2d" : "d2h", bytes, dev_page, row);
    return PA_OK;
  }
  const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
  return e == cudaSuccess ? PA_OK : quarantine(a, "cudaMemcpyAsync", e);
}

int op_table(kv_arena* a, cudaStream_t s, int slot, const TableParams& p) {
  if (injected_failure(a)) return quarantine(a, "page-table kernel launch", cudaSuccess);
  if (a->record_only) {
    std::string line;
    char buf[96];
    snprintf(buf, sizeof(buf), "%s table slot=%d runs=%d", stream_name(a, s), slot, p.n_runs);
    line = buf;
    for (int i = 0; i < p.n_runs; ++i) {
      snprintf(buf, sizeof(buf), " %d:%d+%d->%lld", p.runs[i].request, p.runs[i].logical_page,
               p.runs[i].n_pages, p.runs[i].first_page);
      line += buf;
    }
    a->log += line;
    a->log += '\n';
    return PA_OK;
  }
  const int blocks = p.n_runs < 1 ? 1 : p.n_runs;
  fill_page_table_kernel<<<blocks, 256, 0, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : quarantine(a, "page-table kernel launch", e);
}

int op_expand(kv_arena* a, cudaStream_t s, int slot, const ExpandParams& p) {
  if (injected_failure(a)) return quarantine(a, "expand kernel launch", cudaSuccess);
  if (a->record_only) {
    std::string line;
    char buf[96];
    snprintf(buf, sizeof(buf), "%s expand slot=%d runs=%d", stream_name(a, s), slot, p.n_runs);
    line = buf;
    for (int i = 0; i < p.n_runs; ++i) {
      snprintf(buf, sizeof(buf), " +%lld:%d->%lld", p.runs[i].landing_off, p.runs[i].n_pages,
               p.runs[i].first_page);
      line += buf;
    }
    a->log += line;
    a->log += '\n';
    return PA_OK;
  }
  const long long blocks = std::min<long long>(p.total_rows, 8192);
  expand_compact_kernel<<<(unsigned)(blocks < 1 ? 1 : blocks), 128, 0, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : quarantine(a, "expand kernel launch", e);
}

// Checks a stage request list against the arena; submits nothing.
int validate_stage(kv_arena* a, const kv_stage_req* reqs, int n_reqs) {
  const kv_arena_desc& d = a->d;
  PA_REQUIRE(n_reqs >= 0 && (n_reqs == 0 || reqs), "bad request list");
  std::vector<char> seen(d.max_requests, 0);
  int64_t staged_pages = 0;
  uint64_t landing_used = 0;
  for (int i = 0; i < n_reqs; ++i) {
    const kv_stage_req& r = reqs[i];
    PA_REQUIRE(r.request >= 0 && r.request < d.max_requests, "request %d outside [0, %d)",
               r.request, d.max_requests);
    PA_REQUIRE(!seen[r.request], "request %d staged twice", r.request);
    seen[r.request] = 1;
    PA_REQUIRE(r.n_runs >= 0 && (r.n_runs == 0 || r.runs), "request %d: bad run list",
               r.request);
    for (int k = 0; k < r.n_runs; ++k) {
      const kv_page_run& run = r.runs[k];
      PA_REQUIRE(run.logical_page >= 0 && run.n_pages >= 1 &&
                     (int64_t)run.logical_page + run.n_pages <= d.max_pages,
                 "request %d run %d: pages [%d, +%d) outside the table", r.request, k,
                 run.logical_page, run.n_pages);
      if (run.host_compact) {
        PA_REQUIRE(!run.host_rows, "request %d run %d: both exact and compact", r.request, k);
        PA_REQUIRE(a->cpage_bytes > 0, "request %d run %d: this arena has no landing area",
                   r.request, k);
        PA_REQUIRE(run.n_rows == (int64_t)run.n_pages * d.page_tokens,
                   "request %d run %d: a compact run holds fully written pages only", r.request,
                   k);
        if (!a->record_only) {
          cudaPointerAttributes attr;
          const cudaError_t e = cudaPointerGetAttributes(&attr, run.host_compact);
          PA_REQUIRE(e == cudaSuccess && attr.type == cudaMemoryTypeHost,
                     "request %d run %d: compact pages must be pinned host memory", r.request, k);
        }
        landing_used += (uint64_t)run.n_pages * a->cpage_bytes;
        staged_pages += run.n_pages;
      } else if (run.host_rows) {
        PA_REQUIRE(run.n_rows >= 0 && run.n_rows <= (int64_t)run.n_pages * d.page_tokens,
                   "request %d run %d: %" PRId64 " rows do not fit %d pages", r.request, k,
                   run.n_rows, run.n_pages);
        if (!a->record_only) {
          cudaPointerAttributes attr;
          const cudaError_t e = cudaPointerGetAttributes(&attr, run.host_rows);
          PA_REQUIRE(e == cudaSuccess && attr.type == cudaMemoryTypeHost,
                     "request %d run %d: host rows must be pinned host memory", r.request, k);
        }
        staged_pages += run.n_pages;
      } else {
        PA_REQUIRE(run.resident_page >= 0 && run.resident_page + run.n_pages <= a->arena_pages,
                   "request %d run %d: resident pages outside the arena", r.request, k);
        const int64_t slots_end = d.slot_first_page + (int64_t)d.n_slots * d.slot_pages;
        PA_REQUIRE(run.resident_page + run.n_pages <= d.slot_first_page ||
                       run.resident_page >= slots_end,
                   "request %d run %d: resident pages [%" PRId64 ", +%d) overlap the staging "
                   "slots [%" PRId64 ", %" PRId64 ")",
                   r.request, k, run.resident_page, run.n_pages, d.slot_first_page, slots_end);
      }
    }
  }
  PA_REQUIRE(staged_pages <= d.slot_pages, "stage needs %" PRId64 " pages, a slot holds %" PRId64,
             staged_pages, d.slot_pages);
  PA_REQUIRE(landing_used <= d.landing_bytes,
             "compact runs need %" PRIu64 " landing bytes, a slot has %" PRIu64, landing_used,
             (uint64_t)d.landing_bytes);
  return PA_OK;
}

// Enqueues a validated stage into `slot`: optional waits on the slot's
// previous readers, one H2D copy per staged run, the page-table fill, the copy
// event and the compute stream's wait on it.  Returns the run records and the
// bytes copied per request.
int submit_stage(kv_arena* a, int slot, bool wait_prior_readers, const kv_stage_req* reqs,
                 int n_reqs, std::vector<ReqRecord>* records, std::vector<uint64_t>* bytes) {
  const kv_arena_desc& d = a->d;
  Slot& S = a->slots[slot];
  const cudaStream_t h2d = d.h2d_stream;
  int rc;
  if (wait_prior_readers) {
    ++a->slot_reuses;
    if ((rc = op_wait(a, h2d, "attn", slot, a->ev_attn[slot])) != PA_OK) return rc;
    if (S.written_back && (rc = op_wait(a, h2d, "wb", slot, a->ev_wb[slot])) != PA_OK) return rc;
  }
  uint8_t* base = static_cast<uint8_t*>(d.device_base);
  const int64_t slot_page0 = d.slot_first_page + (int64_t)slot * d.slot_pages;
  records->clear();
  records->reserve(n_reqs);
  bytes->assign(n_reqs, 0);
  std::vector<TableRun> table_runs;
  std::vector<ExpandRun> expand_runs;
  int64_t cursor = 0;
  long long landing_cursor = 0;
  uint8_t* landing = base + d.landing_offset + (uint64_t)slot * d.landing_bytes;
  for (int i = 0; i < n_reqs; ++i) {
    const kv_stage_req& r = reqs[i];
    ReqRecord rec;
    rec.request = r.request;
    rec.owner = r.owner;
    for (int k = 0; k < r.n_runs; ++k) {
      const kv_page_run& run = r.runs[k];
      int64_t first;
      if (run.host_compact) {
        first = slot_page0 + cursor;
        cursor += run.n_pages;
        const size_t nb = (size_t)run.n_pages * a->cpage_bytes;
        if ((rc = op_copy(a, h2d, landing + landing_cursor, run.host_compact, nb,
                          cudaMemcpyHostToDevice, first, -1)) != PA_OK)
          return rc;
        a->staged_bytes += nb;
        (*bytes)[i] += nb;
        expand_runs.push_back(ExpandRun{landing_cursor, first, 0, run.n_pages, 0});
        landing_cursor += (long long)nb;
      } else if (run.host_rows) {
        first = slot_page0 + cursor;
        cursor += run.n_pages;
        const size_t nb = (size_t)run.n_rows * d.row_bytes;
        if (nb > 0) {
          if ((rc = op_copy(a, h2d, base + first * a->page_bytes, run.host_rows, nb,
                            cudaMemcpyHostToDevice, first, 0)) != PA_OK)
            return rc;
          a->staged_bytes += nb;
          (*bytes)[i] += nb;
        }
      } else {
        first = run.resident_page;
      }
      rec.runs.push_back(run);
      rec.first_page.push_back(first);
      table_runs.push_back(TableRun{r.request, run.logical_page, run.n_pages, 0, first});
    }
    records->push_back(std::move(rec));
  }
  int32_t* table = d.page_tables + (size_t)slot * d.max_requests * d.max_pages;
  for (size_t r0 = 0; r0 < table_runs.size(); r0 += kMaxRunsPerLaunch) {
    TableParams tp{};
    tp.table = table;
    tp.max_pages = d.max_pages;
    tp.n_runs = static_cast<int>(std::min<size_t>(kMaxRunsPerLaunch, table_runs.size() - r0));
    std::memcpy(tp.runs, table_runs.data() + r0, tp.n_runs * sizeof(TableRun));
    if ((rc = op_table(a, h2d, slot, tp)) != PA_OK) return rc;
  }
  if ((rc = op_record(a, h2d, "copy", slot, a->ev_copy[slot])) != PA_OK) return rc;
  if ((rc = op_wait(a, d.compute_stream, "copy", slot, a->ev_copy[slot])) != PA_OK) return rc;
  // Compact runs are expanded on the compute stream, after the copy event and
  // before the attention: the H2D stream is free to copy the next layer
  // meanwhile, and the slot's landing area is rewritten only after this
  // layer's attention (the slot-reuse wait), hence after its expansion.
  for (size_t r0 = 0; r0 < expand_runs.size(); r0 += kMaxRunsPerLaunch) {
    ExpandParams ep{};
    ep.landing = landing;
    ep.base = base;
    ep.page_bytes = a->page_bytes;
    ep.cpage_bytes = a->cpage_bytes;
    ep.row_elems = d.row_bytes / 2;
    ep.head_dim = d.compact_head_dim;
    ep.n_runs = static_cast<int>(std::min<size_t>(kMaxRunsPerLaunch, expand_runs.size() - r0));
    long long rows = 0;
    for (int k = 0; k < ep.n_runs; ++k) {
      ep.runs[k] = expand_runs[r0 + k];
      ep.runs[k].row_start = rows;
      rows += (long long)ep.runs[k].n_pages * d.page_tokens;
    }
    ep.total_rows = rows;
    if ((rc = op_expand(a, d.compute_stream, slot, ep)) != PA_OK) return rc;
  }
  return PA_OK;
}

// Resolves each tail row's device address in `slot` and checks its owner;
// submits nothing.
int resolve_tails(kv_arena* a, int slot, int layer, const kv_tail_req* reqs, int n_reqs,
                  std::vector<uint8_t*>* src) {
  const kv_arena_desc& d = a->d;
  const Slot& S = a->slots[slot];
  PA_REQUIRE(n_reqs >= 0 && (n_reqs == 0 || reqs), "bad request list");
  src->assign(n_reqs, nullptr);
  for (int i = 0; i < n_reqs; ++i) {
    const kv_tail_req& t = reqs[i];
    PA_REQUIRE(t.host_row != nullptr, "tail %d: null host row", i);
    const ReqRecord* rec = nullptr;
    for (const auto& r : S.reqs)
      if (r.request == t.request) rec = &r;
    PA_REQUIRE(rec != nullptr, "tail %d: request %d was not staged for layer %d", i, t.request,
               layer);
    if (rec->owner != t.owner)
      return fail(PA_ERR_OWNER,
                  "tail %d: owner %" PRIu64 " differs from the owner %" PRIu64
                  " request %d was staged with",
                  i, t.owner, rec->owner, t.request);
    PA_REQUIRE(t.position >= 0, "tail %d: negative position", i);
    const int64_t lp = t.position / d.page_tokens;
    int64_t page = -1;
    for (size_t k = 0; k < rec->runs.size(); ++k) {
      const kv_page_run& run = rec->runs[k];
      if (lp >= run.logical_page && lp < (int64_t)run.logical_page + run.n_pages)
        page = rec->first_page[k] + (lp - run.logical_page);
    }
    PA_REQUIRE(page >= 0, "tail %d: position %" PRId64 " is not in a staged or resident run", i,
               t.position);
    (*src)[i] = static_cast<uint8_t*>(d.device_base) +
                (page * d.page_tokens + t.position % d.page_tokens) * (int64_t)d.row_bytes;
  }
  return PA_OK;
}

// Enqueues the tail write-backs of `slot` after its attention event and
// records the write-back event.
int submit_tails(kv_arena* a, int slot, const kv_tail_req* reqs, int n_reqs,
                 const std::vector<uint8_t*>& src, uint64_t* bytes) {
  const kv_arena_desc& d = a->d;
  int rc;
  if ((rc = op_wait(a, d.d2h_stream, "attn", slot, a->ev_attn[slot])) != PA_OK) return rc;
  for (int i = 0; i < n_reqs; ++i) {
    const int64_t off = src[i] - static_cast<uint8_t*>(d.device_base);
    if ((rc = op_copy(a, d.d2h_stream, reqs[i].host_row, src[i], d.row_bytes,
                      cudaMemcpyDeviceToHost, off / a->page_bytes,
                      (off % a->page_bytes) / d.row_bytes)) != PA_OK)
      return rc;
    a->written_back_bytes += d.row_bytes;
    *bytes += d.row_bytes;
  }
  if ((rc = op_record(a, d.d2h_stream, "wb", slot, a->ev_wb[slot])) != PA_OK) return rc;
  a->slots[slot].written_back = true;
  a->last_wb_slot = slot;
  return PA_OK;
}

int use_mode(kv_arena* a, Mode m) {
  if (a->mode == kModeUnset) a->mode = m;
  if (a->mode != m)
    return fail(PA_ERR_ORDER, "this arena is driven by %s calls; do not mix the two",
                a->mode == kModeStage ? "stage" : "lease");
  return PA_OK;
}

}  // namespace

}  // namespace arena
}  // namespace pa

using pa::fail;
using namespace pa::arena;

extern "C" int kv_arena_create(const kv_arena_desc* desc, kv_arena** out) {
  pa::clear_error();
  PA_REQUIRE(desc && out, "null pointer argument");
  *out = nullptr;
  const kv_arena_desc& d = *desc;
  PA_REQUIRE(d.device_base != nullptr, "device_base is null");
  PA_REQUIRE(reinterpret_cast<uintptr_t>(d.device_base) % 256 == 0,
             "device_base must be 256-byte aligned");
  PA_REQUIRE(d.row_bytes > 0 && d.row_bytes % 16 == 0,
             "row_bytes (%d) must be a positive multiple of 16", d.row_bytes);
  PA_REQUIRE(d.page_tokens == PA_PAGE_TOKENS, "page_tokens must be %d", PA_PAGE_TOKENS);
  PA_REQUIRE(d.n_slots >= 1 && d.n_slots <= 64, "n_slots (%d) must be in 1..64", d.n_slots);
  PA_REQUIRE(d.slot_pages >= 1 && d.slot_first_page >= 0, "bad slot geometry");
  PA_REQUIRE(d.page_tables != nullptr && d.max_requests >= 1 && d.max_pages >= 1,
             "page_tables, max_requests and max_pages are required");
  const int64_t page_bytes = (int64_t)d.row_bytes * d.page_tokens;
  // Pages end where the landing areas begin (if there are any).
  const uint64_t page_area = (d.landing_bytes > 0 && d.landing_offset < d.device_bytes)
                                 ? d.landing_offset : d.device_bytes;
  const int64_t arena_pages = (int64_t)(page_area / (uint64_t)page_bytes);
  PA_REQUIRE(d.slot_first_page + (int64_t)d.n_slots * d.slot_pages <= arena_pages,
             "slots need %" PRId64 " pages of %" PRId64 " bytes but device_bytes holds %" PRId64,
             d.slot_first_page + (int64_t)d.n_slots * d.slot_pages, page_bytes, arena_pages);
  PA_REQUIRE(arena_pages < (1ll << 31), "arena too large for 32-bit page ids");
  int64_t cpage_bytes = 0;
  if (d.landing_bytes > 0 || d.compact_head_dim != 0) {
    const int64_t row_elems = d.row_bytes / 2;
    PA_REQUIRE(d.compact_head_dim >= 16 && d.compact_head_dim % 16 == 0 &&
                   row_elems % (2 * d.compact_head_dim) == 0,
               "compact_head_dim (%d) must be a multiple of 16 dividing a row's K and V",
               d.compact_head_dim);
    cpage_bytes = (int64_t)kv_compact_page_bytes(
        static_cast<int>(row_elems / (2 * d.compact_head_dim)), d.compact_head_dim);
    PA_REQUIRE(d.landing_bytes >= (uint64_t)cpage_bytes,
               "landing_bytes (%" PRIu64 ") holds no compact page of %" PRId64 " bytes",
               (uint64_t)d.landing_bytes, cpage_bytes);
    PA_REQUIRE(d.landing_offset % 256 == 0, "landing_offset must be 256-byte aligned");
    PA_REQUIRE(d.landing_offset >= (uint64_t)((d.slot_first_page + (int64_t)d.n_slots *
                                                                       d.slot_pages) *
                                              page_bytes),
               "the landing areas must follow every page");
    PA_REQUIRE(d.landing_offset + (uint64_t)d.n_slots * d.landing_bytes <= d.device_bytes,
               "landing areas end past device_bytes");
  }

  kv_arena* a = new kv_arena;
  a->d = d;
  a->record_only = (d.flags & PA_ARENA_RECORD_ONLY) != 0;
  a->page_bytes = page_bytes;
  a->arena_pages = arena_pages;
  a->cpage_bytes = cpage_bytes;
  a->slots.resize(d.n_slots);
  a->ev_copy.assign(d.n_slots, nullptr);
  a->ev_attn.assign(d.n_slots, nullptr);
  a->ev_wb.assign(d.n_slots, nullptr);
  if (!a->record_only) {
    for (int s = 0; s < d.n_slots; ++s) {
      cudaError_t e = cudaEventCreateWithFlags(&a->ev_copy[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a->ev_attn[s], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a->ev_wb[s], cudaEventDisableTiming);
      if (e == cudaSuccess && s == 0)
        e = cudaEventCreateWithFlags(&a->ev_load, cudaEventDisableTiming);
      if (e != cudaSuccess) {
        kv_arena_destroy(a);
        return fail(PA_ERR_CUDA, "cudaEventCreateWithFlags failed: %s", cudaGetErrorString(e));
      }
    }
  }
  *out = a;
  return PA_OK;
}

extern "C" int kv_arena_destroy(kv_arena* a) {
  pa::clear_error();
  if (!a) return PA_OK;
  // Never waits: destroying an event with work pending releases it when done.
  for (auto* v : {&a->ev_copy, &a->ev_attn, &a->ev_wb})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  if (a->ev_load) cudaEventDestroy(a->ev_load);
  delete a;
  return PA_OK;
}

extern "C" int kv_arena_drain(kv_arena* a) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->record_only) {
    if (injected_failure(a)) return quarantine(a, "drain", cudaSuccess);
    logf_(a, "drain");
  } else {
    for (cudaStream_t s : {a->d.h2d_stream, a->d.d2h_stream, a->d.compute_stream}) {
      const cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return quarantine(a, "cudaStreamSynchronize", e);
    }
  }
  // Completion is established: every slot is free again; leases that were
  // in flight are dropped (their copies are known to be finished) and their
  // tickets released.
  for (auto& s : a->slots) {
    s.state = kFree;
    s.written_back = false;
    s.retired = false;
    s.lease_id = 0;
    s.reqs.clear();
  }
  for (auto& kv : a->leases)
    for (const Ticket& t : kv.second.tickets) a->owners[t.owner].live_tickets -= 1;
  a->leases.clear();
  a->last_lease = 0;
  a->layer_slot.clear();
  a->last_attn_slot = -1;
  a->last_wb_slot = -1;
  a->quarantined = false;
  return PA_OK;
}

// ---------------------------------------------------------------------------
// Stage calls.
// ---------------------------------------------------------------------------

extern "C" int kv_stage_layer(kv_arena* a, int layer, const kv_stage_req* reqs, int n_reqs,
                              int* slot_out, const int32_t** page_table_out) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  PA_REQUIRE(layer >= 0, "layer must be >= 0");
  int rc = use_mode(a, kModeStage);
  if (rc != PA_OK) return rc;
  const kv_arena_desc& d = a->d;
  const int slot = static_cast<int>(a->generation % (uint64_t)d.n_slots);
  Slot& S = a->slots[slot];
  if (S.state == kStaged)
    return fail(PA_ERR_ORDER,
                "slot %d still holds layer %d, which was never marked attention-done", slot,
                S.layer);
  if ((rc = validate_stage(a, reqs, n_reqs)) != PA_OK) return rc;
  std::vector<ReqRecord> records;
  std::vector<uint64_t> bytes;
  if ((rc = submit_stage(a, slot, S.state != kFree, reqs, n_reqs, &records, &bytes)) != PA_OK)
    return rc;
  S.state = kStaged;
  S.layer = layer;
  S.generation = ++a->generation;
  S.written_back = false;
  S.reqs = std::move(records);
  a->layer_slot[layer] = slot;
  if (slot_out) *slot_out = slot;
  if (page_table_out) *page_table_out = d.page_tables + (size_t)slot * d.max_requests * d.max_pages;
  return PA_OK;
}

extern "C" int kv_mark_attention_done(kv_arena* a, int layer) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  int rc = use_mode(a, kModeStage);
  if (rc != PA_OK) return rc;
  const auto it = a->layer_slot.find(layer);
  if (it == a->layer_slot.end()) return fail(PA_ERR_ORDER, "layer %d has no current stage", layer);
  Slot& S = a->slots[it->second];
  if (S.layer != layer || S.state != kStaged)
    return fail(PA_ERR_ORDER, "layer %d is not awaiting attention (slot %d)", layer, it->second);
  rc = op_record(a, a->d.compute_stream, "attn", it->second, a->ev_attn[it->second]);
  if (rc != PA_OK) return rc;
  a->last_attn_slot = it->second;
  S.state = kAttended;
  return PA_OK;
}

extern "C" int kv_writeback_tail(kv_arena* a, int layer, const kv_tail_req* reqs, int n_reqs) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  int rc = use_mode(a, kModeStage);
  if (rc != PA_OK) return rc;
  const auto it = a->layer_slot.find(layer);
  if (it == a->layer_slot.end()) return fail(PA_ERR_ORDER, "layer %d has no current stage", layer);
  const int slot = it->second;
  Slot& S = a->slots[slot];
  if (S.layer != layer || S.state != kAttended)
    return fail(PA_ERR_ORDER, "write-back of layer %d before its attention was marked done",
                layer);
  std::vector<uint8_t*> src;
  if ((rc = resolve_tails(a, slot, layer, reqs, n_reqs, &src)) != PA_OK) return rc;
  uint64_t bytes = 0;
  return submit_tails(a, slot, reqs, n_reqs, src, &bytes);
}

// ---------------------------------------------------------------------------
// Copy-in of resident pages.
// ---------------------------------------------------------------------------

extern "C" int kv_load_resident(kv_arena* a, const kv_resident_load* loads, int n_loads) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  PA_REQUIRE(n_loads >= 0 && (n_loads == 0 || loads), "bad load list");
  const kv_arena_desc& d = a->d;
  const int64_t slots_end = d.slot_first_page + (int64_t)d.n_slots * d.slot_pages;
  for (int i = 0; i < n_loads; ++i) {
    const kv_resident_load& L = loads[i];
    PA_REQUIRE(L.resident_page >= 0 && L.resident_page < a->arena_pages,
               "load %d: page %" PRId64 " outside the arena's %" PRId64 " pages", i,
               L.resident_page, a->arena_pages);
    PA_REQUIRE(L.resident_page < d.slot_first_page || L.resident_page >= slots_end,
               "load %d: page %" PRId64 " lies in the staging slots [%" PRId64 ", %" PRId64 ")",
               i, L.resident_page, d.slot_first_page, slots_end);
    PA_REQUIRE(L.n_rows >= 1 && L.n_rows <= d.page_tokens, "load %d: n_rows %d outside 1..%d", i,
               L.n_rows, d.page_tokens);
    PA_REQUIRE(L.host_rows != nullptr, "load %d: null host rows", i);
    if (!a->record_only) {
      cudaPointerAttributes attr;
      const cudaError_t e = cudaPointerGetAttributes(&attr, L.host_rows);
      PA_REQUIRE(e == cudaSuccess && attr.type == cudaMemoryTypeHost,
                 "load %d: host rows must be pinned host memory", i);
    }
  }
  if (n_loads == 0) return PA_OK;
  const cudaStream_t h2d = d.h2d_stream;
  int rc;
  // The pages being replaced may still be read by earlier attention (through
  // a page table) or by a tail write-back (the new row of a resident page).
  if (a->last_attn_slot >= 0 &&
      (rc = op_wait(a, h2d, "attn", a->last_attn_slot, a->ev_attn[a->last_attn_slot])) != PA_OK)
    return rc;
  if (a->last_wb_slot >= 0 &&
      (rc = op_wait(a, h2d, "wb", a->last_wb_slot, a->ev_wb[a->last_wb_slot])) != PA_OK)
    return rc;
  uint8_t* base = static_cast<uint8_t*>(d.device_base);
  for (int i = 0; i < n_loads; ++i) {
    const kv_resident_load& L = loads[i];
    const size_t nb = (size_t)L.n_rows * d.row_bytes;
    if ((rc = op_copy(a, h2d, base + L.resident_page * a->page_bytes, L.host_rows, nb,
                      cudaMemcpyHostToDevice, L.resident_page, 0)) != PA_OK)
      return rc;
    a->loaded_bytes += nb;
  }
  if ((rc = op_record(a, h2d, "load", 0, a->ev_load)) != PA_OK) return rc;
  return op_wait(a, d.compute_stream, "load", 0, a->ev_load);
}

// ---------------------------------------------------------------------------
// Leases.
// ---------------------------------------------------------------------------

extern "C" int kv_lease_begin(kv_arena* a, int layer, int64_t step, const kv_stage_req* reqs,
                              int n_reqs, kv_lease* out) {
  pa::clear_error();
  PA_REQUIRE(a && out, "null pointer argument");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  PA_REQUIRE(layer >= 0, "layer must be >= 0");
  int rc = use_mode(a, kModeLease);
  if (rc != PA_OK) return rc;
  // A new lease may begin only once the previous one is sealed or retired.
  if (a->last_lease != 0) {
    const auto prev = a->leases.find(a->last_lease);
    if (prev != a->leases.end() && prev->second.state != kSealed)
      return fail(PA_ERR_ORDER, "lease %" PRIu64 " (layer %d) is neither sealed nor retired",
                  prev->second.id, prev->second.layer);
  }
  const kv_arena_desc& d = a->d;
  const int slot = static_cast<int>(a->generation % (uint64_t)d.n_slots);
  Slot& S = a->slots[slot];
  if ((rc = validate_stage(a, reqs, n_reqs)) != PA_OK) return rc;
  // The previous user of the slot is sealed (checked above or earlier).  If
  // it is not retired, its attention and write-back are prior readers of this
  // lease: the copies wait for them on the device.
  const bool wait_prior = S.state != kFree && !S.retired;
  std::vector<ReqRecord> records;
  std::vector<uint64_t> bytes;
  if ((rc = submit_stage(a, slot, wait_prior, reqs, n_reqs, &records, &bytes)) != PA_OK) return rc;
  Lease L;
  L.id = ++a->generation;
  L.layer = layer;
  L.step = step;
  L.slot = slot;
  L.n_requests = n_reqs;
  for (int i = 0; i < n_reqs; ++i) {
    L.staged_bytes += bytes[i];
    bool staged = false;
    for (int k = 0; k < reqs[i].n_runs; ++k) staged |= reqs[i].runs[k].host_rows != nullptr;
    if (staged) {
      HostOwner& o = a->owners[reqs[i].owner];
      o.live_tickets += 1;
      L.tickets.push_back(Ticket{reqs[i].owner, o.generation, bytes[i]});
    }
  }
  S.state = kStaged;
  S.layer = layer;
  S.generation = L.id;
  S.written_back = false;
  S.retired = false;
  S.lease_id = L.id;
  S.reqs = std::move(records);
  a->leases[L.id] = L;
  a->last_lease = L.id;
  out->lease_id = L.id;
  out->slot = slot;
  out->page_table = d.page_tables + (size_t)slot * d.max_requests * d.max_pages;
  return PA_OK;
}

namespace {
pa::arena::Lease* find_lease(kv_arena* a, uint64_t id) {
  const auto it = a->leases.find(id);
  return it == a->leases.end() ? nullptr : &it->second;
}
}  // namespace

extern "C" int kv_lease_attention_done(kv_arena* a, uint64_t lease_id, uint64_t* token) {
  pa::clear_error();
  PA_REQUIRE(a && token, "null pointer argument");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  Lease* L = find_lease(a, lease_id);
  if (!L) return fail(PA_ERR_ORDER, "lease %" PRIu64 " is not live", lease_id);
  if (L->state != kBegun)
    return fail(PA_ERR_ORDER, "lease %" PRIu64 " already has its attention event", lease_id);
  const int rc = op_record(a, a->d.compute_stream, "attn", L->slot, a->ev_attn[L->slot]);
  if (rc != PA_OK) return rc;
  a->last_attn_slot = L->slot;
  L->state = kLeaseAttended;
  L->attention_token = ++a->event_tokens;
  a->slots[L->slot].state = kAttended;
  *token = L->attention_token;
  return PA_OK;
}

extern "C" int kv_lease_writeback(kv_arena* a, uint64_t lease_id, const kv_tail_req* reqs,
                                  int n_reqs, uint64_t* token) {
  pa::clear_error();
  PA_REQUIRE(a && token, "null pointer argument");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  Lease* L = find_lease(a, lease_id);
  if (!L) return fail(PA_ERR_ORDER, "lease %" PRIu64 " is not live", lease_id);
  if (L->state != kLeaseAttended)
    return fail(PA_ERR_ORDER, "lease %" PRIu64 ": write-back needs its attention event first%s",
                lease_id, L->state == kSealed ? " (and the lease is already sealed)" : "");
  std::vector<uint8_t*> src;
  int rc = resolve_tails(a, L->slot, L->layer, reqs, n_reqs, &src);
  if (rc != PA_OK) return rc;
  if ((rc = submit_tails(a, L->slot, reqs, n_reqs, src, &L->written_back_bytes)) != PA_OK)
    return rc;
  L->writeback_token = ++a->event_tokens;
  *token = L->writeback_token;
  return PA_OK;
}

extern "C" int kv_lease_seal(kv_arena* a, uint64_t lease_id, uint64_t attention_token,
                             uint64_t writeback_token) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  Lease* L = find_lease(a, lease_id);
  if (!L) return fail(PA_ERR_ORDER, "lease %" PRIu64 " is not live", lease_id);
  if (L->state == kBegun)
    return fail(PA_ERR_ORDER, "lease %" PRIu64 " has no attention event to seal with", lease_id);
  if (L->state == kSealed) return fail(PA_ERR_ORDER, "lease %" PRIu64 " is already sealed", lease_id);
  if (attention_token != L->attention_token)
    return fail(PA_ERR_ORDER,
                "lease %" PRIu64 ": attention event %" PRIu64 " is not the one recorded (%" PRIu64
                "); a substituted event cannot seal",
                lease_id, attention_token, L->attention_token);
  if (writeback_token != L->writeback_token)
    return fail(PA_ERR_ORDER,
                "lease %" PRIu64 ": tail write-back %" PRIu64 " is not the current one (%" PRIu64
                ")",
                lease_id, writeback_token, L->writeback_token);
  L->state = kSealed;
  return PA_OK;
}

extern "C" int kv_lease_retire(kv_arena* a, uint64_t lease_id, kv_receipt* receipt) {
  pa::clear_error();
  PA_REQUIRE(a && receipt, "null pointer argument");
  if (a->quarantined) return fail(PA_ERR_QUARANTINED, "arena is quarantined; drain it first");
  Lease* L = find_lease(a, lease_id);
  if (!L) return fail(PA_ERR_ORDER, "lease %" PRIu64 " is not live", lease_id);
  if (L->state != kSealed)
    return fail(PA_ERR_ORDER, "lease %" PRIu64 " must be sealed before it is retired", lease_id);
  // Waits that fail quarantine the arena and keep the lease and its tickets.
  int rc;
  const int slot = L->slot;
  if ((rc = op_host_wait(a, "copy", slot, a->ev_copy[slot])) != PA_OK) return rc;
  if ((rc = op_host_wait(a, "attn", slot, a->ev_attn[slot])) != PA_OK) return rc;
  if (L->writeback_token != 0 && (rc = op_host_wait(a, "wb", slot, a->ev_wb[slot])) != PA_OK)
    return rc;
  receipt->lease_id = L->id;
  receipt->layer = L->layer;
  receipt->n_requests = L->n_requests;
  receipt->step = L->step;
  receipt->staged_bytes = L->staged_bytes;
  receipt->written_back_bytes = L->written_back_bytes;
  receipt->tickets_released = static_cast<int32_t>(L->tickets.size());
  for (const Ticket& t : L->tickets) a->owners[t.owner].live_tickets -= 1;
  Slot& S = a->slots[slot];
  if (S.lease_id == L->id) S.retired = true;
  a->leases.erase(lease_id);
  return PA_OK;
}

extern "C" int kv_host_generation(kv_arena* a, uint64_t owner, uint64_t* generation,
                                  int64_t* live_tickets) {
  pa::clear_error();
  PA_REQUIRE(a && generation, "null pointer argument");
  const HostOwner& o = a->owners[owner];
  *generation = o.generation;
  if (live_tickets) *live_tickets = o.live_tickets;
  return PA_OK;
}

extern "C" int kv_host_recycle(kv_arena* a, uint64_t owner, uint64_t* new_generation) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  if (a->quarantined)
    return fail(PA_ERR_QUARANTINED, "arena is quarantined: completion of its copies is unknown");
  HostOwner& o = a->owners[owner];
  if (o.live_tickets > 0)
    return fail(PA_ERR_ORDER,
                "host pages of owner %" PRIu64 " are held by %" PRId64
                " copy ticket(s); retire those leases first",
                owner, o.live_tickets);
  o.generation += 1;
  if (new_generation) *new_generation = o.generation;
  return PA_OK;
}

extern "C" int kv_arena_get_stats(const kv_arena* a, kv_arena_stats* out) {
  pa::clear_error();
  PA_REQUIRE(a && out, "null pointer argument");
  out->stage_generation = a->generation;
  out->staged_bytes = a->staged_bytes;
  out->written_back_bytes = a->written_back_bytes;
  out->slot_reuses = a->slot_reuses;
  out->quarantined = a->quarantined ? 1 : 0;
  out->n_slots = a->d.n_slots;
  out->loaded_bytes = a->loaded_bytes;
  return PA_OK;
}

extern "C" int kv_arena_fail_after(kv_arena* a, int64_t n) {
  pa::clear_error();
  PA_REQUIRE(a, "null arena");
  a->fail_after = n;
  return PA_OK;
}

extern "C" size_t kv_arena_call_log(const kv_arena* a, char* buf, size_t buf_bytes) {
  if (!a) return 0;
  if (buf && buf_bytes) {
    const size_t n = std::min(buf_bytes - 1, a->log.size());
    std::memcpy(buf, a->log.data(), n);
    buf[n] = '\0';
  }
  return a->log.size();
}
