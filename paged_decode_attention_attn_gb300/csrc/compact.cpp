// Compact older pages: a second, smaller representation of history pages that
// are fully written in every layer, converted by background threads, checked
// by a CRC and published; until a page is published it is served exact.
//
// Sources ("KV-cache engineering", sections "Exact recent pages, compact older
// pages" and "What the hybrid tier buys"): the planner cuts a request into runs
// of two representations; background threads convert a page only after it is
// fully written in every layer, compute a CRC and publish it; a representation
// is judged by the bytes per token it stops moving over the bus.
//
// The pages name no format.  This library's reading: for every token row and
// every (K or V, kv head) slice of head_dim bf16 values, a binary32 scale
// s = max|x| / 127 and int8 codes round_half_even(x / s) clamped to +-127 (a
// zero slice has s = 0 and zero codes; a page with a non-finite value is not
// convertible).  A compact page is the codes [64][2 Hkv D] then the scales
// [64][2 Hkv] (float32, little-endian), and stands for bf16_rne(c * s).  The
// CRC is CRC-32 (reflected polynomial 0xEDB88320, initial value and final xor
// 0xFFFFFFFF) of those bytes.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <mutex>
#include <thread>
#include <vector>

#include "common.h"

namespace pa {
namespace compact {

constexpr int kCodeMax = PA_COMPACT_CODE_MAX;

float bf16_to_f32(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return f;
}

// CRC-32 tables for slicing by 8: table[0] is the byte-at-a-time table of the
// reflected polynomial; table[k][i] advances table[k-1][i] by one zero byte.
struct CrcTables {
  uint32_t t[8][256];
  CrcTables() {
    for (uint32_t i = 0; i < 256; ++i) {
      uint32_t c = i;
      for (int k = 0; k < 8; ++k) c = (c & 1u) ? (c >> 1) ^ 0xEDB88320u : c >> 1;
      t[0][i] = c;
    }
    for (uint32_t i = 0; i < 256; ++i)
      for (int k = 1; k < 8; ++k) t[k][i] = (t[k - 1][i] >> 8) ^ t[0][t[k - 1][i] & 0xFFu];
  }
};

const CrcTables& crc_tables() {
  static const CrcTables tables;
  return tables;
}

uint32_t crc32(const uint8_t* p, size_t n, uint32_t crc) {
  const CrcTables& T = crc_tables();
  uint32_t c = crc ^ 0xFFFFFFFFu;
  // Eight bytes per step: the low four are folded into the running value,
  // each byte then looked up in the table that advances it to the end of the
  // eight-byte block.  Bytes are assembled explicitly (no endianness assumption).
  while (n >= 8) {
    const uint32_t lo = c ^ (uint32_t(p[0]) | uint32_t(p[1]) << 8 | uint32_t(p[2]) << 16 |
                             uint32_t(p[3]) << 24);
    c = T.t[7][lo & 0xFFu] ^ T.t[6][(lo >> 8) & 0xFFu] ^ T.t[5][(lo >> 16) & 0xFFu] ^
        T.t[4][lo >> 24] ^ T.t[3][p[4]] ^ T.t[2][p[5]] ^ T.t[1][p[6]] ^ T.t[0][p[7]];
    p += 8;
    n -= 8;
  }
  while (n--) c = T.t[0][(c ^ *p++) & 0xFFu] ^ (c >> 8);
  return c ^ 0xFFFFFFFFu;
}

size_t page_bytes(int n_kv_heads, int head_dim) {
  const size_t slices = 2 * (size_t)n_kv_heads;
  return (size_t)PA_PAGE_TOKENS * slices * head_dim + (size_t)PA_PAGE_TOKENS * slices * 4;
}

// One layer's page: 64 rows of bf16 [2 Hkv D] -> codes then scales.  Returns
// false (nothing guaranteed about out) if a value is not finite.
bool convert_page(const uint16_t* rows, int n_kv_heads, int head_dim, uint8_t* out) {
  const int slices = 2 * n_kv_heads;
  const int row_elems = slices * head_dim;
  int8_t* codes = reinterpret_cast<int8_t*>(out);
  uint8_t* scale_bytes = out + (size_t)PA_PAGE_TOKENS * row_elems;
  for (int t = 0; t < PA_PAGE_TOKENS; ++t) {
    for (int k = 0; k < slices; ++k) {
      const uint16_t* x = rows + (size_t)t * row_elems + (size_t)k * head_dim;
      int8_t* c = codes + (size_t)t * row_elems + (size_t)k * head_dim;
      float amax = 0.f;
      for (int d = 0; d < head_dim; ++d) {
        const float v = bf16_to_f32(x[d]);
        if (!std::isfinite(v)) return false;
        amax = std::max(amax, std::fabs(v));
      }
      const float s = amax / static_cast<float>(kCodeMax);   // binary32, nearest even
      for (int d = 0; d < head_dim; ++d) {
        if (s > 0.f) {
          const float q = std::nearbyint(bf16_to_f32(x[d]) / s);  // half to even
          c[d] = static_cast<int8_t>(std::min<float>(kCodeMax, std::max<float>(-kCodeMax, q)));
        } else {
          c[d] = 0;
        }
      }
      uint32_t su;
      std::memcpy(&su, &s, sizeof(su));
      uint8_t* sb = scale_bytes + ((size_t)t * slices + k) * 4;
      sb[0] = su & 0xFFu;
      sb[1] = (su >> 8) & 0xFFu;
      sb[2] = (su >> 16) & 0xFFu;
      sb[3] = su >> 24;
    }
  }
  return true;
}

}  // namespace compact
}  // namespace pa

struct kv_compactor {
  kv_compactor_desc d{};
  std::vector<const uint8_t*> exact;   // [layer * n_requests + request]
  std::vector<uint8_t*> store;         // [layer * n_requests + request]
  size_t row_bytes = 0;
  size_t cpage_bytes = 0;
  std::vector<std::atomic<uint8_t>> state;   // [request * max_pages + page]
  std::vector<uint32_t> crc;                 // [(request * max_pages + page) * n_layers + layer]
  mutable std::mutex mu;
  std::condition_variable cv_work, cv_idle;
  std::deque<int64_t> jobs;            // request * max_pages + page
  int active = 0;
  bool hold = false;
  bool stop = false;
  std::atomic<uint64_t> published{0}, not_convertible{0}, compact_bytes{0};
  std::vector<std::thread> workers;

  explicit kv_compactor(size_t n_pages) : state(n_pages) {}

  void run() {
    for (;;) {
      int64_t job;
      {
        std::unique_lock<std::mutex> lk(mu);
        cv_work.wait(lk, [&] { return stop || (!hold && !jobs.empty()); });
        if (stop) return;
        job = jobs.front();
        jobs.pop_front();
        ++active;
      }
      convert(job);
      {
        std::lock_guard<std::mutex> lk(mu);
        --active;
        if (active == 0 && (jobs.empty() || hold)) cv_idle.notify_all();
      }
    }
  }

  // Converts every layer of one page, then publishes it (or marks it not
  // convertible).  The CRCs are written before the state's release store.
  void convert(int64_t job) {
    const int r = static_cast<int>(job / d.max_pages);
    const int page = static_cast<int>(job % d.max_pages);
    bool ok = true;
    for (int l = 0; l < d.n_layers && ok; ++l) {
      const size_t idx = (size_t)l * d.n_requests + r;
      const uint16_t* rows = reinterpret_cast<const uint16_t*>(
          exact[idx] + (size_t)page * PA_PAGE_TOKENS * row_bytes);
      uint8_t* out = store[idx] + (size_t)page * cpage_bytes;
      ok = pa::compact::convert_page(rows, d.n_kv_heads, d.head_dim, out);
      if (ok) crc[(size_t)job * d.n_layers + l] = pa::compact::crc32(out, cpage_bytes, 0);
    }
    if (ok) {
      compact_bytes += (uint64_t)cpage_bytes * d.n_layers;
      published += 1;
      state[job].store(PA_PAGE_PUBLISHED, std::memory_order_release);
    } else {
      not_convertible += 1;
      state[job].store(PA_PAGE_NOT_CONVERTIBLE, std::memory_order_release);
    }
  }
};

using pa::fail;

extern "C" size_t kv_compact_page_bytes(int n_kv_heads, int head_dim) {
  if (n_kv_heads < 1 || head_dim < 16 || head_dim % 16 != 0) return 0;
  return pa::compact::page_bytes(n_kv_heads, head_dim);
}

extern "C" uint32_t kv_crc32(const void* data, size_t bytes, uint32_t crc) {
  if (!data) return crc;
  return pa::compact::crc32(static_cast<const uint8_t*>(data), bytes, crc);
}

extern "C" int kv_compact_convert_page(const void* rows, int n_kv_heads, int head_dim,
                                       void* out, uint32_t* crc) {
  pa::clear_error();
  PA_REQUIRE(rows && out, "null pointer argument");
  PA_REQUIRE(kv_compact_page_bytes(n_kv_heads, head_dim) > 0,
             "n_kv_heads (%d) must be >= 1 and head_dim (%d) a positive multiple of 16",
             n_kv_heads, head_dim);
  if (!pa::compact::convert_page(static_cast<const uint16_t*>(rows), n_kv_heads, head_dim,
                                 static_cast<uint8_t*>(out)))
    return fail(PA_ERR_INVALID, "page holds a non-finite value: not convertible");
  if (crc)
    *crc = pa::compact::crc32(static_cast<const uint8_t*>(out),
                              pa::compact::page_bytes(n_kv_heads, head_dim), 0);
  return PA_OK;
}

extern "C" int kv_compactor_create(const kv_compactor_desc* desc, kv_compactor** out) {
  pa::clear_error();
  PA_REQUIRE(desc && out, "null pointer argument");
  *out = nullptr;
  const kv_compactor_desc& d = *desc;
  PA_REQUIRE(d.n_layers >= 1 && d.n_requests >= 1 && d.max_pages >= 1,
             "n_layers, n_requests and max_pages must be >= 1");
  PA_REQUIRE(kv_compact_page_bytes(d.n_kv_heads, d.head_dim) > 0, "unsupported geometry");
  PA_REQUIRE(d.n_threads >= 1 && d.n_threads <= 256, "n_threads (%d) must be in 1..256",
             d.n_threads);
  PA_REQUIRE(d.exact_rows && d.compact_pages, "exact_rows and compact_pages are required");
  const size_t n = (size_t)d.n_layers * d.n_requests;
  for (size_t i = 0; i < n; ++i)
    PA_REQUIRE(d.exact_rows[i] && d.compact_pages[i], "null segment address at %zu", i);
  kv_compactor* c = new kv_compactor((size_t)d.n_requests * d.max_pages);
  c->d = d;
  c->exact.assign(n, nullptr);
  c->store.assign(n, nullptr);
  for (size_t i = 0; i < n; ++i) {
    c->exact[i] = static_cast<const uint8_t*>(d.exact_rows[i]);
    c->store[i] = static_cast<uint8_t*>(d.compact_pages[i]);
  }
  c->d.exact_rows = nullptr;     // the copies above are the ones used
  c->d.compact_pages = nullptr;
  c->row_bytes = (size_t)4 * d.n_kv_heads * d.head_dim;
  c->cpage_bytes = pa::compact::page_bytes(d.n_kv_heads, d.head_dim);
  c->crc.assign((size_t)d.n_requests * d.max_pages * d.n_layers, 0);
  for (auto& s : c->state) s.store(PA_PAGE_EXACT, std::memory_order_relaxed);
  try {
    for (int i = 0; i < d.n_threads; ++i) c->workers.emplace_back([c] { c->run(); });
  } catch (...) {
    kv_compactor_destroy(c);
    return fail(PA_ERR_INVALID, "cannot start %d converter threads", d.n_threads);
  }
  *out = c;
  return PA_OK;
}

extern "C" int kv_compactor_destroy(kv_compactor* c) {
  pa::clear_error();
  if (!c) return PA_OK;
  {
    std::lock_guard<std::mutex> lk(c->mu);
    c->stop = true;
  }
  c->cv_work.notify_all();
  for (auto& t : c->workers)
    if (t.joinable()) t.join();     // a page in progress finishes first (milliseconds)
  delete c;
  return PA_OK;
}

extern "C" int kv_compactor_mark_written(kv_compactor* c, int request, int full_pages) {
  pa::clear_error();
  PA_REQUIRE(c, "null compactor");
  PA_REQUIRE(request >= 0 && request < c->d.n_requests, "request %d outside [0, %d)", request,
             c->d.n_requests);
  PA_REQUIRE(full_pages >= 0 && full_pages <= c->d.max_pages, "full_pages %d outside [0, %d]",
             full_pages, c->d.max_pages);
  int queued = 0;
  {
    std::lock_guard<std::mutex> lk(c->mu);
    for (int p = 0; p < full_pages; ++p) {
      const int64_t job = (int64_t)request * c->d.max_pages + p;
      uint8_t expect = PA_PAGE_EXACT;
      if (c->state[job].compare_exchange_strong(expect, PA_PAGE_QUEUED)) {
        c->jobs.push_back(job);
        ++queued;
      }
    }
  }
  if (queued) c->cv_work.notify_all();
  return PA_OK;
}

extern "C" int kv_compactor_hold(kv_compactor* c, int hold) {
  pa::clear_error();
  PA_REQUIRE(c, "null compactor");
  {
    std::lock_guard<std::mutex> lk(c->mu);
    c->hold = hold != 0;
  }
  c->cv_work.notify_all();
  c->cv_idle.notify_all();   // a waiter for idleness re-checks: held counts as idle
  return PA_OK;
}

extern "C" int kv_compactor_wait_idle(kv_compactor* c, int timeout_ms) {
  pa::clear_error();
  PA_REQUIRE(c, "null compactor");
  PA_REQUIRE(timeout_ms >= 0, "timeout_ms must be >= 0");
  std::unique_lock<std::mutex> lk(c->mu);
  const bool idle = c->cv_idle.wait_for(lk, std::chrono::milliseconds(timeout_ms), [&] {
    return c->active == 0 && (c->jobs.empty() || c->hold);
  });
  if (!idle) return fail(PA_ERR_TIMEOUT, "converter not idle after %d ms", timeout_ms);
  if (!c->jobs.empty())
    return fail(PA_ERR_ORDER, "converter is held with %zu pages queued", c->jobs.size());
  return PA_OK;
}

extern "C" int kv_compactor_states(const kv_compactor* c, int request, int first_page,
                                   int n_pages, uint8_t* states) {
  pa::clear_error();
  PA_REQUIRE(c && states, "null pointer argument");
  PA_REQUIRE(request >= 0 && request < c->d.n_requests, "request %d outside [0, %d)", request,
             c->d.n_requests);
  PA_REQUIRE(first_page >= 0 && n_pages >= 0 && (int64_t)first_page + n_pages <= c->d.max_pages,
             "pages [%d, +%d) outside [0, %d)", first_page, n_pages, c->d.max_pages);
  for (int i = 0; i < n_pages; ++i)
    states[i] = c->state[(size_t)request * c->d.max_pages + first_page + i].load(
        std::memory_order_acquire);
  return PA_OK;
}

extern "C" int kv_compactor_crc(const kv_compactor* c, int layer, int request, int page,
                                uint32_t* crc) {
  pa::clear_error();
  PA_REQUIRE(c && crc, "null pointer argument");
  PA_REQUIRE(layer >= 0 && layer < c->d.n_layers && request >= 0 && request < c->d.n_requests &&
                 page >= 0 && page < c->d.max_pages,
             "layer %d, request %d or page %d out of range", layer, request, page);
  const size_t job = (size_t)request * c->d.max_pages + page;
  if (c->state[job].load(std::memory_order_acquire) != PA_PAGE_PUBLISHED)
    return fail(PA_ERR_ORDER, "page %d of request %d is not published", page, request);
  *crc = c->crc[job * c->d.n_layers + layer];
  return PA_OK;
}

extern "C" int kv_compactor_verify(const kv_compactor* c, int request, int page) {
  pa::clear_error();
  PA_REQUIRE(c, "null compactor");
  PA_REQUIRE(request >= 0 && request < c->d.n_requests && page >= 0 && page < c->d.max_pages,
             "request %d or page %d out of range", request, page);
  const size_t job = (size_t)request * c->d.max_pages + page;
  if (c->state[job].load(std::memory_order_acquire) != PA_PAGE_PUBLISHED)
    return fail(PA_ERR_ORDER, "page %d of request %d is not published", page, request);
  for (int l = 0; l < c->d.n_layers; ++l) {
    const uint8_t* p = c->store[(size_t)l * c->d.n_requests + request] + page * c->cpage_bytes;
    const uint32_t got = pa::compact::crc32(p, c->cpage_bytes, 0);
    if (got != c->crc[job * c->d.n_layers + l])
      return fail(PA_ERR_CRC, "layer %d page %d of request %d: CRC %08x, published %08x", l,
                  page, request, got, c->crc[job * c->d.n_layers + l]);
  }
  return PA_OK;
}

extern "C" int kv_compactor_get_counters(const kv_compactor* c, kv_compactor_counters* out) {
  pa::clear_error();
  PA_REQUIRE(c && out, "null pointer argument");
  out->published_pages = c->published.load();
  out->not_convertible_pages = c->not_convertible.load();
  out->compact_bytes = c->compact_bytes.load();
  {
    std::lock_guard<std::mutex> lk(c->mu);
    out->queued_pages = c->jobs.size() + c->active;
  }
  return PA_OK;
}
