// Admission planner: which pages of each context are device-resident.
//
// Sources: "Staging without a stall", section "Admission that does
// arithmetic"; "GPU memory management", sections "Pages held by right,
// borrowed or free" and "A host pool that explains its own size".
//
//   * The device page pool is an explicit whole number of GiB; an automatic
//     size is refused.  One pool page holds one 64-token logical page of one
//     context for every dense layer.
//   * Each context has a target it holds by right, an optional burst it may
//     borrow while pages are free, and a floor of the sink pages plus one.
//   * Each step the planner computes the pages a context wants hot (the sink
//     plus its newest pages), and fills each missing one in order: reuse one
//     of the context's own pages that left its window, take a free page,
//     reclaim (only while the context is below its target), or else shrink
//     the window from its oldest page, keeping the tail hot.
//   * Reclamation takes, least-recently-active first: borrowed pages, then
//     other pages above a target, then whole idle contexts; a context that
//     cannot reach its floor is refused for the step.
//   * Every decision is counted; pages that turn hot are copied in once.
//   * Host pool fit: concurrency = min(limit, floor(pool / (layers x context
//     length x row bytes))), reported with its formula; refuse mode stops when
//     the geometry does not fit, shrink mode lowers the concurrency.
#include <algorithm>
#include <cinttypes>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "common.h"

namespace pa {
namespace planner {

struct Ctx {
  uint64_t id = 0;
  int target = 0;
  int burst = 0;
  int64_t length = 0;
  int64_t last_active = 0;
  uint64_t order = 0;                   // admission order (ties in LRU)
  std::map<int32_t, int32_t> pages;     // logical page -> pool page
  int borrowed = 0;                     // pages held beyond the target as burst
  std::vector<int32_t> copied;          // pages made resident at the last step
  bool refused = false;
};

}  // namespace planner
}  // namespace pa

struct kv_planner {
  kv_planner_desc d{};
  int64_t pool_pages = 0;
  int concurrency = 0;
  std::string formula;
  std::map<uint64_t, pa::planner::Ctx> ctxs;
  std::set<int32_t> free_pages;
  int64_t step = 0;
  uint64_t admissions = 0;
  kv_planner_counters c{};
};

namespace pa {
namespace planner {
namespace {

int n_pages_of(const kv_planner* P, int64_t length) {
  return static_cast<int>((length + P->d.page_tokens - 1) / P->d.page_tokens);
}

int floor_of(const kv_planner* P, const Ctx& c) {
  const int n = n_pages_of(P, c.length);
  return std::min(n, std::min(P->d.sink_pages, n) + 1);
}

// Oldest logical page of c that is not a sink page (the shrink victim).
int32_t oldest_victim(const kv_planner* P, const Ctx& c) {
  for (const auto& kv : c.pages)
    if (kv.first >= P->d.sink_pages) return kv.first;
  return -1;
}

// Keeps the borrowed count within the pages actually held beyond the target.
void clamp_borrowed(Ctx& c) {
  c.borrowed = std::max(0, std::min(c.borrowed, (int)c.pages.size() - c.target));
}

void drop_page(kv_planner* P, Ctx& c, int32_t logical) {
  const auto it = c.pages.find(logical);
  if (it == c.pages.end()) return;
  P->free_pages.insert(it->second);
  c.pages.erase(it);
}

bool lru_less(const Ctx& a, const Ctx& b) {
  if (a.last_active != b.last_active) return a.last_active < b.last_active;
  return a.order < b.order;
}

// Frees one pool page for `needer` by reclamation; false if nothing may be
// taken.  Active contexts of this step are in `active`.
bool reclaim_one(kv_planner* P, const Ctx& needer, const std::set<uint64_t>& active) {
  auto victims = [&](auto pred) {
    std::vector<Ctx*> v;
    for (auto& kv : P->ctxs)
      if (kv.first != needer.id && pred(kv.second)) v.push_back(&kv.second);
    std::sort(v.begin(), v.end(), [](const Ctx* a, const Ctx* b) { return lru_less(*a, *b); });
    return v;
  };
  // Victims always give their oldest non-sink page, so their tail stays hot.
  // 1. borrowed pages (burst beyond a target), least recently active first
  for (Ctx* v : victims([](const Ctx& c) { return c.borrowed > 0; })) {
    const int32_t lp = oldest_victim(P, *v);
    if (lp < 0) continue;
    drop_page(P, *v, lp);
    v->borrowed -= 1;
    clamp_borrowed(*v);
    P->c.reclaimed_borrowed += 1;
    return true;
  }
  // 2. other pages above a target (a target lowered after the pages were taken)
  for (Ctx* v : victims([](const Ctx& c) { return (int)c.pages.size() - c.borrowed > c.target; })) {
    const int32_t lp = oldest_victim(P, *v);
    if (lp < 0) continue;
    drop_page(P, *v, lp);
    clamp_borrowed(*v);
    P->c.reclaimed_above_target += 1;
    return true;
  }
  // 3. whole idle contexts (not stepping now)
  for (Ctx* v : victims([&](const Ctx& c) { return !active.count(c.id) && !c.pages.empty(); })) {
    P->c.reclaimed_idle_contexts += 1;
    P->c.reclaimed_idle_pages += v->pages.size();
    std::vector<int32_t> all;
    for (const auto& kv : v->pages) all.push_back(kv.first);
    for (int32_t lp : all) drop_page(P, *v, lp);
    v->borrowed = 0;
    return true;
  }
  return false;
}

}  // namespace
}  // namespace planner
}  // namespace pa

using pa::fail;
using namespace pa::planner;

extern "C" int kv_planner_create(const kv_planner_desc* desc, kv_planner** out, char* formula,
                                 size_t formula_bytes) {
  pa::clear_error();
  PA_REQUIRE(desc && out, "null pointer argument");
  *out = nullptr;
  const kv_planner_desc& d = *desc;
  PA_REQUIRE(d.pool_gib >= 1,
             "the device page pool must be an explicit whole number of GiB (got %u); an "
             "automatic size is refused",
             d.pool_gib);
  PA_REQUIRE(d.n_layers >= 1 && d.row_bytes > 0 && d.page_tokens >= 1, "bad geometry");
  PA_REQUIRE(d.sink_pages >= 0, "sink_pages must be >= 0");
  PA_REQUIRE(d.max_contexts >= 1, "max_contexts must be >= 1");
  PA_REQUIRE(d.max_context_tokens >= 1, "max_context_tokens must be >= 1");
  const uint64_t page_all_layers = (uint64_t)d.n_layers * d.page_tokens * d.row_bytes;
  const int64_t pool_pages = (int64_t)(((uint64_t)d.pool_gib << 30) / page_all_layers);
  PA_REQUIRE(pool_pages >= 1 && pool_pages < (1ll << 31), "pool of %u GiB holds %" PRId64 " pages",
             d.pool_gib, pool_pages);
  const uint64_t history = (uint64_t)d.n_layers * (uint64_t)d.max_context_tokens * d.row_bytes;
  const uint64_t fits = d.host_pool_bytes / history;
  const int concurrency = (int)std::min<uint64_t>((uint64_t)d.max_contexts, fits);
  char buf[512];
  snprintf(buf, sizeof(buf),
           "concurrency = min(max_contexts=%d, floor(host_pool_bytes=%" PRIu64
           " / (n_layers=%d x max_context_tokens=%" PRId64 " x row_bytes=%d))) = min(%d, %" PRIu64
           ") = %d; device pool = %u GiB / (%d x %d x %d B) = %" PRId64 " pages",
           d.max_contexts, d.host_pool_bytes, d.n_layers, d.max_context_tokens, d.row_bytes,
           d.max_contexts, fits, concurrency, d.pool_gib, d.n_layers, d.page_tokens, d.row_bytes,
           pool_pages);
  if (formula && formula_bytes) {
    strncpy(formula, buf, formula_bytes - 1);
    formula[formula_bytes - 1] = '\0';
  }
  if ((uint64_t)d.max_contexts > fits && !d.shrink_mode)
    return fail(PA_ERR_INVALID,
                "host pool does not fit: %s; raise host_pool_bytes to %" PRIu64
                " or lower max_contexts to %" PRIu64 " (or use shrink mode)",
                buf, history * (uint64_t)d.max_contexts, fits);
  if (concurrency < 1)
    return fail(PA_ERR_INVALID, "host pool holds no history: %s; raise host_pool_bytes to %" PRIu64,
                buf, history);
  kv_planner* P = new kv_planner;
  P->d = d;
  P->pool_pages = pool_pages;
  P->concurrency = concurrency;
  P->formula = buf;
  for (int32_t i = 0; i < pool_pages; ++i) P->free_pages.insert(i);
  *out = P;
  return PA_OK;
}

extern "C" int kv_planner_destroy(kv_planner* P) {
  delete P;
  return PA_OK;
}

extern "C" int kv_planner_info(const kv_planner* P, int64_t* pool_pages, int* concurrency,
                               char* formula, size_t formula_bytes) {
  pa::clear_error();
  PA_REQUIRE(P, "null planner");
  if (pool_pages) *pool_pages = P->pool_pages;
  if (concurrency) *concurrency = P->concurrency;
  if (formula && formula_bytes) {
    strncpy(formula, P->formula.c_str(), formula_bytes - 1);
    formula[formula_bytes - 1] = '\0';
  }
  return PA_OK;
}

extern "C" int kv_planner_admit(kv_planner* P, uint64_t ctx, int target_pages, int burst_pages) {
  pa::clear_error();
  PA_REQUIRE(P, "null planner");
  PA_REQUIRE(target_pages >= 0 && burst_pages >= 0, "target and burst must be >= 0");
  PA_REQUIRE(!P->ctxs.count(ctx), "context %" PRIu64 " is already admitted", ctx);
  if ((int)P->ctxs.size() >= P->concurrency)
    return fail(PA_ERR_REFUSED, "concurrency %d reached (%s); the serving layer queues context %" PRIu64,
                P->concurrency, P->formula.c_str(), ctx);
  Ctx c;
  c.id = ctx;
  c.target = target_pages;
  c.burst = burst_pages;
  c.order = ++P->admissions;
  P->ctxs[ctx] = c;
  return PA_OK;
}

extern "C" int kv_planner_set_target(kv_planner* P, uint64_t ctx, int target_pages,
                                     int burst_pages) {
  pa::clear_error();
  PA_REQUIRE(P, "null planner");
  PA_REQUIRE(target_pages >= 0 && burst_pages >= 0, "target and burst must be >= 0");
  const auto it = P->ctxs.find(ctx);
  PA_REQUIRE(it != P->ctxs.end(), "context %" PRIu64 " is not admitted", ctx);
  it->second.target = target_pages;
  it->second.burst = burst_pages;
  return PA_OK;
}

extern "C" int kv_planner_release(kv_planner* P, uint64_t ctx) {
  pa::clear_error();
  PA_REQUIRE(P, "null planner");
  const auto it = P->ctxs.find(ctx);
  PA_REQUIRE(it != P->ctxs.end(), "context %" PRIu64 " is not admitted", ctx);
  for (const auto& kv : it->second.pages) P->free_pages.insert(kv.second);
  P->ctxs.erase(it);
  return PA_OK;
}

extern "C" int kv_planner_step(kv_planner* P, const uint64_t* ctx_ids, const int64_t* lengths,
                               int n, int32_t* admitted) {
  pa::clear_error();
  PA_REQUIRE(P, "null planner");
  PA_REQUIRE(n >= 0 && (n == 0 || (ctx_ids && lengths)), "bad context list");
  std::set<uint64_t> active;
  for (int i = 0; i < n; ++i) {
    const auto it = P->ctxs.find(ctx_ids[i]);
    PA_REQUIRE(it != P->ctxs.end(), "context %" PRIu64 " is not admitted", ctx_ids[i]);
    PA_REQUIRE(lengths[i] >= 1, "context %" PRIu64 ": length must be >= 1", ctx_ids[i]);
    PA_REQUIRE(!active.count(ctx_ids[i]), "context %" PRIu64 " listed twice", ctx_ids[i]);
    active.insert(ctx_ids[i]);
  }
  ++P->step;
  P->c.steps += 1;
  for (int i = 0; i < n; ++i) {
    Ctx& c = P->ctxs[ctx_ids[i]];
    c.length = lengths[i];
    c.last_active = P->step;
    c.copied.clear();
    c.refused = false;
  }
  const int sink = P->d.sink_pages;
  for (int i = 0; i < n; ++i) {
    Ctx& c = P->ctxs[ctx_ids[i]];
    const int np = n_pages_of(P, c.length);
    const int want = std::min(np, c.target + c.burst);
    const int n_sink = std::min(sink, np);
    // Desired hot pages, in fill priority: the sink, then newest to oldest.
    std::vector<int32_t> desired;
    for (int32_t p = 0; p < n_sink; ++p) desired.push_back(p);
    for (int32_t p = np - 1; p >= n_sink && (int)desired.size() < want; --p) desired.push_back(p);
    std::set<int32_t> desired_set(desired.begin(), desired.end());
    // Own pages that left the window are reusable first.
    std::vector<int32_t> own_spare;
    for (const auto& kv : c.pages)
      if (!desired_set.count(kv.first)) own_spare.push_back(kv.first);
    size_t held = 0;
    for (int32_t p : desired)
      if (c.pages.count(p)) ++held;
    for (size_t k = 0; k < desired.size(); ++k) {
      const int32_t lp = desired[k];
      if (c.pages.count(lp)) continue;
      int32_t pool = -1;
      bool taken_from_window = false;
      if (!own_spare.empty()) {
        const int32_t old = own_spare.front();
        own_spare.erase(own_spare.begin());
        pool = c.pages[old];
        c.pages.erase(old);
        P->c.reused_own += 1;
      } else if (!P->free_pages.empty()) {
        pool = *P->free_pages.begin();
        P->free_pages.erase(P->free_pages.begin());
        P->c.took_free += 1;
      } else if ((int)held < c.target && reclaim_one(P, c, active)) {
        pool = *P->free_pages.begin();
        P->free_pages.erase(P->free_pages.begin());
      } else {
        // Shrink from the oldest page, keeping the tail hot: the context's
        // oldest non-sink resident page older than lp gives up its pool page.
        int32_t victim = -1;
        for (const auto& kv : c.pages) {
          if (kv.first >= sink && kv.first < lp) {
            victim = kv.first;
            break;
          }
        }
        if (victim < 0) break;  // nothing older to give: the rest stays cold
        pool = c.pages[victim];
        c.pages.erase(victim);
        taken_from_window = true;
      }
      if (!taken_from_window) ++held;
      c.pages[lp] = pool;
      if (!taken_from_window && (int)held > c.target) c.borrowed += 1;
      c.copied.push_back(lp);
    }
    for (int32_t p : desired)
      if (!c.pages.count(p)) P->c.shrunk_pages += 1;
    for (int32_t old : own_spare) drop_page(P, c, old);
    clamp_borrowed(c);
    // A refused context keeps what it holds and retries at the next step.
    const bool ok = (int)c.pages.size() >= floor_of(P, c);
    c.refused = !ok;
    if (!ok) P->c.refused += 1;
    if (admitted) admitted[i] = ok ? 1 : 0;
  }
  // A page made hot for one context may have been reclaimed by a later one
  // in the same step: only pages still resident at the boundary are copied.
  for (int i = 0; i < n; ++i) {
    Ctx& c = P->ctxs[ctx_ids[i]];
    std::vector<int32_t> kept;
    for (int32_t lp : c.copied)
      if (c.pages.count(lp)) kept.push_back(lp);
    c.copied.swap(kept);
    P->c.copied_in += c.copied.size();
  }
  return PA_OK;
}

extern "C" int kv_planner_resident(const kv_planner* P, uint64_t ctx, int32_t* logical,
                                   int32_t* pool, int cap, int* n_out) {
  pa::clear_error();
  PA_REQUIRE(P && n_out, "null pointer argument");
  const auto it = P->ctxs.find(ctx);
  PA_REQUIRE(it != P->ctxs.end(), "context %" PRIu64 " is not admitted", ctx);
  int k = 0;
  for (const auto& kv : it->second.pages) {
    if (k < cap) {
      if (logical) logical[k] = kv.first;
      if (pool) pool[k] = kv.second;
    }
    ++k;
  }
  *n_out = k;
  return PA_OK;
}

extern "C" int kv_planner_copied(const kv_planner* P, uint64_t ctx, int32_t* logical, int cap,
                                 int* n_out) {
  pa::clear_error();
  PA_REQUIRE(P && n_out, "null pointer argument");
  const auto it = P->ctxs.find(ctx);
  PA_REQUIRE(it != P->ctxs.end(), "context %" PRIu64 " is not admitted", ctx);
  const auto& v = it->second.copied;
  for (int k = 0; k < (int)v.size() && k < cap; ++k)
    if (logical) logical[k] = v[k];
  *n_out = (int)v.size();
  return PA_OK;
}

extern "C" int kv_planner_get_counters(const kv_planner* P, kv_planner_counters* out) {
  pa::clear_error();
  PA_REQUIRE(P && out, "null pointer argument");
  *out = P->c;
  out->free_pages = (int64_t)P->free_pages.size();
  return PA_OK;
}
