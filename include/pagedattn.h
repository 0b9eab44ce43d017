/*
 * pagedattn.h -- C ABI of libpagedattn: paged GQA decode attention with a
 * per-tile log-sum-exp, an FP32 LSE merge, a staging arena that moves KV
 * history from pinned host memory into bounded device slots (stage calls or
 * leases), an admission planner for a device pool, and a background converter
 * of fully written pages into a compact representation.
 *
 * Sources (web pages, cited by title and section):
 *   [KVE-exact]  "KV-cache engineering", section "Exact recent pages, compact
 *                older pages": tiles each return a normalised output and its
 *                log-sum-exp; an FP32 merge weights each by exp(LSE_i - max),
 *                sums, divides by the summed weights, LSE = max + log(sum).
 *   [KVE-bus]    "KV-cache engineering", section "Costing the bus before
 *                changing anything": pinned host memory owns the cache, the
 *                device keeps a bounded working set, the exact path re-reads
 *                every history byte per generated token.
 *   [KVE-lease]  "KV-cache engineering", section "Staging layers under a lease".
 *   [SWS-queues] "Staging without a stall", section "Two copy queues and
 *                device-side ordering": dedicated H2D and D2H queues; compute
 *                waits on an event recorded after the history copy; write-back
 *                waits on an event recorded after attention; the host never
 *                blocks on the hot path.
 *   [SWS-lease]  "Staging without a stall", section "Leases instead of
 *                buffers": a buffer is reused only after the previous
 *                attention and write-back that read it; only changed rows go
 *                back to the pinned host rows; a different host owner is
 *                refused; any failure quarantines the transport; the
 *                destructor never waits.
 *   [SWS-admit]  "Staging without a stall", section "Admission that does
 *                arithmetic": one explicit device allocation, sink page plus
 *                newest pages kept hot.
 *   [GMM-host]   "GPU memory management", section "A host pool that explains
 *                its own size": a history is, per layer, a segment of
 *                context length x 4,096 bytes.
 *   [KVE-tier]   "KV-cache engineering", section "What the hybrid tier buys":
 *                a representation is judged by the bytes per token it stops
 *                moving over the bus.
 *
 * Conventions for every entry point:
 *   - All memory is allocated and owned by the caller.  The library keeps raw
 *     pointers only for the lifetime the call documents and never frees them.
 *   - Streams are the caller's.  Kernels and copies are enqueued
 *     asynchronously; no entry point waits for the device except
 *     kv_arena_drain and kv_lease_retire (documented host waits);
 *     kv_compactor_wait_idle and kv_compactor_destroy wait for the library's
 *     converter threads, never for the device.
 *   - Return value: PA_OK (0) or a negative PA_ERR_* code; a thread-local
 *     message is available from kv_last_error().  No C++ exception crosses
 *     the ABI.
 *   - Layouts are dense row-major in the order the brackets list.
 *   - Threads: the decode, merge and row-append entry points keep no state
 *     between calls (except the fixed scratch of the _noalloc variant) and
 *     may be called from several host threads.  An arena, planner or
 *     compactor handle is used by one thread at a time (the caller
 *     serialises); distinct handles are independent.
 *
 * Data layout (the "pool"): a page is PA_PAGE_TOKENS consecutive token rows;
 * a row is [K of kv heads 0..Hkv-1 | V of kv heads 0..Hkv-1], head_dim bf16
 * values per head, so row_bytes = 4 * Hkv * head_dim (4,096 at Hkv = 4,
 * head_dim = 256, as in [GMM-host]).  Token j of a request lives in row
 * j % PA_PAGE_TOKENS of physical page page_table[request][j / PA_PAGE_TOKENS].
 * Query head h attends with kv head h / (Hq / Hkv).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_PAGE_TOKENS 64

#define PA_OK                0
#define PA_ERR_INVALID      -1  /* bad argument (null, size, range, alignment) */
#define PA_ERR_CUDA         -2  /* a CUDA call failed; arena calls then quarantine */
#define PA_ERR_QUARANTINED  -3  /* arena is quarantined after an earlier failure */
#define PA_ERR_ORDER        -4  /* slot busy or call out of order */
#define PA_ERR_OWNER        -5  /* write-back owner differs from the staged owner */
#define PA_ERR_UNSUPPORTED  -6  /* geometry not built into this library */
#define PA_ERR_REFUSED      -7  /* admission refused (the caller queues the request) */
#define PA_ERR_TIMEOUT      -8  /* a bounded host wait gave up */
#define PA_ERR_CRC          -9  /* a compact page does not match its published CRC */

/* Bits OR-ed into the int32 status word at byte 0 of the decode workspace
 * (and of the optional status word of kv_append_rows) by device code. */
#define PA_STATUS_BAD_PAGE   1  /* a page id outside [0, pool_pages): tile output is NaN */
#define PA_STATUS_TIMEOUT    2  /* a bounded device wait gave up: outputs are invalid */
#define PA_STATUS_BAD_ROW    4  /* kv_append_rows: position or page outside the table/pool */

/* Thread-local message for the last failing call on this thread ("" if none). */
const char* kv_last_error(void);

/* Pinned host memory for histories and compact stores ([GMM-host]): an
 * explicit-size cudaHostAlloc (page-locked, mapped into the device's address
 * space), owned by the caller until kv_host_free.  Copies from it ran at a
 * steady ~211 GB/s on GB300, against 150-200 GB/s from malloc'd memory pinned
 * afterwards with cudaHostRegister. */
int kv_host_alloc(size_t bytes, void** out);
int kv_host_free(void* p);

/* Library build string (compiler, target architecture). */
const char* pa_version(void);

/* ------------------------------------------------------------------------ */
/* Decode attention with per-tile LSE  ([KVE-exact], [KVE-bus])             */
/* ------------------------------------------------------------------------ */

/* Workspace bytes paged_decode_attn_lse, paged_decode_attn_lse_cuda_core and
 * paged_decode_attn_lse_append need for B requests x T tiles of this geometry
 * (an upper bound that does not depend on tile contents): status word, split
 * counters, per-(request, kv head) tile counters, partial slots.  Returns 0
 * for an unsupported geometry. */
size_t paged_decode_attn_lse_workspace_bytes(int B, int T, int n_q_heads,
                                             int n_kv_heads, int head_dim);

/* For every request b and tile t = [tiles[b][t][0], tiles[b][t][1]) of its
 * logical token history, and every query head h:
 *     s_j        = scale * <q[b][h], K_j of kv head h / G>,   j in the tile
 *     out[b][t][h] = sum_j exp(s_j - m) V_j / sum_j exp(s_j - m)   (FP32)
 *     lse[b][t][h] = m + ln sum_j exp(s_j - m)                      (FP32)
 * with m = max_j s_j.  An empty tile gives out 0 and lse -inf.
 *
 *   q          device bf16 [B][n_q_heads][head_dim], 16-byte aligned.
 *   pool       device bf16 pages (layout above), 16-byte aligned; its row
 *              stride 4*Hkv*head_dim bytes must be a multiple of 16.
 *   pool_pages number of pages addressable from pool; a page id outside
 *              [0, pool_pages) is never read: the tile's output becomes NaN and
 *              PA_STATUS_BAD_PAGE is set in the workspace status word.
 *   page_table device int32 [B][max_pages].
 *   tiles      HOST int32 [B][T][2]; 0 <= start <= end <= max_pages*64 is
 *              checked (PA_ERR_INVALID).  Tiles may overlap and need not be
 *              page aligned; rows outside a tile are masked, whatever they hold.
 *   out, lse   device fp32 [B][T][n_q_heads][head_dim] (16-byte aligned) and
 *              [B][T][n_q_heads].
 *   workspace  device buffer of at least the bytes the query above returns,
 *              256-byte aligned, ZERO-FILLED before its first use; every call
 *              leaves it ready for the next (counters return to their start
 *              state).  Byte 0 holds the int32 status word (PA_STATUS_* bits,
 *              sticky until the caller clears it); byte 4 an int32 diagnostic
 *              count of CTAs that stopped waiting for the other CTAs of a
 *              split unit (their share of its merge went to the unit's last
 *              CTA: same results, a slower launch; normally 0).  Calls that
 *              share a workspace must be ordered on one stream.
 * Supported: head_dim 256, n_q_heads / n_kv_heads in 1..8, n_kv_heads >= 1.
 * Results depend only on the logical tiles and the device's SM count, not on
 * physical page placement or timing: two calls that differ only in where the
 * pages sit return bit-identical outputs.  The CTAs of one launch wait for
 * each other only to share a split unit's merge, and a CTA that sees no other
 * CTA of the unit arrive for 50 us leaves its share to the last one, so
 * launches never depend on all CTAs being resident at once.
 * Tensor-core (mma.sync bf16) variant. */
int paged_decode_attn_lse(const void* q, const void* pool, int64_t pool_pages,
                          const int32_t* page_table, int max_pages,
                          const int32_t* tiles, int B, int T,
                          int n_q_heads, int n_kv_heads, int head_dim,
                          float scale, float* out, float* lse,
                          void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Same contract, evaluated with FP32 CUDA-core FMAs instead of tensor cores
 * (kept as the measured alternative). */
int paged_decode_attn_lse_cuda_core(const void* q, const void* pool, int64_t pool_pages,
                                    const int32_t* page_table, int max_pages,
                                    const int32_t* tiles, int B, int T,
                                    int n_q_heads, int n_kv_heads, int head_dim,
                                    float scale, float* out, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/* The same computation as paged_decode_attn_lse (tensor-core kernel), for
 * callers that cannot allocate device memory: there is no workspace argument.
 * The source pages have no counterpart to this entry point.
 *
 * Who needs it: code that fixes its device-memory budget before it starts
 * serving and forbids allocation afterwards, or that cannot pay for
 * cudaMalloc's possible device-wide synchronisation in its hot loop, and so
 * cannot hand this library a workspace.  The scratch instead lives in a fixed
 * array of PA_NOALLOC_SCRATCH_BYTES (16 MiB) among the library's device
 * globals, which every GPU that loads the library keeps until the process
 * exits.  Nothing here calls cudaMalloc, cudaFree or an allocating routine.
 *
 *   All arguments as for paged_decode_attn_lse, except:
 *   status  optional device int32; receives the call's PA_STATUS_* bits (the
 *           copy is enqueued on the stream after the kernel), or NULL.
 * Every argument is checked before the GPU is touched: a refused call
 * enqueues nothing and leaves the array as it was.  Returns PA_ERR_INVALID
 * when the call would need more scratch than the array holds (above ~1,000
 * (request, tile, kv head) units); paged_decode_attn_lse with a caller
 * workspace has no such limit.  The first call in each device's context
 * looks up the array's device address with that device current (and looks
 * it up again if the context is later destroyed and made anew, as after
 * cudaDeviceReset); make that first call before any stream capture.  Every
 * call clears the start of the array and reuses the rest, so calls whose
 * kernels may overlap on the GPU (unordered streams) race and must not be
 * issued. */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
int paged_decode_attn_lse_noalloc(const void* q, const void* pool, int64_t pool_pages,
                                  const int32_t* page_table, int max_pages,
                                  const int32_t* tiles, int B, int T,
                                  int n_q_heads, int n_kv_heads, int head_dim,
                                  float scale, float* out, float* lse,
                                  int32_t* status, cudaStream_t stream);

/* paged_decode_attn_lse and kv_append_rows in one launch ([KVE-exact],
 * [SWS-lease]): the step's new token of each request is written into its page
 * AND attended, so the pool does not have to hold the row before the call.
 *
 *   All arguments as for paged_decode_attn_lse, except:
 *   pool       writable: row new_rows[b] is stored at the pool row of token
 *              positions[b] of request b (page page_table[b][positions[b]/64],
 *              row positions[b] % 64), as kv_append_rows stores it.
 *   positions  device int32 [B].
 *   new_rows   device bf16 [B][2*n_kv_heads*head_dim] (K heads, then V
 *              heads), 16-byte aligned.
 * Every tile that covers positions[b] uses new_rows[b] for that token, whatever
 * the pool held there, so outputs are bit-identical to kv_append_rows followed
 * by paged_decode_attn_lse on the same stream.  An out-of-range position or
 * page id skips the store and ORs PA_STATUS_BAD_ROW into the workspace status
 * word.  No other call may read or write that pool row while this one runs.
 *   merged_out, merged_lse  optional (both NULL or both set): device fp32
 *              [B][n_q_heads][head_dim] (16-byte aligned) and [B][n_q_heads]
 *              receive the FP32 LSE merge of every request's T tiles, computed
 *              in the same launch by the CTA that finishes a (request, kv head)
 *              last, bit-identical to lse_merge over out / lse with
 *              part_offsets b * T.  With NULL, no merge is done.
 *   flags      0 or PA_DECODE_KV_READY.  The kernels of this library start
 *              under programmatic dependent launch: without the flag a launch
 *              reads nothing in memory until the kernels before it in the
 *              stream are complete.  PA_DECODE_KV_READY promises that the
 *              page table and the pool rows this call reads are written by no
 *              kernel that can still be running when this call's kernel
 *              starts (the kernel just before it in the stream, or one chained
 *              to that kernel by programmatic dependent launch); each CTA may
 *              then load its first pages while those kernels finish.  Results
 *              are the same with or without it when the promise holds. */
#define PA_DECODE_KV_READY 1u
int paged_decode_attn_lse_append(const void* q, void* pool, int64_t pool_pages,
                                 const int32_t* page_table, int max_pages,
                                 const int32_t* tiles, int B, int T,
                                 int n_q_heads, int n_kv_heads, int head_dim,
                                 float scale, const int32_t* positions,
                                 const void* new_rows, float* out, float* lse,
                                 float* merged_out, float* merged_lse,
                                 void* workspace, size_t workspace_bytes,
                                 unsigned flags, cudaStream_t stream);

/* Test hook for failure detection (no counterpart in the source pages): the
 * next decode call made on this thread (any paged_decode_attn_lse* entry
 * point) gives every bounded device wait up after wait_limit_ns (instead of
 * 2 s), and CTA 0 leaves its page load number `iteration` unarmed, so the
 * wait for that page runs out: the kernel sets PA_STATUS_TIMEOUT, lets the
 * loads it issued land and returns; the context stays usable.  Outputs of
 * that call are invalid and its workspace must be zero-filled again before
 * reuse.  (-1, 0) clears a pending setting.  PA_ERR_INVALID otherwise unless
 * iteration >= 0 and 0 < wait_limit_ns <= 2 s.  Nothing else calls it;
 * production calls never stall. */
int paged_decode_attn_test_stall(int iteration, uint64_t wait_limit_ns);

/* Test hook for the split-unit merge (no counterpart in the source pages):
 * the next decode call made on this thread waits at most slice_wait_ns
 * (instead of 50 us) without seeing another CTA of a split unit arrive
 * before it leaves its merge slice to the unit's last CTA, so a test can
 * drive the path that a grid not resident all at once takes; results are the
 * same bits either way.  -1 clears a pending setting; PA_ERR_INVALID outside
 * [-1, 50 us].  Production calls never use it. */
int paged_decode_attn_test_slice_wait(int64_t slice_wait_ns);

/* ------------------------------------------------------------------------ */
/* FP32 LSE merge  ([KVE-exact])                                            */
/* ------------------------------------------------------------------------ */

/* For every request b, head h over its partials i in [part_offsets[b],
 * part_offsets[b+1]), in increasing i:
 *     M = max_i lse_i;  w_i = exp(lse_i - M);
 *     out = sum_i w_i out_i / sum_i w_i;  lse = M + ln sum_i w_i.
 * No partials, or all lse_i = -inf: out 0, lse -inf.  A NaN lse_i gives NaN.
 * A single partial is returned bit for bit.
 *   out_parts    device fp32 [n_parts][H][D];  lse_parts device fp32 [n_parts][H]
 *   part_offsets device int32 [B+1], non-decreasing, part_offsets[0] = 0.
 *   out, lse     device fp32 [B][H][D], [B][H].
 * D must be a positive multiple of 4 and the fp32 arrays 16-byte aligned.
 * Every pointer must be non-NULL whenever B * H > 0 (PA_ERR_INVALID
 * otherwise), out_parts and lse_parts included: the offsets are on the
 * device, so the call cannot know that no partial will be read. */
int lse_merge(const float* out_parts, const float* lse_parts,
              const int32_t* part_offsets, int B, int H, int D,
              float* out, float* lse, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Device tail write: the new token's row into its page  ([SWS-lease])      */
/* ------------------------------------------------------------------------ */

/* For b < B: copy rows[b] (row_bytes bytes) to the pool row of token
 * positions[b] of request b, i.e. page page_table[b][positions[b] / 64],
 * row positions[b] % 64.  An out-of-range position or page id skips the row
 * and ORs PA_STATUS_BAD_ROW into *status (if status is not NULL).
 *   pool device; rows device [B][row_bytes]; positions device int32 [B];
 *   row_bytes a multiple of 16; status device int32 or NULL. */
int kv_append_rows(void* pool, int64_t pool_pages, const int32_t* page_table,
                   int max_pages, const int32_t* positions, const void* rows,
                   int B, int row_bytes, int32_t* status, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Staging arena  ([KVE-bus], [KVE-lease], [SWS-queues], [SWS-lease])       */
/* ------------------------------------------------------------------------ */

typedef struct kv_arena kv_arena;

#define PA_ARENA_RECORD_ONLY 1u  /* flags: log every CUDA submission instead of
                                    making it (host-side tests; no GPU needed) */

typedef struct {
    void*        device_base;     /* caller-owned device memory (256-B aligned)   */
    uint64_t     device_bytes;    /* explicit size, never inferred  ([SWS-admit]) */
    int          row_bytes;       /* bytes per token row                           */
    int          page_tokens;     /* must equal PA_PAGE_TOKENS                     */
    int          n_slots;         /* staging slots (>= 1; 2 lets copy overlap)     */
    int64_t      slot_first_page; /* page id, relative to device_base, of slot 0   */
    int64_t      slot_pages;      /* pages per slot; slot s starts at
                                     slot_first_page + s * slot_pages              */
    int32_t*     page_tables;     /* device int32 [n_slots][max_requests][max_pages],
                                     caller-owned; one table per slot              */
    int          max_requests;
    int          max_pages;
    cudaStream_t compute_stream;  /* attention runs here                           */
    cudaStream_t h2d_stream;      /* history copies                                */
    cudaStream_t d2h_stream;      /* tail write-back                               */
    uint32_t     flags;           /* PA_ARENA_* */
    /* Compact runs ([KVE-exact] "runs of two representations"; optional): a
     * staged compact page lands in the slot's landing area and is expanded on
     * the compute stream into a full bf16 page of the slot.  0 / 0 / 0: refused. */
    int32_t      compact_head_dim;  /* head_dim of the compact format            */
    uint64_t     landing_offset;    /* bytes from device_base to slot 0's landing
                                       area (256-B aligned, after every page)    */
    uint64_t     landing_bytes;     /* landing bytes per slot; slot s's area
                                       starts s * landing_bytes later            */
} kv_arena_desc;

/* A run of consecutive logical pages of one request.  host_rows != NULL: a
 * staged run, n_rows rows (<= n_pages * page_tokens) are copied from pinned
 * host memory into the slot.  host_rows == NULL: a resident run whose pages
 * already sit in the arena at resident_page, resident_page + 1, ... (outside
 * the staging slots; a run overlapping them is refused). */
typedef struct {
    int32_t     logical_page;
    int32_t     n_pages;
    int64_t     n_rows;
    const void* host_rows;      /* exact run: pinned host rows, n_rows of them  */
    int64_t     resident_page;  /* resident run (host_rows and host_compact NULL) */
    const void* host_compact;   /* compact run: pinned host compact pages (n_pages
                                   of kv_compact_page_bytes each, consecutive);
                                   n_rows must be n_pages * 64 (fully written)   */
} kv_page_run;

typedef struct {
    int32_t            request;  /* row of the slot's page table               */
    int32_t            n_runs;
    const kv_page_run* runs;
    uint64_t           owner;    /* host owner id the write-back must present  */
} kv_stage_req;

typedef struct {
    int32_t  request;   /* request as staged                                   */
    int32_t  pad_;
    int64_t  position;  /* token row to write back (its page must be staged or
                           resident in the layer's stage)                       */
    void*    host_row;  /* pinned host destination of row_bytes bytes           */
    uint64_t owner;     /* must equal the owner given to kv_stage_layer (else
                           PA_ERR_OWNER)                                        */
} kv_tail_req;

typedef struct {
    uint64_t stage_generation;  /* stages begun so far; strictly increasing     */
    uint64_t staged_bytes;      /* bytes enqueued host->device by stages/leases  */
    uint64_t written_back_bytes;/* bytes enqueued device->host                   */
    uint64_t slot_reuses;       /* stages that had to wait on a slot's readers   */
    int32_t  quarantined;       /* 1 after any failure                           */
    int32_t  n_slots;
    uint64_t loaded_bytes;      /* bytes enqueued host->device by kv_load_resident
                                   (not in staged_bytes)                         */
} kv_arena_stats;

/* Create an arena over caller memory.  Creates one copy, attention and
 * write-back event per slot.  Fails with PA_ERR_INVALID if the slots do not
 * fit in device_bytes. */
int kv_arena_create(const kv_arena_desc* desc, kv_arena** out);

/* Release the arena's events and bookkeeping.  Never waits, submits or drains
 * ([SWS-lease]); call kv_arena_drain first if work may still be in flight. */
int kv_arena_destroy(kv_arena* arena);

/* The one host-synchronising call: waits for the H2D, D2H and compute streams.
 * Returns PA_ERR_CUDA if completion cannot be established (the arena then stays
 * quarantined and keeps every buffer). */
int kv_arena_drain(kv_arena* arena);

/* Stage one layer: picks the next slot (round robin), makes the H2D stream
 * wait on that slot's previous attention and write-back events, enqueues one
 * H2D copy per staged run, writes the slot's page-table rows for every run
 * (staged runs, exact or compact, get consecutive slot pages in request/run
 * order), records the slot's copy event and makes the compute stream wait on
 * it.  A compact run is copied into the slot's landing area and expanded, on
 * the compute stream after that wait (so the H2D stream moves on to the next
 * layer), into bf16 pages holding bf16_rne(c * s) (the values the compact
 * page stands for); an attention enqueued next on the compute stream reads it
 * like any page.  PA_ERR_ORDER if the slot's previous stage was never
 * marked attention-done.
 *   *slot_out        the slot used; *page_table_out its device page table
 *                    ([max_requests][max_pages]) to pass to the attention. */
int kv_stage_layer(kv_arena* arena, int layer, const kv_stage_req* reqs,
                   int n_reqs, int* slot_out, const int32_t** page_table_out);

/* Record the layer's attention-done event on the compute stream; call after
 * the last kernel that reads the layer's slot. */
int kv_mark_attention_done(kv_arena* arena, int layer);

/* Tail write-back: the D2H stream waits on the layer's attention event, then
 * copies each requested row (row_bytes) from the arena to its pinned host row,
 * and records the slot's write-back event.  Refuses (PA_ERR_OWNER, nothing
 * enqueued) an owner other than the one the layer was staged with. */
int kv_writeback_tail(kv_arena* arena, int layer, const kv_tail_req* reqs,
                      int n_reqs);

/* One page (or its leading rows) copied into the arena's resident region. */
typedef struct {
    int64_t     resident_page;  /* arena page (relative to device_base) outside
                                   the staging slots                            */
    int32_t     n_rows;         /* rows copied into the page from its row 0,
                                   1..page_tokens                               */
    int32_t     pad_;
    const void* host_rows;      /* pinned host source: n_rows consecutive rows  */
} kv_resident_load;

/* Copy-in of resident pages ([SWS-admit]; "GPU memory management", section
 * "Pages held by right, borrowed or free": a page that turns hot is copied
 * into the device pool once and then served from there): the initial fill of
 * a static window, or the pages the admission planner made hot.  On the
 * device, in this order: the H2D stream waits on the most recent attention
 * and write-back events of this arena (their streams run in order, so every
 * earlier attention and write-back that may read the pages being replaced is
 * then done), one cudaMemcpyAsync per load, the arena's load event, and the
 * compute stream's wait on it (attention enqueued after this call sees the
 * pages; a later stage's copies follow them on the H2D stream).  The caller
 * marks attention done (kv_mark_attention_done / kv_lease_attention_done)
 * after every kernel that reads resident pages, as for staged ones: a load
 * waits only on attention already marked done, so every kernel that read the
 * pages being replaced must be marked before the load is made.  Refused
 * before anything is enqueued (PA_ERR_INVALID): a page inside the staging
 * slots or outside the arena, n_rows outside 1..page_tokens, host rows not in
 * pinned host memory.  A failed submission quarantines the arena.  Works with
 * stage calls and with leases. */
int kv_load_resident(kv_arena* arena, const kv_resident_load* loads, int n_loads);

/* ------------------------------------------------------------------------ */
/* Leases  ([SWS-lease], [KVE-lease], "GPU memory management" / "Staging as   */
/* a lease")                                                                */
/* ------------------------------------------------------------------------ */
/* Every staged layer is a transaction.  A lease is begun (the layer's pages
 * are copied into a slot), given its attention event after the attention
 * kernels, optionally given its tail write-back, sealed with exactly those two
 * events, and retired: the host waits for its copy, attention and write-back
 * events, receives a receipt, and the lease's copy tickets are released.
 * Rules enforced (PA_ERR_ORDER otherwise, nothing submitted):
 *   - a lease may begin only when the previously begun lease is sealed or
 *     retired;
 *   - a slot whose previous lease is sealed but not retired is refilled only
 *     after that lease's attention and write-back events (device-side waits,
 *     listed as the new lease's prior readers);
 *   - seal must present the attention token and the write-back token (0 if
 *     none was issued) returned for this lease: a substituted event is an
 *     error;
 *   - retire requires a sealed lease;
 *   - the host pages of an owner cannot be recycled (their generation
 *     advanced) while a live lease holds a copy ticket on them.
 * The stage generation of each lease is strictly increasing.  An arena is
 * driven either by these calls or by the stage calls above, not both. */

typedef struct {
    uint64_t       lease_id;    /* the lease's stage generation                 */
    int32_t        slot;
    int32_t        pad_;
    const int32_t* page_table;  /* device [max_requests][max_pages] of the slot */
} kv_lease;

typedef struct {
    uint64_t lease_id;
    int32_t  layer;
    int32_t  n_requests;
    int64_t  step;
    uint64_t staged_bytes;        /* bytes the lease copied host->device        */
    uint64_t written_back_bytes;  /* bytes its tail write-back copied back      */
    int32_t  tickets_released;    /* copy tickets (host owners) released        */
    int32_t  pad_;
} kv_receipt;

/* Begin a lease for `layer` at decode `step`: validates and stages `reqs`
 * like kv_stage_layer (each request's owner identifies the host pages it
 * copies from; a copy ticket records that owner's current generation). */
int kv_lease_begin(kv_arena* arena, int layer, int64_t step, const kv_stage_req* reqs,
                   int n_reqs, kv_lease* out);

/* Record the lease's attention (consumer) event on the compute stream, after
 * the last kernel that reads its slot; returns the event's token. */
int kv_lease_attention_done(kv_arena* arena, uint64_t lease_id, uint64_t* token);

/* Tail write-back as kv_writeback_tail (owner-checked, after the attention
 * event, on the D2H stream); returns the write-back event's token. */
int kv_lease_writeback(kv_arena* arena, uint64_t lease_id, const kv_tail_req* reqs,
                       int n_reqs, uint64_t* token);

/* Seal with the lease's own attention token and current write-back token. */
int kv_lease_seal(kv_arena* arena, uint64_t lease_id, uint64_t attention_token,
                  uint64_t writeback_token);

/* Host waits on the lease's copy, attention and write-back events, then the
 * receipt; a failing wait quarantines the arena and keeps the lease. */
int kv_lease_retire(kv_arena* arena, uint64_t lease_id, kv_receipt* receipt);

/* Current generation of an owner's host pages and the live copy tickets on it. */
int kv_host_generation(kv_arena* arena, uint64_t owner, uint64_t* generation,
                       int64_t* live_tickets);

/* Advance an owner's host-page generation (its pages may be reused for other
 * data); refused while any live lease holds a copy ticket on them, and while
 * the arena is quarantined. */
int kv_host_recycle(kv_arena* arena, uint64_t owner, uint64_t* new_generation);

/* Counters of the arena. */
int kv_arena_get_stats(const kv_arena* arena, kv_arena_stats* out);

/* Host-side test hooks.  kv_arena_fail_after: the n-th CUDA submission from
 * now (0 = the next) reports failure without being made, as a failing driver
 * call would; the arena then quarantines.  kv_arena_call_log: copies the
 * record of submissions made under PA_ARENA_RECORD_ONLY (one per line) into
 * buf, returns the full length. */
int kv_arena_fail_after(kv_arena* arena, int64_t n);
size_t kv_arena_call_log(const kv_arena* arena, char* buf, size_t buf_bytes);

/* ------------------------------------------------------------------------ */
/* Admission planner  ("Staging without a stall" / "Admission that does      */
/* arithmetic"; "GPU memory management" / "Pages held by right, borrowed or  */
/* free", "A host pool that explains its own size")                         */
/* ------------------------------------------------------------------------ */
/* Host-side bookkeeping of which logical pages of each context sit in the
 * device page pool.  A pool page holds one page_tokens-token logical page of
 * one context for all n_layers layers.  Each step, per listed context, the
 * planner wants the sink pages plus the newest pages up to target + burst,
 * and fills each missing page (sink first, then newest to oldest) by:
 *   1. reusing one of the context's own pool pages that left its window,
 *   2. taking a free pool page,
 *   3. reclaiming, only while the context holds fewer than its target:
 *      borrowed (burst) pages of other contexts, then other pages above a
 *      target, then whole idle contexts (not listed this step), each least
 *      recently active first,
 *   4. else the rest of the window (its older pages) stays cold.
 * Pages taken beyond the target are borrowed.  A context that ends the step
 * with fewer than its floor (sink pages + 1, capped by its length) is
 * refused for the step.  Every decision is counted; pages that became
 * resident are reported as copied in (once).  Changes happen only inside
 * kv_planner_step. */

typedef struct kv_planner kv_planner;

typedef struct {
    uint32_t pool_gib;           /* explicit whole GiB of device pool; 0 refused   */
    int32_t  n_layers;           /* dense layers sharing the pool                  */
    int32_t  row_bytes;          /* bytes per token per layer (4,096 here)         */
    int32_t  page_tokens;        /* tokens per page (PA_PAGE_TOKENS)               */
    int32_t  sink_pages;         /* attention-sink pages kept hot (1)              */
    int32_t  max_contexts;       /* configured concurrency limit                   */
    uint64_t host_pool_bytes;    /* pinned host pool owning the histories          */
    int64_t  max_context_tokens; /* context length each history must hold          */
    int32_t  shrink_mode;        /* 0: refuse a host pool that does not fit;
                                    1: lower the concurrency to what fits          */
    int32_t  pad_;
} kv_planner_desc;

typedef struct {
    uint64_t steps;
    uint64_t reused_own;             /* pages refilled from the context's own spare */
    uint64_t took_free;              /* pages taken from the free list              */
    uint64_t reclaimed_borrowed;     /* borrowed pages taken from other contexts    */
    uint64_t reclaimed_above_target; /* other above-target pages taken              */
    uint64_t reclaimed_idle_contexts;/* idle contexts emptied                       */
    uint64_t reclaimed_idle_pages;   /* pages freed by emptying idle contexts       */
    uint64_t shrunk_pages;           /* wanted pages left cold                      */
    uint64_t refused;                /* context-steps refused (below the floor)     */
    uint64_t copied_in;              /* pages that turned hot (one copy each)       */
    int64_t  free_pages;             /* free pool pages now                         */
} kv_planner_counters;

/* Create a planner.  The concurrency is min(max_contexts, floor(host_pool_bytes
 * / (n_layers x max_context_tokens x row_bytes))); the formula (and the pool
 * size in pages) is written to `formula`.  Refuse mode: PA_ERR_INVALID naming
 * the settings to change when the host pool holds fewer than max_contexts
 * histories; shrink mode lowers the concurrency instead. */
int kv_planner_create(const kv_planner_desc* desc, kv_planner** out, char* formula,
                      size_t formula_bytes);
int kv_planner_destroy(kv_planner* planner);
int kv_planner_info(const kv_planner* planner, int64_t* pool_pages, int* concurrency,
                    char* formula, size_t formula_bytes);

/* Admit a context (PA_ERR_REFUSED at the concurrency limit: queue it). */
int kv_planner_admit(kv_planner* planner, uint64_t ctx, int target_pages, int burst_pages);
int kv_planner_set_target(kv_planner* planner, uint64_t ctx, int target_pages,
                          int burst_pages);
/* Free every pool page of a finished context. */
int kv_planner_release(kv_planner* planner, uint64_t ctx);

/* One step boundary: the contexts running this step with their lengths
 * (tokens, including the new one).  admitted[i] (optional) = 1 if context i
 * reached its floor, 0 if refused for this step. */
int kv_planner_step(kv_planner* planner, const uint64_t* ctx_ids, const int64_t* lengths,
                    int n, int32_t* admitted);

/* The context's resident pages after the last step, by increasing logical
 * page: logical[k] lives in pool page pool[k].  *n_out = count (may exceed
 * cap; only cap entries are written). */
int kv_planner_resident(const kv_planner* planner, uint64_t ctx, int32_t* logical,
                        int32_t* pool, int cap, int* n_out);
/* Logical pages that became resident at the last step (to copy in once). */
int kv_planner_copied(const kv_planner* planner, uint64_t ctx, int32_t* logical, int cap,
                      int* n_out);
int kv_planner_get_counters(const kv_planner* planner, kv_planner_counters* out);

/* ------------------------------------------------------------------------ */
/* Compact older pages  ([KVE-exact], [KVE-tier])                           */
/* ------------------------------------------------------------------------ */

/* A history page that is fully written in every layer gets a second, smaller
 * representation, converted by background threads, checked by a CRC and
 * published; until it is published the page is served exact.  The source
 * pages name no format; this library's reading, per layer and page:
 *   - per token row and per (K or V, kv head) slice x of head_dim bf16 values:
 *     s = max|x| / 127 (binary32), codes c = clamp(round_half_even(x / s),
 *     -127, 127) as int8 (x / s a binary32 division; s = 0 gives zero codes);
 *     a page holding a non-finite value is not convertible and stays exact;
 *   - the page's bytes: codes int8 [64][2*Hkv*D], then scales float32
 *     little-endian [64][2*Hkv] (133,120 bytes at 4 x 256 instead of 262,144);
 *   - it stands for the values bf16_rne(binary32(c) * s);
 *   - its CRC is CRC-32 (reflected polynomial 0xEDB88320, initial value and
 *     final xor 0xFFFFFFFF) of those bytes. */
#define PA_COMPACT_CODE_MAX 127

/* Bytes of one layer's compact page; 0 for an unsupported geometry
 * (n_kv_heads >= 1 and head_dim a positive multiple of 16 are supported). */
size_t kv_compact_page_bytes(int n_kv_heads, int head_dim);

/* CRC-32 as above of `bytes` bytes, continuing `crc` (0 to start). */
uint32_t kv_crc32(const void* data, size_t bytes, uint32_t crc);

/* Convert one layer's page synchronously.  rows: host bf16 [64][2*Hkv*D];
 * out: host buffer of kv_compact_page_bytes bytes; crc (optional) receives
 * its CRC.  PA_ERR_INVALID if a value is not finite (out then unspecified). */
int kv_compact_convert_page(const void* rows, int n_kv_heads, int head_dim,
                            void* out, uint32_t* crc);

typedef struct kv_compactor kv_compactor;

typedef struct {
    int32_t n_layers;
    int32_t n_requests;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t max_pages;        /* logical pages per request                      */
    int32_t n_threads;        /* background converter threads, 1..256           */
    const void* const* exact_rows;   /* [n_layers * n_requests]: host address of
                                        token 0 of (layer l, request r) at index
                                        l * n_requests + r; rows are contiguous
                                        in token order, 4*Hkv*D bytes each      */
    void* const* compact_pages;      /* [n_layers * n_requests]: host address of
                                        compact page 0 of (l, r); page p starts
                                        p * kv_compact_page_bytes later          */
} kv_compactor_desc;

/* Page states. */
#define PA_PAGE_EXACT            0  /* not known to be fully written: exact     */
#define PA_PAGE_QUEUED           1  /* fully written, waiting for a converter   */
#define PA_PAGE_PUBLISHED        2  /* compact form and CRCs of every layer ready */
#define PA_PAGE_NOT_CONVERTIBLE  3  /* a non-finite value: stays exact          */

typedef struct {
    uint64_t published_pages;
    uint64_t not_convertible_pages;
    uint64_t compact_bytes;    /* bytes of compact pages written, all layers   */
    uint64_t queued_pages;     /* queued or being converted                    */
} kv_compactor_counters;

/* Start the converter threads.  All memory (exact history and compact store)
 * is the caller's and must outlive the compactor; the two address arrays are
 * copied. */
int kv_compactor_create(const kv_compactor_desc* desc, kv_compactor** out);

/* Stop the threads; a page being converted is finished first (the call waits
 * for it, milliseconds).  Queued pages are dropped. */
int kv_compactor_destroy(kv_compactor* c);

/* The caller states that pages [0, full_pages) of `request` are fully written
 * in every layer, in host memory (the write-backs that wrote them have
 * completed).  Pages not yet known are queued for conversion; the rest are
 * left as they are.  Never blocks on a conversion. */
int kv_compactor_mark_written(kv_compactor* c, int request, int full_pages);

/* hold != 0: converters start no new page (queued pages stay queued, served
 * exact); hold == 0: resume. */
int kv_compactor_hold(kv_compactor* c, int hold);

/* Wait until no page is queued or being converted.  PA_ERR_TIMEOUT after
 * timeout_ms; PA_ERR_ORDER if the converter is held with pages queued. */
int kv_compactor_wait_idle(kv_compactor* c, int timeout_ms);

/* States (PA_PAGE_*) of pages [first_page, first_page + n_pages) of a
 * request.  A page read as PA_PAGE_PUBLISHED has its compact bytes and CRCs
 * visible to this thread. */
int kv_compactor_states(const kv_compactor* c, int request, int first_page, int n_pages,
                        uint8_t* states);

/* The published CRC of (layer, request, page); PA_ERR_ORDER if unpublished. */
int kv_compactor_crc(const kv_compactor* c, int layer, int request, int page, uint32_t* crc);

/* Recompute every layer's CRC of a published page and compare with the
 * published ones: PA_OK or PA_ERR_CRC. */
int kv_compactor_verify(const kv_compactor* c, int request, int page);

int kv_compactor_get_counters(const kv_compactor* c, kv_compactor_counters* out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
