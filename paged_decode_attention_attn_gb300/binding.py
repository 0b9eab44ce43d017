"""ctypes binding of libpagedattn (argument marshalling only).

Every function here checks shapes, dtypes and devices of torch tensors, takes
their raw pointers and calls the C-ABI entry point of the same name; all work
runs in the library's CUDA kernels and copies.  If the shared library is
missing, importing this module raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedattn.so")

PA_OK = 0
PA_ERR_INVALID = -1
PA_ERR_CUDA = -2
PA_ERR_QUARANTINED = -3
PA_ERR_ORDER = -4
PA_ERR_OWNER = -5
PA_ERR_UNSUPPORTED = -6
PA_ERR_REFUSED = -7
PA_ERR_TIMEOUT = -8
PA_ERR_CRC = -9
PA_STATUS_BAD_PAGE = 1
PA_STATUS_TIMEOUT = 2
PA_STATUS_BAD_ROW = 4
PA_ARENA_RECORD_ONLY = 1
PA_PAGE_EXACT, PA_PAGE_QUEUED, PA_PAGE_PUBLISHED, PA_PAGE_NOT_CONVERTIBLE = 0, 1, 2, 3
PA_DECODE_KV_READY = 1
PAGE_TOKENS = 64

# Every symbol pagedattn.h declares.
EXPORTED = [
    "kv_last_error", "pa_version", "kv_host_alloc", "kv_host_free",
    "paged_decode_attn_lse_workspace_bytes", "paged_decode_attn_lse",
    "paged_decode_attn_lse_cuda_core", "paged_decode_attn_lse_noalloc",
    "paged_decode_attn_lse_append", "paged_decode_attn_test_stall",
    "paged_decode_attn_test_slice_wait", "lse_merge",
    "kv_append_rows",
    "kv_arena_create", "kv_arena_destroy", "kv_arena_drain", "kv_stage_layer",
    "kv_mark_attention_done", "kv_writeback_tail", "kv_load_resident", "kv_arena_get_stats",
    "kv_arena_fail_after", "kv_arena_call_log",
    "kv_lease_begin", "kv_lease_attention_done", "kv_lease_writeback", "kv_lease_seal",
    "kv_lease_retire", "kv_host_generation", "kv_host_recycle",
    "kv_planner_create", "kv_planner_destroy", "kv_planner_info", "kv_planner_admit",
    "kv_planner_set_target", "kv_planner_release", "kv_planner_step", "kv_planner_resident",
    "kv_planner_copied", "kv_planner_get_counters",
    "kv_compact_page_bytes", "kv_crc32", "kv_compact_convert_page", "kv_compactor_create",
    "kv_compactor_destroy", "kv_compactor_mark_written", "kv_compactor_hold",
    "kv_compactor_wait_idle", "kv_compactor_states", "kv_compactor_crc", "kv_compactor_verify",
    "kv_compactor_get_counters",
]


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class KvArenaDesc(ctypes.Structure):
    _fields_ = [
        ("device_base", ctypes.c_void_p),
        ("device_bytes", ctypes.c_uint64),
        ("row_bytes", ctypes.c_int),
        ("page_tokens", ctypes.c_int),
        ("n_slots", ctypes.c_int),
        ("slot_first_page", ctypes.c_int64),
        ("slot_pages", ctypes.c_int64),
        ("page_tables", ctypes.c_void_p),
        ("max_requests", ctypes.c_int),
        ("max_pages", ctypes.c_int),
        ("compute_stream", ctypes.c_void_p),
        ("h2d_stream", ctypes.c_void_p),
        ("d2h_stream", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("compact_head_dim", ctypes.c_int32),
        ("landing_offset", ctypes.c_uint64),
        ("landing_bytes", ctypes.c_uint64),
    ]


class KvPageRun(ctypes.Structure):
    _fields_ = [
        ("logical_page", ctypes.c_int32),
        ("n_pages", ctypes.c_int32),
        ("n_rows", ctypes.c_int64),
        ("host_rows", ctypes.c_void_p),
        ("resident_page", ctypes.c_int64),
        ("host_compact", ctypes.c_void_p),
    ]


class KvStageReq(ctypes.Structure):
    _fields_ = [
        ("request", ctypes.c_int32),
        ("n_runs", ctypes.c_int32),
        ("runs", ctypes.POINTER(KvPageRun)),
        ("owner", ctypes.c_uint64),
    ]


class KvTailReq(ctypes.Structure):
    _fields_ = [
        ("request", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("position", ctypes.c_int64),
        ("host_row", ctypes.c_void_p),
        ("owner", ctypes.c_uint64),
    ]


class KvResidentLoad(ctypes.Structure):
    _fields_ = [
        ("resident_page", ctypes.c_int64),
        ("n_rows", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("host_rows", ctypes.c_void_p),
    ]


class KvArenaStats(ctypes.Structure):
    _fields_ = [
        ("stage_generation", ctypes.c_uint64),
        ("staged_bytes", ctypes.c_uint64),
        ("written_back_bytes", ctypes.c_uint64),
        ("slot_reuses", ctypes.c_uint64),
        ("quarantined", ctypes.c_int32),
        ("n_slots", ctypes.c_int32),
        ("loaded_bytes", ctypes.c_uint64),
    ]


class KvLease(ctypes.Structure):
    _fields_ = [
        ("lease_id", ctypes.c_uint64),
        ("slot", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
    ]


class KvReceipt(ctypes.Structure):
    _fields_ = [
        ("lease_id", ctypes.c_uint64),
        ("layer", ctypes.c_int32),
        ("n_requests", ctypes.c_int32),
        ("step", ctypes.c_int64),
        ("staged_bytes", ctypes.c_uint64),
        ("written_back_bytes", ctypes.c_uint64),
        ("tickets_released", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
    ]


class KvCompactorDesc(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("n_requests", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_pages", ctypes.c_int32),
        ("n_threads", ctypes.c_int32),
        ("exact_rows", ctypes.POINTER(ctypes.c_void_p)),
        ("compact_pages", ctypes.POINTER(ctypes.c_void_p)),
    ]


class KvCompactorCounters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "published_pages", "not_convertible_pages", "compact_bytes", "queued_pages")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class KvPlannerDesc(ctypes.Structure):
    _fields_ = [
        ("pool_gib", ctypes.c_uint32),
        ("n_layers", ctypes.c_int32),
        ("row_bytes", ctypes.c_int32),
        ("page_tokens", ctypes.c_int32),
        ("sink_pages", ctypes.c_int32),
        ("max_contexts", ctypes.c_int32),
        ("host_pool_bytes", ctypes.c_uint64),
        ("max_context_tokens", ctypes.c_int64),
        ("shrink_mode", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
    ]


class KvPlannerCounters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "steps", "reused_own", "took_free", "reclaimed_borrowed", "reclaimed_above_target",
        "reclaimed_idle_contexts", "reclaimed_idle_pages", "shrunk_pages", "refused",
        "copied_in")] + [("free_pages", ctypes.c_int64)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m paged_decode_attention_attn_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.kv_last_error.restype = ctypes.c_char_p
    lib.kv_last_error.argtypes = []
    lib.pa_version.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.kv_host_alloc.restype = ctypes.c_int
    lib.kv_host_alloc.argtypes = [ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)]
    lib.kv_host_free.restype = ctypes.c_int
    lib.kv_host_free.argtypes = [ctypes.c_void_p]
    lib.paged_decode_attn_lse_workspace_bytes.restype = sz
    lib.paged_decode_attn_lse_workspace_bytes.argtypes = [i32] * 5
    dec = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, sz, vp]
    for name in ("paged_decode_attn_lse", "paged_decode_attn_lse_cuda_core"):
        getattr(lib, name).restype = i32
        getattr(lib, name).argtypes = dec
    lib.paged_decode_attn_lse_noalloc.restype = i32
    lib.paged_decode_attn_lse_noalloc.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, ctypes.c_float, vp, vp, vp, vp]
    lib.paged_decode_attn_lse_append.restype = i32
    lib.paged_decode_attn_lse_append.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, i32,
                                                 i32, ctypes.c_float, vp, vp, vp, vp, vp, vp,
                                                 vp, sz, ctypes.c_uint, vp]
    lib.paged_decode_attn_test_stall.restype = i32
    lib.paged_decode_attn_test_stall.argtypes = [i32, ctypes.c_uint64]
    lib.paged_decode_attn_test_slice_wait.restype = i32
    lib.paged_decode_attn_test_slice_wait.argtypes = [i64]
    lib.lse_merge.restype = i32
    lib.lse_merge.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
    lib.kv_append_rows.restype = i32
    lib.kv_append_rows.argtypes = [vp, i64, vp, i32, vp, vp, i32, i32, vp, vp]
    lib.kv_arena_create.restype = i32
    lib.kv_arena_create.argtypes = [ctypes.POINTER(KvArenaDesc), ctypes.POINTER(vp)]
    for name in ("kv_arena_destroy", "kv_arena_drain"):
        getattr(lib, name).restype = i32
        getattr(lib, name).argtypes = [vp]
    lib.kv_stage_layer.restype = i32
    lib.kv_stage_layer.argtypes = [vp, i32, ctypes.POINTER(KvStageReq), i32,
                                   ctypes.POINTER(i32), ctypes.POINTER(vp)]
    lib.kv_mark_attention_done.restype = i32
    lib.kv_mark_attention_done.argtypes = [vp, i32]
    lib.kv_writeback_tail.restype = i32
    lib.kv_writeback_tail.argtypes = [vp, i32, ctypes.POINTER(KvTailReq), i32]
    lib.kv_load_resident.restype = i32
    lib.kv_load_resident.argtypes = [vp, ctypes.POINTER(KvResidentLoad), i32]
    lib.kv_arena_get_stats.restype = i32
    lib.kv_arena_get_stats.argtypes = [vp, ctypes.POINTER(KvArenaStats)]
    lib.kv_arena_fail_after.restype = i32
    lib.kv_arena_fail_after.argtypes = [vp, i64]
    lib.kv_arena_call_log.restype = sz
    lib.kv_arena_call_log.argtypes = [vp, ctypes.c_char_p, sz]
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.kv_lease_begin.restype = i32
    lib.kv_lease_begin.argtypes = [vp, i32, i64, ctypes.POINTER(KvStageReq), i32,
                                   ctypes.POINTER(KvLease)]
    lib.kv_lease_attention_done.restype = i32
    lib.kv_lease_attention_done.argtypes = [vp, ctypes.c_uint64, u64p]
    lib.kv_lease_writeback.restype = i32
    lib.kv_lease_writeback.argtypes = [vp, ctypes.c_uint64, ctypes.POINTER(KvTailReq), i32, u64p]
    lib.kv_lease_seal.restype = i32
    lib.kv_lease_seal.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
    lib.kv_lease_retire.restype = i32
    lib.kv_lease_retire.argtypes = [vp, ctypes.c_uint64, ctypes.POINTER(KvReceipt)]
    lib.kv_host_generation.restype = i32
    lib.kv_host_generation.argtypes = [vp, ctypes.c_uint64, u64p, ctypes.POINTER(ctypes.c_int64)]
    lib.kv_host_recycle.restype = i32
    lib.kv_host_recycle.argtypes = [vp, ctypes.c_uint64, u64p]
    lib.kv_planner_create.restype = i32
    lib.kv_planner_create.argtypes = [ctypes.POINTER(KvPlannerDesc), ctypes.POINTER(vp),
                                      ctypes.c_char_p, sz]
    lib.kv_planner_destroy.restype = i32
    lib.kv_planner_destroy.argtypes = [vp]
    lib.kv_planner_info.restype = i32
    lib.kv_planner_info.argtypes = [vp, ctypes.POINTER(ctypes.c_int64),
                                    ctypes.POINTER(ctypes.c_int), ctypes.c_char_p, sz]
    lib.kv_planner_admit.restype = i32
    lib.kv_planner_admit.argtypes = [vp, ctypes.c_uint64, i32, i32]
    lib.kv_planner_set_target.restype = i32
    lib.kv_planner_set_target.argtypes = [vp, ctypes.c_uint64, i32, i32]
    lib.kv_planner_release.restype = i32
    lib.kv_planner_release.argtypes = [vp, ctypes.c_uint64]
    lib.kv_planner_step.restype = i32
    lib.kv_planner_step.argtypes = [vp, u64p, ctypes.POINTER(ctypes.c_int64), i32,
                                    ctypes.POINTER(ctypes.c_int32)]
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.kv_planner_resident.restype = i32
    lib.kv_planner_resident.argtypes = [vp, ctypes.c_uint64, i32p, i32p, i32,
                                        ctypes.POINTER(ctypes.c_int)]
    lib.kv_planner_copied.restype = i32
    lib.kv_planner_copied.argtypes = [vp, ctypes.c_uint64, i32p, i32, ctypes.POINTER(ctypes.c_int)]
    lib.kv_planner_get_counters.restype = i32
    lib.kv_planner_get_counters.argtypes = [vp, ctypes.POINTER(KvPlannerCounters)]
    u32 = ctypes.c_uint32
    lib.kv_compact_page_bytes.restype = sz
    lib.kv_compact_page_bytes.argtypes = [i32, i32]
    lib.kv_crc32.restype = u32
    lib.kv_crc32.argtypes = [vp, sz, u32]
    lib.kv_compact_convert_page.restype = i32
    lib.kv_compact_convert_page.argtypes = [vp, i32, i32, vp, ctypes.POINTER(u32)]
    lib.kv_compactor_create.restype = i32
    lib.kv_compactor_create.argtypes = [ctypes.POINTER(KvCompactorDesc), ctypes.POINTER(vp)]
    lib.kv_compactor_destroy.restype = i32
    lib.kv_compactor_destroy.argtypes = [vp]
    lib.kv_compactor_mark_written.restype = i32
    lib.kv_compactor_mark_written.argtypes = [vp, i32, i32]
    lib.kv_compactor_hold.restype = i32
    lib.kv_compactor_hold.argtypes = [vp, i32]
    lib.kv_compactor_wait_idle.restype = i32
    lib.kv_compactor_wait_idle.argtypes = [vp, i32]
    lib.kv_compactor_states.restype = i32
    lib.kv_compactor_states.argtypes = [vp, i32, i32, i32, ctypes.POINTER(ctypes.c_uint8)]
    lib.kv_compactor_crc.restype = i32
    lib.kv_compactor_crc.argtypes = [vp, i32, i32, i32, ctypes.POINTER(u32)]
    lib.kv_compactor_verify.restype = i32
    lib.kv_compactor_verify.argtypes = [vp, i32, i32]
    lib.kv_compactor_get_counters.restype = i32
    lib.kv_compactor_get_counters.argtypes = [vp, ctypes.POINTER(KvCompactorCounters)]
    return lib


lib = _load()


def last_error() -> str:
    return lib.kv_last_error().decode()


def _check(rc: int):
    if rc != PA_OK:
        raise PagedAttnError(rc, last_error())
    return rc


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str, contiguous: bool = True):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host_tiles(tiles) -> ctypes.Array:
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(tiles, dtype=np.int32))
    return arr, arr.ctypes.data


def workspace_bytes(B: int, T: int, n_q_heads: int, n_kv_heads: int, head_dim: int) -> int:
    return int(lib.paged_decode_attn_lse_workspace_bytes(B, T, n_q_heads, n_kv_heads, head_dim))


def alloc_workspace(B, T, n_q_heads, n_kv_heads, head_dim, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of the size the library asks for (256-B aligned)."""
    n = workspace_bytes(B, T, n_q_heads, n_kv_heads, head_dim)
    if n == 0:
        raise PagedAttnError(PA_ERR_UNSUPPORTED, "geometry not supported")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def paged_decode_attn_lse(q, pool, page_table, tiles, scale, out, lse, workspace,
                          stream=None, cuda_core=False, pool_pages=None):
    """q bf16 [B][Hq][D]; pool bf16 [pages][64][2*Hkv*D] (or any view whose
    storage starts at the first page); page_table int32 [B][max_pages];
    tiles host int32 [B][T][2]; out fp32 [B][T][Hq][D]; lse fp32 [B][T][Hq]."""
    B, Hq, D = q.shape
    row_elems = pool.shape[-1]
    n_kv = row_elems // (2 * D)
    arr, tiles_ptr = _host_tiles(tiles)
    T = arr.shape[1]
    if arr.shape[0] != B:
        raise ValueError("tiles must be [B][T][2]")
    if pool_pages is None:
        pool_pages = pool.numel() // (PAGE_TOKENS * row_elems)
    fn = lib.paged_decode_attn_lse_cuda_core if cuda_core else lib.paged_decode_attn_lse
    _check(fn(_dev(q, torch.bfloat16, "q"), _dev(pool, torch.bfloat16, "pool", False),
              int(pool_pages), _dev(page_table, torch.int32, "page_table"),
              int(page_table.shape[1]), tiles_ptr, B, T, Hq, n_kv, D, float(scale),
              _dev(out, torch.float32, "out"), _dev(lse, torch.float32, "lse"),
              _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
              _stream_handle(stream)))


def paged_decode_attn_lse_noalloc(q, pool, page_table, tiles, scale, out, lse, status=None,
                                  stream=None, pool_pages=None):
    """Same as paged_decode_attn_lse without a workspace argument: for callers
    that cannot allocate device memory, the library uses its own fixed device
    scratch array.  ``status`` (optional int32 CUDA tensor of 1 element)
    receives the call's status bits."""
    Bn, Hq, D = q.shape
    row_elems = pool.shape[-1]
    n_kv = row_elems // (2 * D)
    arr, tiles_ptr = _host_tiles(tiles)
    T = arr.shape[1]
    if arr.shape[0] != Bn:
        raise ValueError("tiles must be [B][T][2]")
    if pool_pages is None:
        pool_pages = pool.numel() // (PAGE_TOKENS * row_elems)
    _check(lib.paged_decode_attn_lse_noalloc(
        _dev(q, torch.bfloat16, "q"), _dev(pool, torch.bfloat16, "pool", False), int(pool_pages),
        _dev(page_table, torch.int32, "page_table"), int(page_table.shape[1]), tiles_ptr, Bn, T,
        Hq, n_kv, D, float(scale), _dev(out, torch.float32, "out"),
        _dev(lse, torch.float32, "lse"),
        None if status is None else _dev(status, torch.int32, "status"), _stream_handle(stream)))


def paged_decode_attn_lse_append(q, pool, page_table, tiles, scale, positions, new_rows, out,
                                 lse, workspace, stream=None, pool_pages=None, kv_ready=False,
                                 merged_out=None, merged_lse=None):
    """kv_append_rows and paged_decode_attn_lse in one launch: new_rows bf16
    [B][2*Hkv*D] are stored at token positions int32 [B] (device) of each
    request's pages and attended in place of whatever the pool held there.
    ``kv_ready`` passes PA_DECODE_KV_READY (see pagedattn.h for the promise);
    ``merged_out`` fp32 [B][Hq][D] / ``merged_lse`` [B][Hq] receive the
    merge of every request's tiles, computed in the same launch."""
    B, Hq, D = q.shape
    row_elems = pool.shape[-1]
    n_kv = row_elems // (2 * D)
    arr, tiles_ptr = _host_tiles(tiles)
    T = arr.shape[1]
    if arr.shape[0] != B:
        raise ValueError("tiles must be [B][T][2]")
    if tuple(new_rows.shape) != (B, row_elems) or tuple(positions.shape) != (B,):
        raise ValueError("new_rows must be [B][2*Hkv*D] and positions [B]")
    if pool_pages is None:
        pool_pages = pool.numel() // (PAGE_TOKENS * row_elems)
    _check(lib.paged_decode_attn_lse_append(
        _dev(q, torch.bfloat16, "q"), _dev(pool, torch.bfloat16, "pool", False), int(pool_pages),
        _dev(page_table, torch.int32, "page_table"), int(page_table.shape[1]), tiles_ptr, B, T,
        Hq, n_kv, D, float(scale), _dev(positions, torch.int32, "positions"),
        _dev(new_rows, torch.bfloat16, "new_rows"), _dev(out, torch.float32, "out"),
        _dev(lse, torch.float32, "lse"),
        None if merged_out is None else _dev(merged_out, torch.float32, "merged_out"),
        None if merged_lse is None else _dev(merged_lse, torch.float32, "merged_lse"),
        _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), PA_DECODE_KV_READY if kv_ready else 0, _stream_handle(stream)))


def test_stall(iteration: int, wait_limit_ns: int):
    """Failure-detection test hook: the next decode call on this thread stalls
    CTA 0 at page load ``iteration`` and gives waits up after wait_limit_ns."""
    _check(lib.paged_decode_attn_test_stall(int(iteration), int(wait_limit_ns)))


def test_slice_wait(slice_wait_ns: int):
    """Split-merge test hook: the next decode call on this thread waits at most
    slice_wait_ns for another arrival before a CTA leaves its merge slice to
    the unit's last CTA (-1 clears)."""
    _check(lib.paged_decode_attn_test_slice_wait(int(slice_wait_ns)))


def lse_merge(out_parts, lse_parts, part_offsets, out, lse, stream=None):
    """out_parts fp32 [P][H][D]; lse_parts fp32 [P][H]; part_offsets int32 [B+1]
    (device); out fp32 [B][H][D]; lse fp32 [B][H]."""
    B = part_offsets.shape[0] - 1
    H, D = out.shape[-2], out.shape[-1]
    _check(lib.lse_merge(_dev(out_parts, torch.float32, "out_parts"),
                         _dev(lse_parts, torch.float32, "lse_parts"),
                         _dev(part_offsets, torch.int32, "part_offsets"), B, H, D,
                         _dev(out, torch.float32, "out"), _dev(lse, torch.float32, "lse"),
                         _stream_handle(stream)))


def kv_append_rows(pool, page_table, positions, rows, status=None, stream=None,
                   pool_pages=None):
    """Write rows bf16 [B][row_elems] at token positions int32 [B] of each
    request's pages (device tail write before attention)."""
    B, row_elems = rows.shape
    if pool_pages is None:
        pool_pages = pool.numel() // (PAGE_TOKENS * row_elems)
    _check(lib.kv_append_rows(_dev(pool, torch.bfloat16, "pool", False), int(pool_pages),
                              _dev(page_table, torch.int32, "page_table"),
                              int(page_table.shape[1]), _dev(positions, torch.int32, "positions"),
                              _dev(rows, torch.bfloat16, "rows"), B, row_elems * 2,
                              None if status is None else _dev(status, torch.int32, "status"),
                              _stream_handle(stream)))


class Arena:
    """Owner of a kv_arena handle over caller-allocated device memory."""

    def __init__(self, device_base: int, device_bytes: int, row_bytes: int, n_slots: int,
                 slot_first_page: int, slot_pages: int, page_tables: int, max_requests: int,
                 max_pages: int, compute_stream=None, h2d_stream=None, d2h_stream=None,
                 record_only: bool = False, compact_head_dim: int = 0, landing_offset: int = 0,
                 landing_bytes: int = 0):
        d = KvArenaDesc()
        d.device_base = device_base
        d.device_bytes = device_bytes
        d.row_bytes = row_bytes
        d.page_tokens = PAGE_TOKENS
        d.n_slots = n_slots
        d.slot_first_page = slot_first_page
        d.slot_pages = slot_pages
        d.page_tables = page_tables
        d.max_requests = max_requests
        d.max_pages = max_pages
        d.compute_stream = self._h(compute_stream)
        d.h2d_stream = self._h(h2d_stream)
        d.d2h_stream = self._h(d2h_stream)
        d.flags = PA_ARENA_RECORD_ONLY if record_only else 0
        d.compact_head_dim = compact_head_dim
        d.landing_offset = landing_offset
        d.landing_bytes = landing_bytes
        self._desc = d
        h = ctypes.c_void_p()
        _check(lib.kv_arena_create(ctypes.byref(d), ctypes.byref(h)))
        self.handle = h
        self._keep = []

    @staticmethod
    def _h(s):
        if s is None:
            return None
        if isinstance(s, int):
            return s
        return int(s.cuda_stream)

    def stage_layer(self, layer: int, requests):
        """requests: list of (request, owner, [runs]); a run is a dict with
        logical_page, n_pages and either host_rows (address) + n_rows,
        host_compact (address of compact pages) + n_rows = n_pages * 64, or
        resident_page.  Returns (slot, page_table_address)."""
        reqs, keep = self._stage_reqs(requests)
        slot = ctypes.c_int(-1)
        table = ctypes.c_void_p()
        _check(lib.kv_stage_layer(self.handle, layer, reqs, len(requests), ctypes.byref(slot),
                                  ctypes.byref(table)))
        del keep
        return slot.value, table.value

    def mark_attention_done(self, layer: int):
        _check(lib.kv_mark_attention_done(self.handle, layer))

    def load_resident(self, loads):
        """loads: list of (resident_page, n_rows, host_rows_address)."""
        if not loads:
            return
        arr = (KvResidentLoad * len(loads))()
        for k, (page, n_rows, host) in enumerate(loads):
            arr[k].resident_page = page
            arr[k].n_rows = n_rows
            arr[k].host_rows = host
        _check(lib.kv_load_resident(self.handle, arr, len(loads)))

    def writeback_tail(self, layer: int, tails):
        """tails: list of (request, position, host_row_address, owner)."""
        _check(lib.kv_writeback_tail(self.handle, layer, self._tail_reqs(tails), len(tails)))

    @staticmethod
    def _stage_reqs(requests):
        reqs = (KvStageReq * max(1, len(requests)))()
        keep = []
        for i, (request, owner, runs) in enumerate(requests):
            arr = (KvPageRun * max(1, len(runs)))()
            for k, r in enumerate(runs):
                arr[k].logical_page = r["logical_page"]
                arr[k].n_pages = r["n_pages"]
                arr[k].n_rows = r.get("n_rows", 0)
                arr[k].host_rows = r.get("host_rows")
                arr[k].resident_page = r.get("resident_page", 0)
                arr[k].host_compact = r.get("host_compact")
            keep.append(arr)
            reqs[i].request = request
            reqs[i].n_runs = len(runs)
            reqs[i].runs = ctypes.cast(arr, ctypes.POINTER(KvPageRun))
            reqs[i].owner = owner
        return reqs, keep

    @staticmethod
    def _tail_reqs(tails):
        arr = (KvTailReq * max(1, len(tails)))()
        for i, (request, position, host_row, owner) in enumerate(tails):
            arr[i].request = request
            arr[i].position = position
            arr[i].host_row = host_row
            arr[i].owner = owner
        return arr

    # ---- leases ----
    def lease_begin(self, layer: int, step: int, requests) -> KvLease:
        reqs, keep = self._stage_reqs(requests)
        out = KvLease()
        _check(lib.kv_lease_begin(self.handle, layer, step, reqs, len(requests),
                                  ctypes.byref(out)))
        del keep
        return out

    def lease_attention_done(self, lease_id: int) -> int:
        tok = ctypes.c_uint64()
        _check(lib.kv_lease_attention_done(self.handle, lease_id, ctypes.byref(tok)))
        return tok.value

    def lease_writeback(self, lease_id: int, tails) -> int:
        tok = ctypes.c_uint64()
        _check(lib.kv_lease_writeback(self.handle, lease_id, self._tail_reqs(tails), len(tails),
                                      ctypes.byref(tok)))
        return tok.value

    def lease_seal(self, lease_id: int, attention_token: int, writeback_token: int = 0):
        _check(lib.kv_lease_seal(self.handle, lease_id, attention_token, writeback_token))

    def lease_retire(self, lease_id: int) -> KvReceipt:
        r = KvReceipt()
        _check(lib.kv_lease_retire(self.handle, lease_id, ctypes.byref(r)))
        return r

    def host_generation(self, owner: int):
        g = ctypes.c_uint64()
        n = ctypes.c_int64()
        _check(lib.kv_host_generation(self.handle, owner, ctypes.byref(g), ctypes.byref(n)))
        return g.value, n.value

    def host_recycle(self, owner: int) -> int:
        g = ctypes.c_uint64()
        _check(lib.kv_host_recycle(self.handle, owner, ctypes.byref(g)))
        return g.value

    def drain(self):
        _check(lib.kv_arena_drain(self.handle))

    def stats(self) -> KvArenaStats:
        s = KvArenaStats()
        _check(lib.kv_arena_get_stats(self.handle, ctypes.byref(s)))
        return s

    def fail_after(self, n: int):
        _check(lib.kv_arena_fail_after(self.handle, n))

    def call_log(self) -> list:
        n = lib.kv_arena_call_log(self.handle, None, 0)
        buf = ctypes.create_string_buffer(n + 1)
        lib.kv_arena_call_log(self.handle, buf, n + 1)
        return [line for line in buf.value.decode().split("\n") if line]

    def close(self):
        if self.handle:
            lib.kv_arena_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Planner:
    """Owner of a kv_planner handle (admission and device-window bookkeeping)."""

    def __init__(self, pool_gib: int, n_layers: int = 16, row_bytes: int = 4096,
                 page_tokens: int = PAGE_TOKENS, sink_pages: int = 1, max_contexts: int = 8,
                 host_pool_bytes: int = 1 << 40, max_context_tokens: int = 131072,
                 shrink_mode: bool = False):
        d = KvPlannerDesc()
        d.pool_gib = pool_gib
        d.n_layers = n_layers
        d.row_bytes = row_bytes
        d.page_tokens = page_tokens
        d.sink_pages = sink_pages
        d.max_contexts = max_contexts
        d.host_pool_bytes = host_pool_bytes
        d.max_context_tokens = max_context_tokens
        d.shrink_mode = 1 if shrink_mode else 0
        h = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(1024)
        self.handle = None
        _check(lib.kv_planner_create(ctypes.byref(d), ctypes.byref(h), buf, 1024))
        self.handle = h
        self.formula = buf.value.decode()

    def info(self):
        n = ctypes.c_int64()
        c = ctypes.c_int()
        _check(lib.kv_planner_info(self.handle, ctypes.byref(n), ctypes.byref(c), None, 0))
        return n.value, c.value

    def admit(self, ctx: int, target: int, burst: int = 0):
        _check(lib.kv_planner_admit(self.handle, ctx, target, burst))

    def set_target(self, ctx: int, target: int, burst: int = 0):
        _check(lib.kv_planner_set_target(self.handle, ctx, target, burst))

    def release(self, ctx: int):
        _check(lib.kv_planner_release(self.handle, ctx))

    def step(self, contexts) -> list:
        """contexts: list of (ctx, length_tokens).  Returns admitted flags."""
        n = len(contexts)
        ids = (ctypes.c_uint64 * max(1, n))(*[c for c, _ in contexts])
        lens = (ctypes.c_int64 * max(1, n))(*[L for _, L in contexts])
        adm = (ctypes.c_int32 * max(1, n))()
        _check(lib.kv_planner_step(self.handle, ids, lens, n, adm))
        return [bool(adm[i]) for i in range(n)]

    def resident(self, ctx: int) -> dict:
        n = ctypes.c_int()
        _check(lib.kv_planner_resident(self.handle, ctx, None, None, 0, ctypes.byref(n)))
        lg = (ctypes.c_int32 * max(1, n.value))()
        pl = (ctypes.c_int32 * max(1, n.value))()
        _check(lib.kv_planner_resident(self.handle, ctx, lg, pl, n.value, ctypes.byref(n)))
        return {lg[i]: pl[i] for i in range(n.value)}

    def copied(self, ctx: int) -> list:
        n = ctypes.c_int()
        _check(lib.kv_planner_copied(self.handle, ctx, None, 0, ctypes.byref(n)))
        lg = (ctypes.c_int32 * max(1, n.value))()
        _check(lib.kv_planner_copied(self.handle, ctx, lg, n.value, ctypes.byref(n)))
        return [lg[i] for i in range(n.value)]

    def counters(self) -> dict:
        c = KvPlannerCounters()
        _check(lib.kv_planner_get_counters(self.handle, ctypes.byref(c)))
        return c.as_dict()

    def close(self):
        if self.handle:
            lib.kv_planner_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------------------
# Compact older pages
# ---------------------------------------------------------------------------

def compact_page_bytes(n_kv_heads: int, head_dim: int) -> int:
    return int(lib.kv_compact_page_bytes(n_kv_heads, head_dim))


def crc32(data: bytes, crc: int = 0) -> int:
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    return int(lib.kv_crc32(buf, len(data), crc))


def compact_convert_page(rows, n_kv_heads: int, head_dim: int):
    """rows: host bf16 tensor [64][2*Hkv*D].  Returns (page bytes, crc)."""
    if rows.device.type != "cpu" or rows.dtype != torch.bfloat16 or not rows.is_contiguous():
        raise ValueError("rows must be a contiguous CPU bf16 tensor")
    n = compact_page_bytes(n_kv_heads, head_dim)
    out = ctypes.create_string_buffer(n)
    crc = ctypes.c_uint32()
    _check(lib.kv_compact_convert_page(rows.data_ptr(), n_kv_heads, head_dim, out,
                                       ctypes.byref(crc)))
    return out.raw, crc.value


class Compactor:
    """Background converter of fully written pages into their compact form.

    exact_rows / compact_pages: host addresses, index layer * n_requests +
    request (see kv_compactor_desc)."""

    def __init__(self, n_layers, n_requests, n_kv_heads, head_dim, max_pages, exact_rows,
                 compact_pages, n_threads=4):
        n = n_layers * n_requests
        if len(exact_rows) != n or len(compact_pages) != n:
            raise ValueError("one exact and one compact address per (layer, request)")
        self._exact = (ctypes.c_void_p * n)(*exact_rows)
        self._compact = (ctypes.c_void_p * n)(*compact_pages)
        d = KvCompactorDesc()
        d.n_layers, d.n_requests, d.n_kv_heads, d.head_dim = (n_layers, n_requests, n_kv_heads,
                                                              head_dim)
        d.max_pages, d.n_threads = max_pages, n_threads
        d.exact_rows = ctypes.cast(self._exact, ctypes.POINTER(ctypes.c_void_p))
        d.compact_pages = ctypes.cast(self._compact, ctypes.POINTER(ctypes.c_void_p))
        h = ctypes.c_void_p()
        _check(lib.kv_compactor_create(ctypes.byref(d), ctypes.byref(h)))
        self.handle = h
        self.max_pages = max_pages
        self.n_layers = n_layers

    def mark_written(self, request: int, full_pages: int):
        _check(lib.kv_compactor_mark_written(self.handle, request, full_pages))

    def hold(self, on: bool):
        _check(lib.kv_compactor_hold(self.handle, 1 if on else 0))

    def wait_idle(self, timeout_ms: int = 600000):
        _check(lib.kv_compactor_wait_idle(self.handle, timeout_ms))

    def states(self, request: int, first_page: int = 0, n_pages=None):
        n = self.max_pages - first_page if n_pages is None else n_pages
        arr = (ctypes.c_uint8 * max(1, n))()
        _check(lib.kv_compactor_states(self.handle, request, first_page, n, arr))
        return list(arr[:n])

    def crc(self, layer: int, request: int, page: int) -> int:
        c = ctypes.c_uint32()
        _check(lib.kv_compactor_crc(self.handle, layer, request, page, ctypes.byref(c)))
        return c.value

    def verify(self, request: int, page: int):
        _check(lib.kv_compactor_verify(self.handle, request, page))

    def counters(self) -> dict:
        c = KvCompactorCounters()
        _check(lib.kv_compactor_get_counters(self.handle, ctypes.byref(c)))
        return c.as_dict()

    def close(self):
        if getattr(self, "handle", None):
            lib.kv_compactor_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PinnedBuffer:
    """Pinned host memory from kv_host_alloc, viewed as a uint8 CPU tensor
    (``.tensor``); freed by close()."""

    def __init__(self, nbytes: int):
        import numpy as np
        ptr = ctypes.c_void_p()
        _check(lib.kv_host_alloc(int(nbytes), ctypes.byref(ptr)))
        self.ptr = ptr.value
        self.nbytes = int(nbytes)
        arr = np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.ptr))
        self.tensor = torch.from_numpy(arr)

    def close(self):
        if getattr(self, "ptr", None):
            self.tensor = None
            lib.kv_host_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
