"""C-ABI checks that need no GPU: every declared symbol is exported, and the
host-side argument checks refuse bad calls before anything reaches CUDA."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kv_arena_create", "kv_stage_layer", "paged_decode_attn_lse", "lse_merge",
                     "kv_writeback_tail", "kv_arena_destroy", "kv_arena_drain",
                     "kv_mark_attention_done", "kv_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(B):
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(B.lib, name), f"{name} declared in pagedattn.h but not exported"
    assert sorted(names) == sorted(B.EXPORTED)


def test_version_string(B):
    assert b"sm_103a" in B.lib.pa_version()


def test_workspace_query(B):
    n = B.workspace_bytes(4, 1, 24, 4, 256)
    assert n > 0 and n % 256 == 0
    assert B.workspace_bytes(4, 1, 24, 4, 128) == 0        # head_dim not built
    assert B.workspace_bytes(4, 1, 36, 4, 256) == 0        # group 9 > 8
    assert B.workspace_bytes(4, 1, 25, 4, 256) == 0        # not a multiple


def _call_decode(B, tiles, head_dim=256, nq=24, nkv=4, ws_bytes=1 << 30, ws_ptr=1 << 20,
                 pool_pages=16, max_pages=8):
    arr = np.ascontiguousarray(np.asarray(tiles, dtype=np.int32))
    Bn, T = arr.shape[0], arr.shape[1]
    fake = 1 << 20  # never dereferenced: the checks below fail before any CUDA call
    return B.lib.paged_decode_attn_lse(fake, fake, pool_pages, fake, max_pages, arr.ctypes.data,
                                       Bn, T, nq, nkv, head_dim, 0.0625, fake, fake, ws_ptr,
                                       ws_bytes, None)


def test_decode_argument_checks(B):
    ok_tiles = [[[0, 64]]]
    assert _call_decode(B, ok_tiles, head_dim=128) == B.PA_ERR_UNSUPPORTED
    assert _call_decode(B, ok_tiles, nq=25) == B.PA_ERR_INVALID
    assert _call_decode(B, ok_tiles, nq=72) == B.PA_ERR_UNSUPPORTED
    assert _call_decode(B, [[[0, 8 * 64 + 1]]]) == B.PA_ERR_INVALID     # past the table
    assert _call_decode(B, [[[10, 5]]]) == B.PA_ERR_INVALID             # start > end
    assert _call_decode(B, [[[-1, 5]]]) == B.PA_ERR_INVALID
    assert _call_decode(B, ok_tiles, ws_bytes=1024) == B.PA_ERR_INVALID  # workspace too small
    assert _call_decode(B, ok_tiles, ws_ptr=(1 << 20) + 16) == B.PA_ERR_INVALID  # misaligned
    assert "workspace" in B.last_error()
    # 2^25 pages = 2^31 rows: past the 32-bit row coordinates of the page loads
    assert _call_decode(B, ok_tiles, pool_pages=(1 << 25)) == B.PA_ERR_INVALID
    assert "pool too large" in B.last_error()
    assert _call_decode(B, ok_tiles, pool_pages=0) == B.PA_ERR_INVALID
    # zero requests is a no-op
    arr = np.zeros((0, 1, 2), dtype=np.int32)
    assert B.lib.paged_decode_attn_lse(0, 0, 0, 0, 0, arr.ctypes.data, 0, 1, 24, 4, 256, 1.0, 0,
                                       0, 0, 0, None) == B.PA_OK


def test_noalloc_refuses_before_touching_the_gpu(B):
    """The allocation-free decode entry point checks every argument before it
    looks up or clears its scratch array: on a machine without a GPU these
    calls fail with the argument's own error, not with a CUDA error."""
    fake = 1 << 20
    ok = np.ascontiguousarray(np.asarray([[[0, 64]]], dtype=np.int32))

    def call(q=fake, tiles=ok, nq=24, nkv=4, head_dim=256, out=fake, max_pages=8):
        return B.lib.paged_decode_attn_lse_noalloc(q, fake, 16, fake, max_pages,
                                                   tiles.ctypes.data, tiles.shape[0],
                                                   tiles.shape[1], nq, nkv, head_dim, 0.0625,
                                                   out, fake, None, None)
    assert call(head_dim=128) == B.PA_ERR_UNSUPPORTED
    assert call(nq=72) == B.PA_ERR_UNSUPPORTED
    assert call(nq=25) == B.PA_ERR_INVALID
    assert call(q=None) == B.PA_ERR_INVALID
    assert call(q=fake + 8) == B.PA_ERR_INVALID
    assert "q must be 16-byte aligned" in B.last_error()
    assert call(out=fake + 4) == B.PA_ERR_INVALID
    bad = np.ascontiguousarray(np.asarray([[[0, 9 * 64]]], dtype=np.int32))
    assert call(tiles=bad) == B.PA_ERR_INVALID                       # past the table
    assert "outside" in B.last_error()


def test_merge_and_append_argument_checks(B):
    fake = 1 << 20
    assert B.lib.lse_merge(fake, fake, fake, 2, 24, 254, fake, fake, None) == B.PA_ERR_INVALID
    assert B.lib.lse_merge(fake, fake, fake, 0, 24, 256, fake, fake, None) == B.PA_OK
    assert B.lib.lse_merge(fake, fake, fake, 2, 24, 0, fake, fake, None) == B.PA_ERR_INVALID
    # the partial arrays are required whenever there are rows to merge
    assert B.lib.lse_merge(None, fake, fake, 2, 24, 256, fake, fake, None) == B.PA_ERR_INVALID
    assert B.lib.lse_merge(fake, None, fake, 2, 24, 256, fake, fake, None) == B.PA_ERR_INVALID
    assert B.lib.kv_append_rows(fake, 4, fake, 4, fake, fake, 1, 4008, None, None) == \
        B.PA_ERR_INVALID
    assert B.lib.kv_append_rows(fake, 4, fake, 4, fake, fake + 8, 1, 4096, None, None) == \
        B.PA_ERR_INVALID


def test_fused_append_argument_checks(B):
    fake = 1 << 20
    arr = np.ascontiguousarray(np.asarray([[[0, 64]]], dtype=np.int32))

    def call(positions, rows, flags=0, merged=None):
        return B.lib.paged_decode_attn_lse_append(fake, fake, 16, fake, 8, arr.ctypes.data, 1, 1,
                                                  24, 4, 256, 0.0625, positions, rows, fake, fake,
                                                  merged, merged, fake, 1 << 30, flags, None)
    assert call(None, fake) == B.PA_ERR_INVALID
    assert call(fake, None) == B.PA_ERR_INVALID
    assert call(fake, fake + 8) == B.PA_ERR_INVALID
    assert "new_rows" in B.last_error()
    assert call(fake, fake, flags=2) == B.PA_ERR_INVALID
    assert "flags" in B.last_error()
    assert call(fake, fake, merged=fake + 4) == B.PA_ERR_INVALID
    assert "merged_out" in B.last_error()


def test_stall_hook_argument_checks(B):
    assert B.lib.paged_decode_attn_test_stall(-1, 1000) == B.PA_ERR_INVALID
    assert B.lib.paged_decode_attn_test_stall(0, 0) == B.PA_ERR_INVALID
    assert B.lib.paged_decode_attn_test_stall(0, 3_000_000_000) == B.PA_ERR_INVALID
    # a valid setting applies to the next call on this thread only; clear it
    assert B.lib.paged_decode_attn_test_stall(2, 50_000_000) == B.PA_OK
    assert B.lib.paged_decode_attn_test_stall(-1, 0) == B.PA_OK


def test_slice_wait_hook_argument_checks(B):
    assert B.lib.paged_decode_attn_test_slice_wait(-2) == B.PA_ERR_INVALID
    assert B.lib.paged_decode_attn_test_slice_wait(50_001) == B.PA_ERR_INVALID
    assert B.lib.paged_decode_attn_test_slice_wait(0) == B.PA_OK
    assert B.lib.paged_decode_attn_test_slice_wait(-1) == B.PA_OK
