"""One decode step of paged GQA attention over every layer, on three routes.

Resident route: the whole history sits in a device pool; per layer one
launch writes the new token's row into its page, returns per-tile (out, LSE)
with that row attended and merges every request's tiles in FP32
(``fused=False`` issues the tail write, the attention and the merge as three
launches).

Staged route ("Staging without a stall"; "KV-cache engineering", section
"Staging layers under a lease"): pinned host memory owns the history; per
layer the arena copies the layer's non-resident pages into a device slot on
the H2D stream, the compute stream waits on the copy's event, the same
kernels run against the slot, attention is marked done, and only the new
token's row is written back to its pinned host row on the D2H stream.

Planned route ("Staging without a stall", section "Admission that does
arithmetic"): the admission planner decides each step which pages stay hot in
a device pool; pages that turn hot are copied in once, the rest are staged.

On the staged and planned routes, pages the background converter has
published ("KV-cache engineering", section "Exact recent pages, compact older
pages") can be staged in their compact form (``CompactStore``).

The routes only sequence C-ABI calls; all data movement and arithmetic run in
libpagedattn's kernels, copies and threads.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .workloads import DecodeWorkload, history_rows


def _layer_kernels(fused, cuda_core, q, pool, table, positions, new_row, tiles, scale, tile_out,
                   tile_lse, workspace, status, part_offsets, out, lse, stream, kv_ready=False):
    """The layer's kernels: tail write + attention + merge of the tiles in one
    launch (fused), or as three launches."""
    geo_h, geo_d = tile_out.shape[-2], tile_out.shape[-1]
    n_tiles = np.asarray(tiles).shape[1]
    if fused and not cuda_core:
        merged = n_tiles > 1
        B.paged_decode_attn_lse_append(q, pool, table, tiles, scale, positions, new_row,
                                       tile_out, tile_lse, workspace, stream=stream,
                                       kv_ready=kv_ready, merged_out=out if merged else None,
                                       merged_lse=lse if merged else None)
        return
    B.kv_append_rows(pool, table, positions, new_row, status=status, stream=stream)
    B.paged_decode_attn_lse(q, pool, table, tiles, scale, tile_out, tile_lse, workspace,
                            stream=stream, cuda_core=cuda_core)
    if n_tiles > 1:
        # With one tile per request the merge is the identity (a single
        # partial is returned bit for bit): out and lse are views of the tile
        # outputs and no merge launch is needed.
        B.lse_merge(tile_out.view(-1, geo_h, geo_d), tile_lse.view(-1, geo_h), part_offsets,
                    out, lse, stream=stream)


class _Outputs:
    def __init__(self, w: DecodeWorkload, n_layers: int, device):
        geo = w.geometry
        self.tile_out = torch.empty((n_layers, w.batch, w.n_tiles, geo.n_q_heads, geo.head_dim),
                                    dtype=torch.float32, device=device)
        self.tile_lse = torch.empty((n_layers, w.batch, w.n_tiles, geo.n_q_heads),
                                    dtype=torch.float32, device=device)
        if w.n_tiles == 1:
            self.out = self.tile_out[:, :, 0]
            self.lse = self.tile_lse[:, :, 0]
        else:
            self.out = torch.empty((n_layers, w.batch, geo.n_q_heads, geo.head_dim),
                                   dtype=torch.float32, device=device)
            self.lse = torch.empty((n_layers, w.batch, geo.n_q_heads), dtype=torch.float32,
                                   device=device)
        self.part_offsets = torch.arange(0, (w.batch + 1) * w.n_tiles, w.n_tiles,
                                         dtype=torch.int32, device=device)


def _stage_marks(timeline, h2d):
    """Timing events of one stage, when ``timeline`` is a list (measurement
    only; the routes run without them).  Five events per stage:
      0  on the H2D stream before the stage's waits and copies are enqueued
      1  on the H2D stream after its copies and page-table fill
      2  on the compute stream after its wait on the copy event
      3  on the compute stream after the attention kernels
      4  on the D2H stream after the tail write-back (or the stage's end)
    """
    if timeline is None:
        return None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    ev[0].record(h2d)
    return ev


def _stage_marks_mid(ev, h2d, compute):
    if ev is not None:
        ev[1].record(h2d)
        ev[2].record(compute)


def _stage_marks_end(timeline, ev, compute):
    if ev is not None:
        ev[3].record(compute)
        timeline.append(ev)


def _stage_marks_wb(ev, d2h):
    if ev is not None:
        ev[4].record(d2h)


class ResidentDecode:
    """Decode step over a device-resident pool [layers][pages][64][row_elems]."""

    def __init__(self, w: DecodeWorkload, t: dict, cuda_core: bool = False,
                 tiles: np.ndarray | None = None, stream=None, fused: bool = True,
                 kv_ready: bool = False):
        self.w = w
        self.t = t
        self.cuda_core = cuda_core
        self.fused = fused
        # The pool and page table change only through this object's own
        # launches (each layer's new row, stored by that layer's launch), so
        # the caller may let each launch load pages before the previous
        # kernel ends; it must then not write them with other kernels
        # between steps without a stream synchronisation.
        self.kv_ready = kv_ready
        self.tiles = np.ascontiguousarray(w.tiles if tiles is None else tiles, dtype=np.int32)
        self.n_layers = t["pool"].shape[0]
        dev = t["pool"].device
        self.stream = stream
        geo = w.geometry
        self.o = _Outputs(w, self.n_layers, dev) if tiles is None else None
        if self.o is None:
            wt = DecodeWorkload(w.name, w.seed, w.n_layers, w.lengths, self.tiles, w.page_table,
                                w.pool_pages, w.spare_pages, w.geometry)
            self.o = _Outputs(wt, self.n_layers, dev)
        self.workspace = B.alloc_workspace(w.batch, self.tiles.shape[1], geo.n_q_heads,
                                           geo.n_kv_heads, geo.head_dim, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def layer(self, i: int, attention_only: bool = False):
        t, o, geo = self.t, self.o, self.w.geometry
        if attention_only:
            B.paged_decode_attn_lse(t["q"][i], t["pool"][i], t["page_table"], self.tiles,
                                    geo.scale, o.tile_out[i], o.tile_lse[i], self.workspace,
                                    stream=self.stream, cuda_core=self.cuda_core)
            return
        _layer_kernels(self.fused, self.cuda_core, t["q"][i], t["pool"][i], t["page_table"],
                       t["positions"], t["new_rows"][i], self.tiles, geo.scale, o.tile_out[i],
                       o.tile_lse[i], self.workspace, self.status, o.part_offsets, o.out[i],
                       o.lse[i], self.stream, kv_ready=self.kv_ready)

    def step(self):
        for i in range(self.n_layers):
            self.layer(i)

    def kernel_status(self) -> int:
        return int(self.workspace[:4].view(torch.int32).item()) | int(self.status.item())


class HostHistory:
    """Pinned host owner of every (layer, request) history segment.

    Segment (l, r) holds L_r rows of row_bytes, contiguous, in logical token
    order, as in "GPU memory management", section "A host pool that explains
    its own size".  Row L_r - 1 is the new token's slot; the write-back fills it.
    """

    def __init__(self, w: DecodeWorkload, t: dict, layers=None):
        geo = w.geometry
        self.w = w
        self.layers = list(range(t["pool"].shape[0])) if layers is None else list(layers)
        lengths = [int(L) for L in w.lengths]
        self.offsets = {}
        total = 0
        for i in range(len(self.layers)):
            for r, L in enumerate(lengths):
                self.offsets[(i, r)] = total
                total += L
        self._mem = B.PinnedBuffer(total * geo.row_bytes)
        self.rows = self._mem.tensor.view(torch.bfloat16).view(total, geo.row_elems)
        for i in range(len(self.layers)):
            for r, L in enumerate(lengths):
                off = self.offsets[(i, r)]
                # device rows straight into the pinned segment
                self.rows[off:off + L].copy_(history_rows(w, t["pool"][i], r))
        # the new token's host row is unknown until the write-back
        for i in range(len(self.layers)):
            for r, L in enumerate(lengths):
                self.rows[self.offsets[(i, r)] + L - 1].zero_()

    def row_address(self, i: int, r: int, row: int) -> int:
        return self.rows.data_ptr() + (self.offsets[(i, r)] + row) * self.w.geometry.row_bytes

    def row(self, i: int, r: int, row: int) -> torch.Tensor:
        return self.rows[self.offsets[(i, r)] + row]

    def close(self):
        if getattr(self, "_mem", None) is not None:
            self.rows = None
            self._mem.close()
            self._mem = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CompactStore:
    """Pinned host store of compact pages beside a HostHistory, filled by the
    library's background converter ("KV-cache engineering", section "Exact
    recent pages, compact older pages").

    Compact page p of (layer i, request r) sits at ``address(i, r, p)``; a
    page is staged compact only once the converter has published it.
    """

    def __init__(self, w: DecodeWorkload, host: HostHistory, n_threads: int = 8):
        geo = w.geometry
        self.w, self.host = w, host
        self.page_bytes = B.compact_page_bytes(geo.n_kv_heads, geo.head_dim)
        self.n_layers = len(host.layers)
        self.offsets = {}
        total = 0
        for i in range(self.n_layers):
            for r in range(w.batch):
                self.offsets[(i, r)] = total
                total += w.max_pages * self.page_bytes
        self._mem = B.PinnedBuffer(total)
        self.buf = self._mem.tensor
        exact = [host.row_address(i, r, 0) for i in range(self.n_layers) for r in range(w.batch)]
        comp = [self.buf.data_ptr() + self.offsets[(i, r)]
                for i in range(self.n_layers) for r in range(w.batch)]
        self.compactor = B.Compactor(self.n_layers, w.batch, geo.n_kv_heads, geo.head_dim,
                                     w.max_pages, exact, comp, n_threads=n_threads)

    def address(self, i: int, r: int, page: int) -> int:
        return self.buf.data_ptr() + self.offsets[(i, r)] + page * self.page_bytes

    def mark_written(self, lengths):
        """Pages below each request's new token are fully written in every
        layer (the rows before L - 1); queue them for conversion."""
        pt = self.w.geometry.page_tokens
        for r, L in enumerate(lengths):
            self.compactor.mark_written(r, max(0, int(L) - 1) // pt)

    def published(self, r: int):
        return [s == B.PA_PAGE_PUBLISHED for s in self.compactor.states(r)]

    def close(self):
        if getattr(self, "compactor", None) is not None:
            self.compactor.close()
            self.compactor = None
        if getattr(self, "_mem", None) is not None:
            self.buf = None
            self._mem.close()
            self._mem = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StagedDecode:
    """Decode step with host-owned history staged per layer into arena slots.

    The arena is one device allocation: an optional resident window region
    (sink + newest pages of every (layer, request), copied in once) followed
    by ``n_slots`` staging slots each big enough for one layer's staged pages.
    """

    def __init__(self, w: DecodeWorkload, t: dict, host: HostHistory, n_slots: int = 2,
                 cuda_core: bool = False, compute_stream=None, h2d_stream=None,
                 d2h_stream=None, leases: bool = False, fused: bool = True,
                 compact: CompactStore | None = None):
        geo = w.geometry
        self.w, self.t, self.host, self.cuda_core = w, t, host, cuda_core
        self.compact = compact
        self.leases = leases
        self.fused = fused
        self.timeline = None       # a list: timing events of every stage (see stage_marks)
        self.step_index = 0
        self.receipts = []
        self.n_layers = t["pool"].shape[0]
        dev = t["pool"].device
        self.compute = compute_stream or torch.cuda.current_stream(dev)
        self.h2d = h2d_stream or torch.cuda.Stream(dev)
        self.d2h = d2h_stream or torch.cuda.Stream(dev)
        self.tiles = np.ascontiguousarray(w.tiles, dtype=np.int32)
        pt = geo.page_tokens
        sink, recent = w.window if w.window else (0, 0)
        self.plan = []          # per layer index: list of (request, owner, runs)
        win_pages = 0
        win_base = {}
        for i in range(self.n_layers):
            for r in range(w.batch):
                n = w.pages_of(r)
                if w.window and n > sink + recent:
                    win_base[(i, r)] = win_pages
                    win_pages += sink + recent
        staged_max = 0
        for i in range(self.n_layers):
            reqs = []
            staged = 0
            for r in range(w.batch):
                L, n = int(w.lengths[r]), w.pages_of(r)
                owner = (i << 32) | r
                if (i, r) in win_base:
                    wb = win_base[(i, r)]
                    mid = n - sink - recent
                    runs = [dict(logical_page=0, n_pages=sink, resident_page=wb),
                            dict(logical_page=sink, n_pages=mid, n_rows=mid * pt,
                                 host_rows=host.row_address(i, r, sink * pt)),
                            dict(logical_page=n - recent, n_pages=recent,
                                 resident_page=wb + sink)]
                    staged += mid
                else:
                    runs = [dict(logical_page=0, n_pages=n, n_rows=L - 1,
                                 host_rows=host.row_address(i, r, 0))]
                    staged += n
                reqs.append((r, owner, runs))
            staged_max = max(staged_max, staged)
            self.plan.append(reqs)
        self.win_pages = win_pages
        self.slot_pages = max(1, staged_max)
        arena_pages = win_pages + n_slots * self.slot_pages
        page_bytes = pt * geo.row_bytes
        landing = 0
        if compact is not None:                 # room for a slot of compact pages
            landing = -(-self.slot_pages * compact.page_bytes // 256) * 256
        self.arena_buf = torch.empty(arena_pages * page_bytes + n_slots * landing,
                                     dtype=torch.uint8, device=dev)
        self.arena = self.arena_buf[: arena_pages * page_bytes].view(torch.bfloat16).view(
            arena_pages, pt, geo.row_elems)
        self.arena.fill_(float("nan"))          # canary: unwritten rows read as NaN
        self.page_tables = torch.zeros((n_slots, w.batch, w.max_pages), dtype=torch.int32,
                                       device=dev)
        torch.cuda.synchronize(dev)
        self.handle = B.Arena(self.arena_buf.data_ptr(), self.arena_buf.numel(), geo.row_bytes,
                              n_slots, win_pages, self.slot_pages, self.page_tables.data_ptr(),
                              w.batch, w.max_pages, compute_stream=self.compute,
                              h2d_stream=self.h2d, d2h_stream=self.d2h,
                              compact_head_dim=geo.head_dim if compact is not None else 0,
                              landing_offset=arena_pages * page_bytes if landing else 0,
                              landing_bytes=landing)
        # The resident window is copied in once, from the pinned host history
        # (the new token's row comes from the step's own tail write).
        loads = []
        for (i, r), wb in win_base.items():
            n, L = w.pages_of(r), int(w.lengths[r])
            for k, lp in enumerate(list(range(sink)) + list(range(n - recent, n))):
                rows = min(L - 1, (lp + 1) * pt) - lp * pt
                if rows > 0:
                    loads.append((wb + k, rows, host.row_address(i, r, lp * pt)))
        self.handle.load_resident(loads)
        self.exact_plan = self.plan
        if compact is not None:
            self.replan()
        self.o = _Outputs(w, self.n_layers, dev)
        self.workspace = B.alloc_workspace(w.batch, w.n_tiles, geo.n_q_heads, geo.n_kv_heads,
                                           geo.head_dim, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.tails = []
        for i in range(self.n_layers):
            self.tails.append([(r, int(w.lengths[r]) - 1,
                                host.row_address(i, r, int(w.lengths[r]) - 1), (i << 32) | r)
                               for r in range(w.batch)])

    def replan(self):
        """Stage every published page of the exact plan's staged runs in its
        compact form ("runs of two representations"); the rest stays exact."""
        pt = self.w.geometry.page_tokens
        published = [self.compact.published(r) for r in range(self.w.batch)]
        plan = []
        for i, reqs in enumerate(self.exact_plan):
            out = []
            for r, owner, runs in reqs:
                L = int(self.w.lengths[r])
                new_runs = []
                for run in runs:
                    if "host_rows" not in run:
                        new_runs.append(run)
                        continue
                    lp, end = run["logical_page"], run["logical_page"] + run["n_pages"]
                    while lp < end:
                        kind = published[r][lp]
                        start = lp
                        while lp < end and published[r][lp] == kind:
                            lp += 1
                        n = lp - start
                        if kind:
                            new_runs.append(dict(logical_page=start, n_pages=n, n_rows=n * pt,
                                                 host_compact=self.compact.address(i, r, start)))
                        else:
                            rows = min(lp * pt, L - 1) - start * pt
                            new_runs.append(dict(logical_page=start, n_pages=n,
                                                 n_rows=max(0, rows),
                                                 host_rows=self.host.row_address(i, r,
                                                                                 start * pt)))
                out.append((r, owner, new_runs))
            plan.append(out)
        self.plan = plan

    def arena_bytes(self) -> int:
        return self.arena_buf.numel()

    def stages_per_step(self) -> int:
        return self.n_layers

    def stage_bytes(self) -> list:
        """Host-to-device bytes of each stage of a step (one per layer)."""
        geo = self.w.geometry
        out = []
        for reqs in self.plan:
            total = 0
            for _, _, runs in reqs:
                for run in runs:
                    if "host_compact" in run:
                        total += run["n_pages"] * self.compact.page_bytes
                    elif "host_rows" in run:
                        total += run["n_rows"] * geo.row_bytes
            out.append(total)
        return out

    def staged_bytes_per_step(self) -> int:
        """Host-to-device bytes the current plan moves per step."""
        return sum(self.stage_bytes())

    def _kernels(self, i: int, table):
        t, o, geo = self.t, self.o, self.w.geometry
        _layer_kernels(self.fused, self.cuda_core, t["q"][i], self.arena, table, t["positions"],
                       t["new_rows"][i], self.tiles, geo.scale, o.tile_out[i], o.tile_lse[i],
                       self.workspace, self.status, o.part_offsets, o.out[i], o.lse[i],
                       self.compute)

    def _lease_step(self):
        """One step as leases: begin, kernels, attention event, tail write-back
        and seal per layer; every lease is retired (host waits, receipts) at
        the end of the step."""
        live = []
        for i in range(self.n_layers):
            lease = self.handle.lease_begin(i, self.step_index, self.plan[i])
            self._kernels(i, self.page_tables[lease.slot])
            att = self.handle.lease_attention_done(lease.lease_id)
            wb = self.handle.lease_writeback(lease.lease_id, self.tails[i])
            self.handle.lease_seal(lease.lease_id, att, wb)
            live.append(lease.lease_id)
        self.receipts = [self.handle.lease_retire(lid) for lid in live]
        self.step_index += 1

    def layer(self, i: int):
        tl = _stage_marks(self.timeline, self.h2d)
        slot, _ = self.handle.stage_layer(i, self.plan[i])
        _stage_marks_mid(tl, self.h2d, self.compute)
        self._kernels(i, self.page_tables[slot])
        _stage_marks_end(self.timeline, tl, self.compute)
        self.handle.mark_attention_done(i)
        self.handle.writeback_tail(i, self.tails[i])
        _stage_marks_wb(tl, self.d2h)

    def step(self):
        if self.leases:
            self._lease_step()
            return
        for i in range(self.n_layers):
            self.layer(i)

    def drain(self):
        self.handle.drain()

    def kernel_status(self) -> int:
        return int(self.workspace[:4].view(torch.int32).item()) | int(self.status.item())

    def close(self):
        self.handle.close()


def tile_units(w: DecodeWorkload):
    """(request, tile index, start, end) of every tile, in request then tile
    order (empty tiles included: their launch writes output 0, LSE -inf)."""
    return [(r, k, int(w.tiles[r, k, 0]), int(w.tiles[r, k, 1]))
            for r in range(w.batch) for k in range(w.n_tiles)]


def tile_kernels(w, t, i, r, k, s, e, pool, table_row, o, workspace, stream):
    """Attention of one (request, tile) as its own launch (B = 1): fused with
    the new row's store and substitution when the tile holds the new token."""
    geo = w.geometry
    tiles = np.array([[[s, e]]], dtype=np.int32)
    out = o.tile_out[i][r:r + 1, k:k + 1]
    lse = o.tile_lse[i][r:r + 1, k:k + 1]
    L = int(w.lengths[r])
    if s <= L - 1 < e:
        B.paged_decode_attn_lse_append(t["q"][i][r:r + 1], pool, table_row, tiles, geo.scale,
                                       t["positions"][r:r + 1], t["new_rows"][i][r:r + 1], out,
                                       lse, workspace, stream=stream)
    else:
        B.paged_decode_attn_lse(t["q"][i][r:r + 1], pool, table_row, tiles, geo.scale, out, lse,
                                workspace, stream=stream)


class TiledStagedDecode:
    """Host-owned history staged per (request, tile) instead of per layer: the
    arena holds ``n_slots`` slots of one tile's pages ("GPU memory
    management", section "Pages held by right, borrowed or free": the arena
    stages pages for 32K-token tiles), each tile is attended by its own launch
    as soon as its
    copy lands, and the layer's tiles are merged after the last one.  The
    device working set is n_slots tiles whatever the context length.

    Results equal, bit for bit, the resident route run with the same launches
    (one per tile; ``resident_tiled_step``); a launch's split points depend on
    its own pages, so they differ from the one-launch-per-layer route at the
    rounding level.  Workloads with a resident window are not supported here.
    """

    def __init__(self, w: DecodeWorkload, t: dict, host: HostHistory, n_slots: int = 2,
                 compute_stream=None):
        if w.window:
            raise ValueError("TiledStagedDecode stages whole tiles; no resident window")
        geo = w.geometry
        pt = geo.page_tokens
        self.w, self.t, self.host = w, t, host
        self.n_layers = t["pool"].shape[0]
        dev = t["pool"].device
        self.compute = compute_stream or torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.units = tile_units(w)
        self.timeline = None       # a list: timing events of every stage (see stage_marks)
        self.slot_pages = max([-(-e // pt) - s // pt for _, _, s, e in self.units if e > s],
                              default=1)
        self.arena = torch.full((n_slots * self.slot_pages, pt, geo.row_elems), float("nan"),
                                dtype=torch.bfloat16, device=dev)
        self.page_tables = torch.zeros((n_slots, w.batch, w.max_pages), dtype=torch.int32,
                                       device=dev)
        torch.cuda.synchronize(dev)
        self.handle = B.Arena(self.arena.data_ptr(), self.arena.numel() * 2, geo.row_bytes,
                              n_slots, 0, self.slot_pages, self.page_tables.data_ptr(),
                              w.batch, w.max_pages, compute_stream=self.compute,
                              h2d_stream=self.h2d, d2h_stream=self.d2h)
        self.o = _Outputs(w, self.n_layers, dev)
        self.workspace = B.alloc_workspace(1, 1, geo.n_q_heads, geo.n_kv_heads, geo.head_dim,
                                           device=dev)

    def arena_bytes(self) -> int:
        return self.arena.numel() * 2

    def stages_per_step(self) -> int:
        return self.n_layers * sum(1 for _, _, s, e in self.units if e > s)

    def stage_bytes(self) -> list:
        """Host-to-device bytes of each stage of a step: one per non-empty
        (layer, request, tile), in issue order."""
        w, pt, rb = self.w, self.w.geometry.page_tokens, self.w.geometry.row_bytes
        out = []
        for _ in range(self.n_layers):
            for r, _, s, e in self.units:
                if e <= s:
                    continue
                L = int(w.lengths[r])
                p0, p1 = s // pt, -(-e // pt)
                out.append(max(0, min(p1 * pt, L - 1) - p0 * pt) * rb)
        return out

    def layer(self, i: int):
        w, geo = self.w, self.w.geometry
        pt = geo.page_tokens
        for u, (r, k, s, e) in enumerate(self.units):
            if e <= s:           # nothing to stage: the launch writes 0 / -inf
                tile_kernels(w, self.t, i, r, k, s, e, self.arena, self.page_tables[0][r:r + 1],
                             self.o, self.workspace, self.compute)
                continue
            L = int(w.lengths[r])
            p0, p1 = s // pt, -(-e // pt)
            rows = min(p1 * pt, L - 1) - p0 * pt
            owner = (i << 32) | r
            key = i * len(self.units) + u
            tl = _stage_marks(self.timeline, self.h2d)
            slot, _ = self.handle.stage_layer(key, [(r, owner, [dict(
                logical_page=p0, n_pages=p1 - p0, n_rows=max(0, rows),
                host_rows=self.host.row_address(i, r, p0 * pt))])])
            _stage_marks_mid(tl, self.h2d, self.compute)
            tile_kernels(w, self.t, i, r, k, s, e, self.arena,
                         self.page_tables[slot][r:r + 1], self.o, self.workspace, self.compute)
            _stage_marks_end(self.timeline, tl, self.compute)
            self.handle.mark_attention_done(key)
            if s <= L - 1 < e:
                self.handle.writeback_tail(key, [(r, L - 1, self.host.row_address(i, r, L - 1),
                                                  owner)])
            _stage_marks_wb(tl, self.d2h)
        if w.n_tiles > 1:
            o = self.o
            B.lse_merge(o.tile_out[i].view(-1, geo.n_q_heads, geo.head_dim),
                        o.tile_lse[i].view(-1, geo.n_q_heads), o.part_offsets, o.out[i],
                        o.lse[i], stream=self.compute)

    def step(self):
        for i in range(self.n_layers):
            self.layer(i)

    def drain(self):
        self.handle.drain()

    def kernel_status(self) -> int:
        return int(self.workspace[:4].view(torch.int32).item())

    def close(self):
        self.handle.close()


def resident_tiled_step(w, t, o, workspace, stream=None):
    """The resident route with TiledStagedDecode's launches: one attention
    launch per (request, tile) over the device pool, then the tile merge."""
    geo = w.geometry
    for i in range(t["pool"].shape[0]):
        for r, k, s, e in tile_units(w):
            tile_kernels(w, t, i, r, k, s, e, t["pool"][i], t["page_table"][r:r + 1], o,
                         workspace, stream)
        if w.n_tiles > 1:
            B.lse_merge(o.tile_out[i].view(-1, geo.n_q_heads, geo.head_dim),
                        o.tile_lse[i].view(-1, geo.n_q_heads), o.part_offsets, o.out[i],
                        o.lse[i], stream=stream)


class PlannedDecode:
    """Decode steps whose device window follows the admission planner.

    The arena holds, per layer, one region of the planner's pool pages (pool
    page p of layer l is arena page l * pool_pages + p) followed by the
    staging slots.  At each step the planner decides every context's hot
    pages ("Staging without a stall", section "Admission that does
    arithmetic"); pages that turned hot are copied in once from pinned host
    memory by the arena (kv_load_resident: after the previous step's
    attention and write-back are done with the pool pages they reuse), and
    each layer stages every page that is not hot.  Contexts are the
    workload's requests; all run every step.

    With a CompactStore, the hot window stays exact and every cold page that
    the background converter has published is staged compact ("KV-cache
    engineering", section "Exact recent pages, compact older pages").  A page
    is handed to the converter only once the device event recorded after the
    write-backs that completed it has fired (checked without blocking at the
    next step), so it is fully written in every layer, in host memory.
    """

    def __init__(self, w: DecodeWorkload, t: dict, host: HostHistory, planner,
                 targets, bursts, n_slots: int = 2, compute_stream=None, fused: bool = True,
                 compact: CompactStore | None = None):
        geo = w.geometry
        self.w, self.t, self.host, self.planner = w, t, host, planner
        self.fused = fused
        self.compact = compact
        self.pending = []          # (event after a step's write-backs, full pages per request)
        self.compact_used = {}     # this step's compact-staged pages per (layer, request)
        self.n_layers = t["pool"].shape[0]
        dev = t["pool"].device
        self.dev = dev
        self.compute = compute_stream or torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.pool_pages, _ = planner.info()
        self.win_pages = self.n_layers * self.pool_pages
        self.slot_pages = max(1, sum(w.pages_of(r) for r in range(w.batch)))
        arena_pages = self.win_pages + n_slots * self.slot_pages
        page_bytes = geo.page_tokens * geo.row_bytes
        landing = 0
        if compact is not None:
            landing = -(-self.slot_pages * compact.page_bytes // 256) * 256
        self.arena_buf = torch.empty(arena_pages * page_bytes + n_slots * landing,
                                     dtype=torch.uint8, device=dev)
        self.arena = self.arena_buf[: arena_pages * page_bytes].view(torch.bfloat16).view(
            arena_pages, geo.page_tokens, geo.row_elems)
        self.arena.fill_(float("nan"))
        self.page_tables = torch.zeros((n_slots, w.batch, w.max_pages), dtype=torch.int32,
                                       device=dev)
        torch.cuda.synchronize(dev)
        self.handle = B.Arena(self.arena_buf.data_ptr(), self.arena_buf.numel(), geo.row_bytes,
                              n_slots, self.win_pages, self.slot_pages,
                              self.page_tables.data_ptr(), w.batch, w.max_pages,
                              compute_stream=self.compute, h2d_stream=self.h2d,
                              d2h_stream=self.d2h,
                              compact_head_dim=geo.head_dim if compact is not None else 0,
                              landing_offset=arena_pages * page_bytes if landing else 0,
                              landing_bytes=landing)
        for r in range(w.batch):
            planner.admit(r, int(targets[r]), int(bursts[r]))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = B.alloc_workspace(w.batch, 1, geo.n_q_heads, geo.n_kv_heads,
                                           geo.head_dim, device=dev)
        self.tile_out = torch.empty((self.n_layers, w.batch, 1, geo.n_q_heads, geo.head_dim),
                                    dtype=torch.float32, device=dev)
        self.tile_lse = torch.empty((self.n_layers, w.batch, 1, geo.n_q_heads),
                                    dtype=torch.float32, device=dev)
        self.out = self.tile_out[:, :, 0]        # one tile per request: no merge
        self.lse = self.tile_lse[:, :, 0]
        self.part_offsets = torch.arange(0, w.batch + 1, dtype=torch.int32, device=dev)
        self.resident = [dict() for _ in range(w.batch)]

    def _copy_in(self, lengths):
        """Copy the pages that turned hot into their pool pages, every layer
        (one kv_load_resident call: ordered after the previous step's
        attention and write-backs, which may read the pool pages reused)."""
        pt = self.w.geometry.page_tokens
        loads = []
        for r in range(self.w.batch):
            res = self.resident[r]
            for lp in self.planner.copied(r):
                lo = lp * pt
                rows = min(int(lengths[r]) - 1, lo + pt) - lo   # the new row comes from append
                if rows <= 0:
                    continue
                for i in range(self.n_layers):
                    loads.append((i * self.pool_pages + res[lp], rows,
                                  self.host.row_address(i, r, lo)))
        self.handle.load_resident(loads)

    def _runs(self, i, r, L, published=None):
        """Page runs of request r for layer i: hot pages from the pool,
        maximal runs of cold pages staged from the host (compact where
        ``published`` says the converter has published the page)."""
        pt = self.w.geometry.page_tokens
        n = -(-L // pt)
        res = self.resident[r]
        runs, lp = [], 0
        used = self.compact_used.setdefault((i, r), [])
        while lp < n:
            if lp in res:
                runs.append(dict(logical_page=lp, n_pages=1,
                                 resident_page=i * self.pool_pages + res[lp]))
                lp += 1
                continue
            start = lp
            kind = bool(published and published[lp])
            while lp < n and lp not in res and bool(published and published[lp]) == kind:
                lp += 1
            if kind:
                runs.append(dict(logical_page=start, n_pages=lp - start,
                                 n_rows=(lp - start) * pt,
                                 host_compact=self.compact.address(i, r, start)))
                used.extend(range(start, lp))
                continue
            rows = min(lp * pt, L - 1) - start * pt
            runs.append(dict(logical_page=start, n_pages=lp - start, n_rows=max(0, rows),
                             host_rows=self.host.row_address(i, r, start * pt)))
        return runs

    def _publish_written(self):
        """Hand the converter every page completed by steps whose write-backs
        have finished (a non-blocking event query per pending step)."""
        while self.pending and self.pending[0][0].query():
            _, full = self.pending.pop(0)
            for r, f in enumerate(full):
                self.compact.compactor.mark_written(r, f)

    def step(self, lengths):
        """One decode step at the given lengths (tokens, including the new one)."""
        w, t, geo = self.w, self.t, self.w.geometry
        admitted = self.planner.step([(r, int(lengths[r])) for r in range(w.batch)])
        if not all(admitted):
            raise RuntimeError(f"planner refused contexts {admitted}")
        self.resident = [self.planner.resident(r) for r in range(w.batch)]
        published = None
        self.compact_used = {}
        if self.compact is not None:
            self._publish_written()
            published = [self.compact.published(r) for r in range(w.batch)]
        self._copy_in(lengths)
        tiles = np.zeros((w.batch, 1, 2), dtype=np.int32)
        tiles[:, 0, 1] = lengths
        for i in range(self.n_layers):
            reqs = [(r, (i << 32) | r,
                     self._runs(i, r, int(lengths[r]), published[r] if published else None))
                    for r in range(w.batch)]
            slot, _ = self.handle.stage_layer(i, reqs)
            _layer_kernels(self.fused, False, t["q"][i], self.arena, self.page_tables[slot],
                           t["positions"], t["new_rows"][i], tiles, geo.scale, self.tile_out[i],
                           self.tile_lse[i], self.workspace, self.status, self.part_offsets,
                           self.out[i], self.lse[i], self.compute)
            self.handle.mark_attention_done(i)
            self.handle.writeback_tail(
                i, [(r, int(lengths[r]) - 1, self.host.row_address(i, r, int(lengths[r]) - 1),
                     (i << 32) | r) for r in range(w.batch)])
        if self.compact is not None:
            ev = torch.cuda.Event()
            ev.record(self.d2h)
            pt = geo.page_tokens
            self.pending.append((ev, [int(L) // pt for L in lengths]))

    def kernel_status(self) -> int:
        return int(self.workspace[:4].view(torch.int32).item()) | int(self.status.item())

    def close(self):
        self.handle.close()
