"""Seeded synthetic workloads for paged GQA decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention or merge arithmetic.  The tests, the smoke check and the bench use it
to feed both the CUDA path and the CPU oracle with the same inputs.

Geometry of every workload: 24 query heads, 4 KV heads (G = 6), head_dim 256,
bf16 K/V, 64-token pages, one 4,096-byte row per token per layer laid out as
[K of kv heads 0..3 | V of kv heads 0..3], scale 1/16.

Random values are float32 N(0, 1) draws from a seeded ``torch.Generator`` on the
device that holds the tensor, rounded to bf16 with round-to-nearest-even.
Index-like choices (page permutations, ragged lengths, scaled-key positions)
come from ``numpy.random.default_rng`` seeded from the workload seed.

Canaries: spare pool pages and the rows past the end of each request's last
page are NaN, so a read of anything the page table and tiles do not name shows
up as NaN in the output.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_TOKENS = 64


@dataclass(frozen=True)
class Geometry:
    n_q_heads: int = 24
    n_kv_heads: int = 4
    head_dim: int = 256
    page_tokens: int = PAGE_TOKENS
    scale: float = 1.0 / 16.0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def row_elems(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim

    @property
    def row_bytes(self) -> int:
        return 2 * self.row_elems


@dataclass
class DecodeWorkload:
    """Shapes, page tables and tiling of one decode-attention workload."""

    name: str
    seed: int
    n_layers: int
    lengths: np.ndarray            # int64 [B]; includes the new token (row L-1)
    tiles: np.ndarray              # int32 [B][T][2], token [start, end); empty tiles pad
    page_table: np.ndarray         # int32 [B][max_pages], physical page of each logical page
    pool_pages: int                # physical pages per layer in the resident pool
    spare_pages: np.ndarray        # int64, NaN-filled canary pages
    geometry: Geometry = field(default_factory=Geometry)
    scaled_key_fraction: float = 0.0   # fraction of positions whose K row is x8
    window: tuple | None = None        # (sink_pages, recent_pages) resident window

    @property
    def batch(self) -> int:
        return int(self.lengths.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def n_tiles(self) -> int:
        return int(self.tiles.shape[1])

    def kv_bytes_per_step(self) -> int:
        """History bytes one decode step reads: sum_r L_r x row_bytes x layers."""
        return int(self.lengths.sum()) * self.geometry.row_bytes * self.n_layers

    def pages_of(self, r: int) -> int:
        return -(-int(self.lengths[r]) // self.geometry.page_tokens)


def _split_tiles(start: int, end: int, tile_tokens: int):
    out = []
    s = start
    while s < end:
        e = min(end, s + tile_tokens)
        out.append((s, e))
        s = e
    return out


def _pad_tiles(per_request):
    n_tiles = max(1, max(len(t) for t in per_request))
    tiles = np.zeros((len(per_request), n_tiles, 2), dtype=np.int32)
    for r, tl in enumerate(per_request):
        for i, (s, e) in enumerate(tl):
            tiles[r, i] = (s, e)
    return tiles


def _shuffled_tables(rng, lengths, max_pages, n_spare, page_tokens=PAGE_TOKENS):
    pages = [-(-int(L) // page_tokens) for L in lengths]
    pool_pages = sum(pages) + n_spare
    perm = rng.permutation(pool_pages)
    table = np.zeros((len(lengths), max_pages), dtype=np.int32)
    cursor = 0
    for r, n in enumerate(pages):
        table[r, :n] = perm[cursor:cursor + n]
        cursor += n
    spare = np.sort(perm[cursor:]).astype(np.int64)
    return table, pool_pages, spare


def tiny_decode(seed: int = 0) -> DecodeWorkload:
    """1 request, 1 layer, 2,048-token history (32 pages) shuffled inside a
    48-page pool whose 16 spare pages are NaN, 4 tiles of 512 tokens."""
    rng = np.random.default_rng(seed)
    lengths = np.array([2048], dtype=np.int64)
    table, pool_pages, spare = _shuffled_tables(rng, lengths, 32, 16)
    tiles = _pad_tiles([_split_tiles(0, 2048, 512)])
    return DecodeWorkload("tiny-decode-1x2048-4tiles", seed, 1, lengths, tiles,
                          table, pool_pages, spare)


def four_requests_31744(seed: int = 2, n_layers: int = 16) -> DecodeWorkload:
    """4 requests x 31,744-token histories (496 pages each), 16 layers, one
    32K tile per request."""
    rng = np.random.default_rng(seed)
    lengths = np.full(4, 31744, dtype=np.int64)
    table, pool_pages, spare = _shuffled_tables(rng, lengths, 496, 16)
    tiles = _pad_tiles([_split_tiles(0, 31744, 32768)] * 4)
    return DecodeWorkload("4x31744-16layers", seed, n_layers, lengths, tiles,
                          table, pool_pages, spare)


def one_request_262144(seed: int = 3, n_layers: int = 16) -> DecodeWorkload:
    """1 request, 262,144-token history (4,096 pages), 16 layers, 8 tiles of
    32,768 tokens."""
    rng = np.random.default_rng(seed)
    lengths = np.array([262144], dtype=np.int64)
    table, pool_pages, spare = _shuffled_tables(rng, lengths, 4096, 16)
    tiles = _pad_tiles([_split_tiles(0, 262144, 32768)])
    return DecodeWorkload("1x262144-16layers-8tiles", seed, n_layers, lengths,
                          tiles, table, pool_pages, spare)


def uniform(batch: int, length: int, tile_tokens: int = 32768, seed: int = 7,
            n_layers: int = 16) -> DecodeWorkload:
    """``batch`` requests of ``length`` tokens each, cut into tiles of
    ``tile_tokens`` (the last one ragged), pages shuffled in a pool with 16
    NaN spare pages: the bench's other shapes."""
    if batch < 1 or length < 1 or tile_tokens < 1:
        raise ValueError("batch, length and tile_tokens must be >= 1")
    rng = np.random.default_rng(seed)
    lengths = np.full(batch, length, dtype=np.int64)
    table, pool_pages, spare = _shuffled_tables(rng, lengths, -(-length // PAGE_TOKENS), 16)
    tiles = _pad_tiles([_split_tiles(0, length, tile_tokens)] * batch)
    return DecodeWorkload(f"{batch}x{length}-{n_layers}layers-{tiles.shape[1]}tiles", seed,
                          n_layers, lengths, tiles, table, pool_pages, spare)


def window_tiles(length: int, sink_pages: int = 1, recent_pages: int = 64,
                 tile_tokens: int = 32768, page_tokens: int = PAGE_TOKENS):
    """Tiles of a request whose sink page and newest pages stay resident.

    Order: the staged middle as tiles of at most ``tile_tokens`` tokens, then
    the sink range, then the recent range.  A request with no more than
    sink + recent pages is one tile.
    """
    n_pages = -(-int(length) // page_tokens)
    if n_pages <= sink_pages + recent_pages:
        return [(0, int(length))]
    mid_start = sink_pages * page_tokens
    mid_end = (n_pages - recent_pages) * page_tokens
    return (_split_tiles(mid_start, mid_end, tile_tokens)
            + [(0, mid_start), (mid_end, int(length))])


def ragged_window(seed: int = 4, n_layers: int = 16, batch: int = 8,
                  min_len: int = 8192, max_len: int = 131072) -> DecodeWorkload:
    """8 requests with lengths uniform in [8,192, 131,072]; sink page + newest
    64 pages resident, the rest staged; 1% of keys scaled x8."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(min_len, max_len, size=batch, endpoint=True).astype(np.int64)
    max_pages = -(-max_len // PAGE_TOKENS)
    table, pool_pages, spare = _shuffled_tables(rng, lengths, max_pages, 16)
    tiles = _pad_tiles([window_tiles(int(L)) for L in lengths])
    return DecodeWorkload(f"8-ragged-{min_len}-{max_len}-window-sink1-recent64",
                          seed, n_layers, lengths, tiles, table, pool_pages,
                          spare, scaled_key_fraction=0.01, window=(1, 64))


def custom(lengths, tiles_per_request, seed: int = 11, n_layers: int = 1,
           n_spare: int = 4, max_pages: int | None = None,
           geometry: Geometry | None = None) -> DecodeWorkload:
    """A workload with caller-chosen lengths and tiles (test edge cases)."""
    geometry = geometry or Geometry()
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    need = max(1, max(-(-int(L) // geometry.page_tokens) for L in lengths))
    table, pool_pages, spare = _shuffled_tables(rng, lengths, max_pages or need,
                                                n_spare, geometry.page_tokens)
    tiles = _pad_tiles([list(t) for t in tiles_per_request])
    return DecodeWorkload("custom", seed, n_layers, lengths, tiles, table,
                          pool_pages, spare, geometry=geometry)


def _bf16_randn(shape, gen, device, chunk_elems=1 << 28):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    pos = 0
    while pos < n:
        m = min(chunk_elems, n - pos)
        flat[pos:pos + m] = torch.randn(m, generator=gen, device=device,
                                        dtype=torch.float32).to(torch.bfloat16)
        pos += m
    return out


def _layer_gen(seed: int, layer: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(layer) * 7919 + 17)
    return g


def scaled_key_positions(w: DecodeWorkload, layer: int, r: int) -> np.ndarray:
    """Token positions (excluding the new token) whose K row is scaled x8."""
    n = int(np.floor(w.scaled_key_fraction * int(w.lengths[r])))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    rng = np.random.default_rng([w.seed, layer, r, 8])
    return np.sort(rng.choice(int(w.lengths[r]) - 1, size=n, replace=False)).astype(np.int64)


def materialize(w: DecodeWorkload, device, layers=None):
    """Device tensors of the workload.

    Returns a dict:
      pool       bf16 [n_layers][pool_pages][page_tokens][row_elems]
      q          bf16 [n_layers][B][Hq][D]
      new_rows   bf16 [n_layers][B][row_elems]  (the new token's K/V row)
      page_table int32 [B][max_pages]
      positions  int32 [B]  (row index L-1 of the new token)
    ``layers`` restricts generation to a subset (list of layer indices); the
    returned layer axis then follows that list.
    """
    geo = w.geometry
    layers = list(range(w.n_layers)) if layers is None else list(layers)
    nl = len(layers)
    pool = torch.empty((nl, w.pool_pages, geo.page_tokens, geo.row_elems),
                       dtype=torch.bfloat16, device=device)
    q = torch.empty((nl, w.batch, geo.n_q_heads, geo.head_dim),
                    dtype=torch.bfloat16, device=device)
    new_rows = torch.empty((nl, w.batch, geo.row_elems), dtype=torch.bfloat16,
                           device=device)
    table = torch.as_tensor(w.page_table, dtype=torch.int32).to(device)
    nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
    kw = geo.n_kv_heads * geo.head_dim
    for i, layer in enumerate(layers):
        gen = _layer_gen(w.seed, layer, device)
        pool[i] = _bf16_randn(pool[i].shape, gen, device)
        q[i] = _bf16_randn(q[i].shape, gen, device)
        new_rows[i] = _bf16_randn(new_rows[i].shape, gen, device)
        if len(w.spare_pages):
            idx = torch.as_tensor(w.spare_pages, dtype=torch.long, device=device)
            pool[i].index_fill_(0, idx, nan)
        for r in range(w.batch):
            L = int(w.lengths[r])
            n_pages = w.pages_of(r)
            last = int(w.page_table[r, n_pages - 1])
            used = L - (n_pages - 1) * geo.page_tokens
            pool[i, last, used:] = nan
            pos = scaled_key_positions(w, layer, r)
            if len(pos):
                pg = torch.as_tensor(w.page_table[r, pos // geo.page_tokens],
                                     dtype=torch.long, device=device)
                rw = torch.as_tensor(pos % geo.page_tokens, dtype=torch.long,
                                     device=device)
                pool[i, pg, rw, :kw] = pool[i, pg, rw, :kw] * 8
    positions = torch.as_tensor(w.lengths - 1, dtype=torch.int32).to(device)
    return dict(pool=pool, q=q, new_rows=new_rows, page_table=table,
                positions=positions)


def history_rows(w: DecodeWorkload, pool_layer: torch.Tensor, r: int) -> torch.Tensor:
    """Request r's rows [L][row_elems] gathered in logical order from one
    layer's pool (a layout copy: used to fill pinned host segments)."""
    n_pages = w.pages_of(r)
    idx = torch.as_tensor(w.page_table[r, :n_pages], dtype=torch.long,
                          device=pool_layer.device)
    rows = pool_layer.index_select(0, idx).reshape(-1, pool_layer.shape[-1])
    return rows[: int(w.lengths[r])]


@dataclass
class MergeStressCase:
    """Random draws of the LSE-merge stress workload (float64 numpy)."""

    tile_logits: list      # per request: list of [H][n_i] arrays
    tile_values: list      # per request: list of [n_i][D] arrays
    tile_bias: list        # per request: list of [H] arrays (uniform +-spread)
    n_heads: int
    head_dim: int


def merge_stress(seed: int = 5, n_requests: int = 64, n_heads: int = 24,
                 head_dim: int = 256, max_parts: int = 64, max_tile: int = 512,
                 spread: float = 80.0) -> MergeStressCase:
    """64 requests, each with 1..64 tiles of 1..512 keys; float32 N(0,1) logits
    and values; every (tile, head) gets a logit bias uniform in [-80, 80]."""
    rng = np.random.default_rng(seed)
    logits, values, bias = [], [], []
    for _ in range(n_requests):
        n_parts = int(rng.integers(1, max_parts, endpoint=True))
        lr, vr, br = [], [], []
        for _ in range(n_parts):
            n = int(rng.integers(1, max_tile, endpoint=True))
            lr.append(rng.standard_normal((n_heads, n), dtype=np.float32).astype(np.float64))
            vr.append(rng.standard_normal((n, head_dim), dtype=np.float32).astype(np.float64))
            br.append(rng.uniform(-spread, spread, size=n_heads))
        logits.append(lr)
        values.append(vr)
        bias.append(br)
    return MergeStressCase(logits, values, bias, n_heads, head_dim)


def merge_stress_layout(seed: int = 5, n_requests: int = 64, max_parts: int = 64) -> np.ndarray:
    """Partial offsets int32 [B+1] of a merge-stress-shaped input: request r
    owns partials [off[r], off[r+1]), a count uniform in 1..max_parts.  Used to
    time the merge on synthetic partials (the values then come from
    ``merge_stress_partials_device``)."""
    rng = np.random.default_rng([seed, 77])
    counts = rng.integers(1, max_parts, size=n_requests, endpoint=True)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def merge_stress_partials_device(offsets: np.ndarray, n_heads: int, head_dim: int, device,
                                 seed: int = 5, spread: float = 80.0):
    """Random fp32 partial outputs N(0,1) [P][H][D] and partial LSEs uniform in
    [-spread, spread] [P][H] on the device, for timing the merge."""
    n_parts = int(offsets[-1])
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 7919 + 3)
    out_parts = torch.randn((n_parts, n_heads, head_dim), generator=g, device=device,
                            dtype=torch.float32)
    lse_parts = (torch.rand((n_parts, n_heads), generator=g, device=device,
                            dtype=torch.float32) * 2 - 1) * spread
    return out_parts, lse_parts
