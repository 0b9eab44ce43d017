"""Compact older pages: the second representation of a fully written page.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code may use it.

Sources, cited by page title and section:

* "KV-cache engineering", section "Exact recent pages, compact older pages":
  a request's history is cut into runs of two representations; a page is
  converted only after it is fully written in every layer, its CRC is computed
  and it is published; until then it is served exact.
* "KV-cache engineering", section "What the hybrid tier buys": a
  representation is judged by the bytes per token it stops moving over the
  bus.

The pages name no format.  The reading used here (listed in the design
notes) is a plain symmetric 8-bit one:

* For every token row and every (K or V, kv head) slice x of head_dim bf16
  values: s = max|x| / 127 in binary32 (round to nearest even), and the codes
  are c = clamp(round_half_even(x / s), -127, 127) with x / s a binary32
  division.  A slice of zeros has s = 0 and codes 0.  A page holding a
  non-finite value is not convertible and stays exact.
* A compact page of one layer is the codes, int8 [page_tokens][2 Hkv D], then
  the scales, float32 little-endian [page_tokens][2 Hkv]: 133,120 bytes for
  64 tokens x 4 kv heads x 256 against 262,144 exact.
* The value a compact page stands for is the bfloat16 (round to nearest even)
  of the binary32 product c * s.
* The CRC is CRC-32 with the reflected polynomial 0xEDB88320, initial value
  0xFFFFFFFF and a final xor with 0xFFFFFFFF (the ISO-HDLC / IEEE 802.3 CRC),
  over the compact page's bytes.

Every function is pinned by ``tests/test_oracle_compact_pins.py``.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "CODE_MAX",
    "compact_page_bytes_len",
    "f32_to_bf16_bits",
    "quantize_rows",
    "dequantize_rows",
    "page_bytes",
    "crc32",
    "convert_page",
    "effective_rows",
]

CODE_MAX = 127


def compact_page_bytes_len(page_tokens: int, n_kv_heads: int, head_dim: int) -> int:
    """Bytes of one layer's compact page: int8 codes then float32 scales."""
    return page_tokens * 2 * n_kv_heads * head_dim + page_tokens * 2 * n_kv_heads * 4


def f32_to_bf16_bits(x) -> np.ndarray:
    """bfloat16 bits (uint16) of binary32 values, rounded to nearest even.

    A bfloat16 keeps the upper 16 bits of a binary32.  Rounding to nearest
    even adds 0x7FFF plus the lowest kept bit before truncating, which rounds
    halfway cases to the value whose last kept bit is 0.  NaN stays a quiet
    NaN.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if np.any(nan):
        rounded = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), rounded)
    return rounded


def _bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_rows(rows_bits, n_kv_heads: int, head_dim: int):
    """Codes and scales of token rows, or None if a value is not finite.

    rows_bits: uint16 [n][2 * Hkv * D] (bf16 bits).  Returns (codes int8
    [n][2 * Hkv * D], scales float32 [n][2 * Hkv]); slice k of a row is
    columns [k * D, (k + 1) * D): K of kv heads 0..Hkv-1, then V.
    """
    x = _bf16_bits_to_f32(rows_bits)
    n = x.shape[0]
    if not np.all(np.isfinite(x)):
        return None
    groups = x.reshape(n, 2 * n_kv_heads, head_dim)
    amax = np.max(np.abs(groups), axis=2)                        # exact in binary32
    scales = np.divide(amax, np.float32(CODE_MAX), dtype=np.float32)
    codes = np.zeros(groups.shape, dtype=np.int8)
    nz = scales > 0
    if np.any(nz):
        ratio = np.divide(groups[nz], scales[nz][:, None], dtype=np.float32)
        q = np.rint(ratio)                                       # half to even
        codes[nz] = np.clip(q, -CODE_MAX, CODE_MAX).astype(np.int8)
    return codes.reshape(n, 2 * n_kv_heads * head_dim), scales


def dequantize_rows(codes, scales, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """bf16 bits [n][2 * Hkv * D] of the values the codes stand for:
    bf16_rne(binary32(c) * s)."""
    c = np.asarray(codes, dtype=np.int8)
    n = c.shape[0]
    groups = c.reshape(n, 2 * n_kv_heads, head_dim).astype(np.float32)
    prod = np.multiply(groups, np.asarray(scales, dtype=np.float32)[:, :, None],
                       dtype=np.float32)
    return f32_to_bf16_bits(prod).reshape(n, 2 * n_kv_heads * head_dim)


def page_bytes(codes, scales) -> bytes:
    """The compact page's byte image: codes (row-major int8), then scales
    (row-major little-endian float32)."""
    return (np.ascontiguousarray(codes, dtype=np.int8).tobytes()
            + np.ascontiguousarray(scales, dtype="<f4").tobytes())


def _crc_table():
    table = []
    for n in range(256):
        c = n
        for _ in range(8):
            c = (c >> 1) ^ 0xEDB88320 if c & 1 else c >> 1
        table.append(c)
    return table


_TABLE = _crc_table()


def crc32(data: bytes, crc: int = 0) -> int:
    """CRC-32 (reflected 0xEDB88320, init and final xor 0xFFFFFFFF), one byte
    at a time; ``crc`` continues a previous value."""
    c = crc ^ 0xFFFFFFFF
    for byte in bytes(data):
        c = _TABLE[(c ^ byte) & 0xFF] ^ (c >> 8)
    return c ^ 0xFFFFFFFF


def convert_page(rows_bits, n_kv_heads: int, head_dim: int):
    """Convert one layer's page (uint16 [page_tokens][2 Hkv D]).

    Returns dict(codes, scales, bytes, crc, values) with ``values`` the bf16
    bits the compact page stands for, or None when the page is not
    convertible (a non-finite value).
    """
    q = quantize_rows(rows_bits, n_kv_heads, head_dim)
    if q is None:
        return None
    codes, scales = q
    data = page_bytes(codes, scales)
    return dict(codes=codes, scales=scales, bytes=data, crc=crc32(data),
                values=dequantize_rows(codes, scales, n_kv_heads, head_dim))


def effective_rows(rows_bits, compact_pages, n_kv_heads: int, head_dim: int,
                   page_tokens: int = 64) -> np.ndarray:
    """A request's history rows as attention sees them when the logical pages
    in ``compact_pages`` are served compact and every other page exact.

    rows_bits: uint16 [L][2 Hkv D] in logical order.  A compact page must be
    fully written (all page_tokens rows inside the history) and convertible.
    """
    rows = np.array(rows_bits, dtype=np.uint16, copy=True)
    for lp in compact_pages:
        lo, hi = lp * page_tokens, (lp + 1) * page_tokens
        if hi > rows.shape[0]:
            raise ValueError(f"page {lp} is not fully written")
        page = convert_page(rows[lo:hi], n_kv_heads, head_dim)
        if page is None:
            raise ValueError(f"page {lp} is not convertible")
        rows[lo:hi] = page["values"]
    return rows
