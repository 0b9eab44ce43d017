"""Plain float64 definition of what the decode-attention path computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code may use it.

Sources, cited by page title and section:

* "KV-cache engineering", section "Exact recent pages, compact older pages":
  a request's history is cut into tiles; each tile's attention returns its
  normalised output and its log-sum-exp; an FP32 merge weights every partial by
  exp(LSE_i - max LSE), sums the weighted outputs, divides by the summed weights
  and returns max + log(sum) as the merged LSE, which is softmax over the union
  of the keys.  Separately normalised outputs are never averaged.
* "KV-cache engineering", section "Costing the bus before changing anything":
  the exact path reads every byte of history for every generated token.
* "GPU memory management", section "A host pool that explains its own size":
  a history is, per dense layer, a segment of context length x 4,096 bytes
  (one 4,096-byte row per token).

Readings where the pages are silent (each one is listed in the design notes):

* GQA: query head h attends with kv head floor(h / G), G = Hq / Hkv.
* Logits are s_j = scale * <q_h, k_j>; the LSE is natural-log based and
  includes the scale.
* A row of the pool is [K of kv heads 0..Hkv-1 | V of kv heads 0..Hkv-1], each
  head_dim bf16 values; a page is ``page_tokens`` consecutive rows.
* An empty tile has output 0 and LSE -inf; merging only empty tiles gives
  output 0 and LSE -inf.  A NaN anywhere propagates.

Nothing here blocks, fuses or reorders beyond the definitions: the attention is
the softmax over all keys written out, and the merge is the four steps of the
merge rule in the order the page gives them.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "request_history",
    "attention",
    "tile_attention",
    "lse_merge",
    "decode_layer",
    "merge_stress_partials",
    "softmax_union",
]


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact conversion of bfloat16 bit patterns (uint16) to float64.

    A bfloat16 is the upper half of an IEEE binary32, so placing the 16 bits in
    the high half of a 32-bit word gives the same number as a float32, which
    float64 holds exactly.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def request_history(pool_bits, page_table_row, length, n_kv_heads, head_dim,
                    page_tokens=64):
    """Gather one request's K and V history in logical token order.

    ``pool_bits`` is uint16 [n_pages][page_tokens][2 * n_kv_heads * head_dim]
    (bf16 bits of one layer's pool).  ``page_table_row[p]`` is the physical page
    that holds logical page p.  Token j lives in row j % page_tokens of physical
    page page_table_row[j // page_tokens].

    Returns (K, V), float64 arrays of shape [length][n_kv_heads][head_dim].
    Follows the row-per-token history segments of "GPU memory management",
    section "A host pool that explains its own size".
    """
    pool_bits = np.asarray(pool_bits, dtype=np.uint16)
    n_pages_used = -(-int(length) // page_tokens)
    pages = np.asarray(page_table_row[:n_pages_used], dtype=np.int64)
    rows = pool_bits[pages].reshape(n_pages_used * page_tokens, -1)[: int(length)]
    kv = bf16_bits_to_f64(rows).reshape(int(length), 2, n_kv_heads, head_dim)
    return kv[:, 0], kv[:, 1]


def attention(q, K, V, scale):
    """Exact softmax attention of every query head over all keys (float64).

    q: [Hq][D]; K, V: [L][Hkv][D].  For query head h with kv head
    g = h // (Hq / Hkv):
        s_j     = scale * sum_d q[h, d] * K[j, g, d]
        m       = max_j s_j
        Z       = sum_j exp(s_j - m)
        out[h]  = sum_j exp(s_j - m) * V[j, g] / Z
        lse[h]  = m + log Z
    The max shift is the textbook way to evaluate the same quantity without
    overflow; it does not change the result.  L == 0 gives out 0, lse -inf.

    Returns (out [Hq][D], lse [Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n_q, d = q.shape
    n_keys, n_kv, _ = K.shape
    group = n_q // n_kv
    out = np.zeros((n_q, d), dtype=np.float64)
    lse = np.full((n_q,), -np.inf, dtype=np.float64)
    if n_keys == 0:
        return out, lse
    for h in range(n_q):
        g = h // group
        s = scale * (K[:, g, :] @ q[h])
        m = np.max(s)
        if np.isnan(m):
            out[h] = np.nan
            lse[h] = np.nan
            continue
        w = np.exp(s - m)
        z = np.sum(w)
        out[h] = (w @ V[:, g, :]) / z
        lse[h] = m + np.log(z)
    return out, lse


def tile_attention(q, K, V, tiles, scale):
    """Per-tile partials: attention over the keys of each token range.

    ``tiles`` is a sequence of [start, end) token ranges over the request's
    logical history (the tiles of "KV-cache engineering", section "Exact recent
    pages, compact older pages").  Each tile returns its own normalised output
    and LSE.

    Returns (outs [T][Hq][D], lses [T][Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    outs = np.zeros((len(tiles),) + q.shape, dtype=np.float64)
    lses = np.zeros((len(tiles), q.shape[0]), dtype=np.float64)
    for i, (start, end) in enumerate(tiles):
        outs[i], lses[i] = attention(q, K[start:end], V[start:end], scale)
    return outs, lses


def lse_merge(outs, lses):
    """Merge per-tile (output, LSE) partials into softmax over the union of keys.

    The rule of "KV-cache engineering", section "Exact recent pages, compact
    older pages", step by step, per head:
        1. M    = max_i LSE_i
        2. w_i  = exp(LSE_i - M)
        3. out  = (sum_i w_i * out_i) / (sum_i w_i)
        4. LSE  = M + log(sum_i w_i)
    Partials are summed in increasing tile order.  When every partial has
    LSE -inf (only empty tiles, or none) the result is out 0, LSE -inf.

    outs: [P][H][D], lses: [P][H].  Returns (out [H][D], lse [H]).
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    n_parts = lses.shape[0]
    n_heads = lses.shape[1] if lses.ndim == 2 else outs.shape[1]
    d = outs.shape[2] if outs.ndim == 3 else 0
    out = np.zeros((n_heads, d), dtype=np.float64)
    lse = np.full((n_heads,), -np.inf, dtype=np.float64)
    if n_parts == 0:
        return out, lse
    for h in range(n_heads):
        col = lses[:, h]
        if np.any(np.isnan(col)):
            out[h] = np.nan
            lse[h] = np.nan
            continue
        big_m = np.max(col)
        if big_m == -np.inf:
            continue
        w = np.exp(col - big_m)
        acc = np.zeros(d, dtype=np.float64)
        wsum = 0.0
        for i in range(n_parts):
            acc = acc + w[i] * outs[i, h]
            wsum = wsum + w[i]
        out[h] = acc / wsum
        lse[h] = big_m + math.log(wsum)
    return out, lse


def decode_layer(q_bits, pool_bits, page_table_row, length, tiles, scale,
                 n_kv_heads, head_dim, page_tokens=64, new_row_bits=None):
    """One request, one layer of a decode step: per-tile partials and the merge.

    ``new_row_bits`` (optional, uint16 [2 * Hkv * D]) is the new token's K/V row;
    it replaces history row ``length - 1`` before attention, as the device tail
    write does (the configured length includes the new token).

    Returns dict(tile_out, tile_lse, out, lse, unsplit_out, unsplit_lse) where
    ``unsplit_*`` is the attention over the whole history in one piece.
    """
    q = bf16_bits_to_f64(q_bits)
    K, V = request_history(pool_bits, page_table_row, length, n_kv_heads,
                           head_dim, page_tokens)
    if new_row_bits is not None and length > 0:
        row = bf16_bits_to_f64(new_row_bits).reshape(2, n_kv_heads, head_dim)
        K = K.copy()
        V = V.copy()
        K[length - 1] = row[0]
        V[length - 1] = row[1]
    tile_out, tile_lse = tile_attention(q, K, V, tiles, scale)
    out, lse = lse_merge(tile_out, tile_lse)
    unsplit_out, unsplit_lse = attention(q, K, V, scale)
    return dict(tile_out=tile_out, tile_lse=tile_lse, out=out, lse=lse,
                unsplit_out=unsplit_out, unsplit_lse=unsplit_lse)


def softmax_union(logits, values):
    """Softmax-weighted average over a key set given its logits directly.

    logits: [H][N] (already scaled, any bias included); values: [N][D] shared by
    all heads.  Returns (out [H][D], lse [H]) with the same definitions as
    ``attention``.
    """
    logits = np.asarray(logits, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    n_heads, n_keys = logits.shape
    out = np.zeros((n_heads, values.shape[1]), dtype=np.float64)
    lse = np.full((n_heads,), -np.inf, dtype=np.float64)
    if n_keys == 0:
        return out, lse
    for h in range(n_heads):
        s = logits[h]
        m = np.max(s)
        w = np.exp(s - m)
        z = np.sum(w)
        out[h] = (w @ values) / z
        lse[h] = m + np.log(z)
    return out, lse


def merge_stress_partials(tile_logits, tile_values, tile_bias):
    """Partials and exact target for the LSE-merge stress case.

    Each tile i has logits [H][n_i] (before bias), values [n_i][D] and a bias
    [H] that is added to every logit of that tile for that head.  The partial
    of tile i is the float64 softmax over its own (biased) keys; the target is
    the float64 softmax over all tiles' biased keys at once, which is what the
    merge must reproduce ("softmax over the union of the keys").

    Returns (outs [P][H][D], lses [P][H], target_out [H][D], target_lse [H]).
    """
    outs = []
    lses = []
    all_logits = []
    all_values = []
    for s, v, c in zip(tile_logits, tile_values, tile_bias):
        biased = np.asarray(s, dtype=np.float64) + np.asarray(c, dtype=np.float64)[:, None]
        o, l = softmax_union(biased, v)
        outs.append(o)
        lses.append(l)
        all_logits.append(biased)
        all_values.append(np.asarray(v, dtype=np.float64))
    target_out, target_lse = softmax_union(np.concatenate(all_logits, axis=1),
                                           np.concatenate(all_values, axis=0))
    return np.stack(outs), np.stack(lses), target_out, target_lse
