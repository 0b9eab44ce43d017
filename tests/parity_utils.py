"""Shared helpers of the GPU parity tests (test infrastructure only)."""

import numpy as np
import torch

import oracle

TOL_OUT = 2e-3      # max-abs on outputs vs the fp64 oracle
TOL_LSE = 1e-4      # max-abs on LSE vs the fp64 oracle
TOL_SPLIT = 1e-5    # tiled+merged vs single-tile, GPU vs GPU


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_request(w, t, i, r, tiles=None, gather_on_device=False):
    """Oracle results of request r in layer index i (new row applied)."""
    geo = w.geometry
    tiles = w.tiles[r] if tiles is None else tiles
    L = int(w.lengths[r])
    n = w.pages_of(r)
    if gather_on_device:
        idx = torch.as_tensor(w.page_table[r, :n], dtype=torch.long, device=t["pool"].device)
        pool_bits = bits(t["pool"][i].index_select(0, idx))
        table = np.arange(n, dtype=np.int32)
    else:
        pool_bits = bits(t["pool"][i])
        table = w.page_table[r]
    return oracle.decode_layer(bits(t["q"][i, r]), pool_bits, table, L, tiles, geo.scale,
                               geo.n_kv_heads, geo.head_dim,
                               new_row_bits=bits(t["new_rows"][i, r]))


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def assert_close_to_oracle(gpu_tile_out, gpu_tile_lse, gpu_out, gpu_lse, ref, tiles, what=""):
    """Per-tile partials and merged output of one request vs the oracle."""
    for k, (s, e) in enumerate(tiles):
        go = gpu_tile_out[k].double().cpu().numpy()
        gl = gpu_tile_lse[k].double().cpu().numpy()
        if e <= s:
            assert np.all(go == 0.0), f"{what} empty tile {k} output not 0"
            assert np.all(gl == -np.inf), f"{what} empty tile {k} lse not -inf"
            continue
        eo = max_abs(go, ref["tile_out"][k])
        el = max_abs(gl, ref["tile_lse"][k])
        assert eo <= TOL_OUT, f"{what} tile {k} [{s},{e}) out err {eo}"
        assert el <= TOL_LSE, f"{what} tile {k} [{s},{e}) lse err {el}"
    if gpu_out is not None:
        # merge of the oracle's own tiles: equals the unsplit attention when
        # the tiles partition the history (pinned in the oracle tests)
        eo = max_abs(gpu_out.double().cpu().numpy(), ref["out"])
        el = max_abs(gpu_lse.double().cpu().numpy(), ref["lse"])
        assert eo <= TOL_OUT, f"{what} merged out err {eo}"
        assert el <= TOL_LSE, f"{what} merged lse err {el}"
