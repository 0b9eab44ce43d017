"""The synthetic workload builders (shapes and page tables; no GPU)."""

import numpy as np
import pytest

from paged_decode_attention_attn_gb300 import workloads as wl


@pytest.mark.parametrize("make", [lambda: wl.four_requests_31744(n_layers=2),
                                  lambda: wl.one_request_262144(n_layers=2),
                                  lambda: wl.ragged_window(n_layers=2),
                                  lambda: wl.uniform(3, 5000, 2048, n_layers=2),
                                  lambda: wl.uniform(1, 1, n_layers=1)])
def test_tables_map_every_page_once(make):
    w = make()
    used = []
    for r in range(w.batch):
        n = w.pages_of(r)
        assert n == -(-int(w.lengths[r]) // 64)
        used.extend(w.page_table[r, :n].tolist())
    assert len(set(used)) == len(used)                      # no page shared
    assert all(0 <= p < w.pool_pages for p in used)
    assert not set(used) & set(np.asarray(w.spare_pages).tolist())
    for r in range(w.batch):                                 # tiles inside the history
        for s, e in w.tiles[r]:
            assert 0 <= s <= e <= int(w.lengths[r])


def test_uniform_tiles_cover_the_history():
    w = wl.uniform(2, 5000, 2048, n_layers=3)
    assert w.name == "2x5000-3layers-3tiles" and w.n_layers == 3
    assert w.tiles[1].tolist() == [[0, 2048], [2048, 4096], [4096, 5000]]
    with pytest.raises(ValueError):
        wl.uniform(0, 10)
