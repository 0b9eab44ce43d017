"""Compact older pages on the GPU: staged compact runs expanded bit-exactly,
and the compact route's attention against the oracle.

"KV-cache engineering", sections "Exact recent pages, compact older pages" and
"What the hybrid tier buys": pages fully written in every layer are served in
their compact form once published, exact before that; a request's history is
then runs of two representations.  The compact form stands for the values
bf16_rne(code * scale) (the format of ``oracle/compact_pages.py``): the
expanded pages must hold exactly those bits, the staged route must equal the
resident route over a pool holding those values bit for bit, and both must
match the oracle's attention over them within the usual tolerances.
"""

import gc

import numpy as np
import pytest
import torch

from oracle import compact_pages as oc
from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import assert_close_to_oracle, bits, oracle_request

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return decode


def compact_pages_of(staged):
    """{(layer, request): logical pages the plan stages compact}."""
    used = {}
    for i, reqs in enumerate(staged.plan):
        for r, _, runs in reqs:
            used[(i, r)] = [run["logical_page"] + k for run in runs if "host_compact" in run
                            for k in range(run["n_pages"])]
    return used


def effective_pool(w, t, used):
    """A copy of the device pool whose compact-staged pages hold the values
    their compact form stands for (oracle quantize + dequantize, all rows of a
    (layer, request) at once)."""
    geo = w.geometry
    pt = geo.page_tokens
    t2 = {k: v.clone() for k, v in t.items()}
    for i in range(t["pool"].shape[0]):
        for r in range(w.batch):
            pages = used.get((i, r), [])
            if not pages:
                continue
            phys = torch.as_tensor(w.page_table[r, pages], dtype=torch.long, device="cuda")
            rows = bits(t["pool"][i].index_select(0, phys)).reshape(-1, geo.row_elems)
            codes, scales = oc.quantize_rows(rows, geo.n_kv_heads, geo.head_dim)
            deq = oc.dequantize_rows(codes, scales, geo.n_kv_heads, geo.head_dim)
            vals = torch.from_numpy(deq.view(np.int16).reshape(len(pages), pt, -1)).to("cuda")
            t2["pool"][i].index_copy_(0, phys, vals.view(torch.bfloat16))
    return t2


def run_compact(D, w, t, n_threads=8, leases=False):
    host = D.HostHistory(w, t)
    store = D.CompactStore(w, host, n_threads=n_threads)
    store.mark_written(w.lengths)
    store.compactor.wait_idle()
    published = [store.published(r) for r in range(w.batch)]
    staged = D.StagedDecode(w, t, host, n_slots=2, compact=store, leases=leases)
    staged.step()
    staged.drain()
    torch.cuda.synchronize()
    return host, store, staged, published


def test_expanded_pages_hold_the_oracle_values(D):
    w = wl.custom([640, 64 * 3 + 1, 100], [[(0, 640)], [(0, 193)], [(0, 100)]], seed=13,
                  n_layers=2, n_spare=3)
    t = wl.materialize(w, "cuda")
    host, store, staged, published = run_compact(D, w, t)
    geo = w.geometry
    assert [sum(p) for p in published] == [9, 3, 1]        # pages below the new token
    used = compact_pages_of(staged)
    assert all(used[(i, r)] == [p for p, ok in enumerate(published[r]) if ok]
               for i in range(2) for r in range(w.batch))
    for i in range(2):                                     # slot i holds layer i
        table = staged.page_tables[i].cpu().numpy()
        for r in range(w.batch):
            for lp in used[(i, r)]:
                exact = bits(host.rows[host.offsets[(i, r)] + lp * 64:
                                       host.offsets[(i, r)] + (lp + 1) * 64])
                ref = oc.convert_page(exact, geo.n_kv_heads, geo.head_dim)
                got = bits(staged.arena[int(table[r, lp])])
                assert np.array_equal(got, ref["values"]), (i, r, lp)
                assert store.compactor.crc(i, r, lp) == ref["crc"]
    st = staged.handle.stats()
    assert st.staged_bytes == staged.staged_bytes_per_step()
    staged.close()
    store.close()
    host.close()


@pytest.mark.parametrize("make,leases", [
    (lambda: wl.custom([640, 300, 64 * 5], [[(0, 640), (100, 400)], [(0, 300), (0, 0)],
                                             [(0, 320), (300, 320)]], seed=14, n_layers=2), False),
    (lambda: wl.ragged_window(n_layers=2, batch=3, min_len=8192, max_len=20000), True),
    (lambda: wl.four_requests_31744(n_layers=2), False),
], ids=["tiles", "ragged-window", "4x31744"])
def test_compact_route_equals_resident_over_the_values_it_stands_for(D, make, leases):
    w = make()
    t = wl.materialize(w, "cuda")
    host, store, staged, published = run_compact(D, w, t, leases=leases)
    te = effective_pool(w, t, compact_pages_of(staged))
    res = D.ResidentDecode(w, te)
    torch.cuda.synchronize()
    res.step()
    torch.cuda.synchronize()
    assert staged.kernel_status() == 0 and res.kernel_status() == 0
    assert torch.equal(staged.o.tile_out, res.o.tile_out)
    assert torch.equal(staged.o.tile_lse, res.o.tile_lse)
    assert torch.equal(staged.o.out, res.o.out) and torch.equal(staged.o.lse, res.o.lse)
    # the new rows went back to the host exact
    for i in range(w.n_layers):
        for r in range(w.batch):
            row = host.row(i, r, int(w.lengths[r]) - 1)
            assert torch.equal(row.view(torch.int16), t["new_rows"][i, r].cpu().view(torch.int16))
    # fewer bytes over the bus than the exact route would move
    exact_bytes = sum(run.get("n_rows", 0) * w.geometry.row_bytes
                      for reqs in staged.exact_plan for _, _, runs in reqs for run in runs
                      if "host_rows" in run)
    assert staged.staged_bytes_per_step() < 0.6 * exact_bytes
    staged.close()
    store.close()
    host.close()
    del te, res, t
    gc.collect()
    torch.cuda.empty_cache()


def test_compact_route_matches_the_oracle(D):
    w = wl.custom([640, 64 * 3 + 1], [[(0, 640), (0, 200)], [(0, 193), (190, 193)]], seed=15,
                  n_layers=1, n_spare=2)
    t = wl.materialize(w, "cuda")
    host, store, staged, published = run_compact(D, w, t)
    te = effective_pool(w, t, compact_pages_of(staged))
    o = staged.o
    for r in range(w.batch):
        ref = oracle_request(w, te, 0, r)
        assert_close_to_oracle(o.tile_out[0, r], o.tile_lse[0, r], o.out[0, r], o.lse[0, r], ref,
                               w.tiles[r], f"compact request {r}")
    # how far the compact representation moves the exact result (not exact by design)
    exact = D.ResidentDecode(w, t)
    exact.step()
    torch.cuda.synchronize()
    assert (o.out - exact.o.out).abs().max().item() < 0.05
    staged.close()
    store.close()
    host.close()
