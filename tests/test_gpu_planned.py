"""Planner-driven device windows on the GPU: over several decode steps with
growing lengths and changing targets, the route whose hot pages follow the
admission planner (the rest staged from pinned host memory) returns the same
bits as the fully resident route, and every new token's row reaches its host
row bit for bit."""

import numpy as np
import pytest
import torch

from paged_decode_attention_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding, decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding, decode


def test_planned_windows_match_the_resident_route(mods):
    B, D = mods
    # one new token per step; the starts sit just below page boundaries so
    # every context's frontier crosses into a new page during the run
    start = np.array([64 * 812 - 2, 64 * 735 - 1, 64 * 860 - 4], dtype=np.int64)
    n_steps, grow = 10, 1
    final = start + grow * (n_steps - 1)
    w = wl.custom(final, [[(0, int(L))] for L in final], seed=23, n_layers=2, n_spare=8)
    t = wl.materialize(w, "cuda")
    host = D.HostHistory(w, t)
    # 1 GiB over 2 layers = 2,048 pool pages; the contexts want 2,400 in total
    planner = B.Planner(1, n_layers=2, max_contexts=4, max_context_tokens=int(final.max()))
    pd = D.PlannedDecode(w, t, host, planner, targets=[600, 600, 600], bursts=[200, 200, 200])
    crossed = 0
    for s in range(n_steps):
        lengths = start + grow * s
        if s == 4:
            planner.set_target(0, 300, 0)      # context 0 now holds pages above its target
            planner.set_target(2, 900, 100)
        t["positions"].copy_(torch.as_tensor(lengths - 1, dtype=torch.int32))
        pd.step(lengths)
        if s > 0:
            crossed += sum(len(planner.copied(r)) for r in range(w.batch))
        tiles = np.zeros((w.batch, 1, 2), dtype=np.int32)
        tiles[:, 0, 1] = lengths
        res = D.ResidentDecode(w, t, tiles=tiles)
        res.step()
        torch.cuda.synchronize()
        pd.handle.drain()
        assert res.kernel_status() == 0 and pd.kernel_status() == 0
        assert torch.equal(pd.out, res.o.out), f"step {s}"
        assert torch.equal(pd.lse, res.o.lse), f"step {s}"
        for i in range(w.n_layers):
            for r in range(w.batch):
                row = host.row(i, r, int(lengths[r]) - 1)
                assert torch.equal(row.view(torch.int16),
                                   t["new_rows"][i, r].cpu().view(torch.int16))
    c = planner.counters()
    assert c["steps"] == n_steps and c["refused"] == 0, c
    assert c["reclaimed_borrowed"] + c["reclaimed_above_target"] > 0, c  # windows moved under pressure
    assert crossed > 0, c                                                # frontiers crossed pages
    pd.close()
    host.close()


def test_planned_route_serves_published_cold_pages_compact(mods):
    """Exact until published: with the converter held the route is the exact
    one; once released, every published cold page is staged compact and the
    route equals the resident route over the values those pages stand for.
    Pages completed by the steps themselves are handed to the converter only
    after their write-backs finished."""
    B, D = mods
    from oracle import compact_pages as oc
    from parity_utils import bits
    start = np.array([64 * 150 - 2, 64 * 130 - 1, 64 * 170 - 4], dtype=np.int64)
    n_steps = 8
    final = start + n_steps - 1
    w = wl.custom(final, [[(0, int(L))] for L in final], seed=29, n_layers=2, n_spare=8)
    geo = w.geometry
    t = wl.materialize(w, "cuda")
    host = D.HostHistory(w, t)
    store = D.CompactStore(w, host, n_threads=4)
    store.compactor.hold(True)
    store.mark_written(start)                    # queued, served exact while held
    planner = B.Planner(1, n_layers=2, max_contexts=4, max_context_tokens=int(final.max()))
    pd = D.PlannedDecode(w, t, host, planner, targets=[40, 40, 40], bursts=[0, 0, 0],
                         compact=store)
    used_steps = []
    for s in range(n_steps):
        if s == 2:
            store.compactor.hold(False)
            store.compactor.wait_idle()
        lengths = start + s
        t["positions"].copy_(torch.as_tensor(lengths - 1, dtype=torch.int32))
        pd.step(lengths)
        torch.cuda.synchronize()
        pd.handle.drain()
        used = {k: list(v) for k, v in pd.compact_used.items()}
        used_steps.append(sum(len(v) for v in used.values()))
        for i in range(w.n_layers):            # the history keeps every step's new row
            B.kv_append_rows(t["pool"][i], t["page_table"], t["positions"], t["new_rows"][i])
        te = {k: v.clone() for k, v in t.items()}
        for (i, r), pages in used.items():
            if not pages:
                continue
            phys = torch.as_tensor(w.page_table[r, pages], dtype=torch.long, device="cuda")
            rows = bits(t["pool"][i].index_select(0, phys)).reshape(-1, geo.row_elems)
            codes, scales = oc.quantize_rows(rows, geo.n_kv_heads, geo.head_dim)
            deq = oc.dequantize_rows(codes, scales, geo.n_kv_heads, geo.head_dim)
            vals = torch.from_numpy(deq.view(np.int16).reshape(len(pages), 64, -1)).to("cuda")
            te["pool"][i].index_copy_(0, phys, vals.view(torch.bfloat16))
        tiles = np.zeros((w.batch, 1, 2), dtype=np.int32)
        tiles[:, 0, 1] = lengths
        res = D.ResidentDecode(w, te, tiles=tiles)
        torch.cuda.synchronize()
        res.step()
        torch.cuda.synchronize()
        assert res.kernel_status() == 0 and pd.kernel_status() == 0
        assert torch.equal(pd.out, res.o.out), f"step {s}"
        assert torch.equal(pd.lse, res.o.lse), f"step {s}"
        del te, res
    assert used_steps[0] == used_steps[1] == 0                 # held: everything exact
    assert all(u > 0 for u in used_steps[2:])                  # published cold pages compact
    hot = sum(len(planner.resident(r)) for r in range(w.batch))
    assert hot == 120                                          # the exact window
    pd.close()
    store.close()
    host.close()
