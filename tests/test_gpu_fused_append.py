"""The fused tail write + attention launch against the two-launch sequence.

"KV-cache engineering", section "Exact decode attention over paged history",
and "Staging without a stall", section "Leases instead of buffers": the step's
new token is stored in its page and attended in the same step.  The fused
entry point must give the outputs of kv_append_rows followed by
paged_decode_attn_lse bit for bit, and leave the same bytes in the pool, even
when the pool row held NaN before the call (the kernel attends the new row
from its argument, not from the pool).
"""

import numpy as np
import pytest
import torch

from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import assert_close_to_oracle, oracle_request

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return decode


def poison_new_rows(w, t):
    """NaN in every request's new-token row of every layer's pool."""
    pt = w.geometry.page_tokens
    for r in range(w.batch):
        pos = int(w.lengths[r]) - 1
        page = int(w.page_table[r, pos // pt])
        t["pool"][:, page, pos % pt] = float("nan")


def clone(t):
    return {k: v.clone() for k, v in t.items()}


def run_both(D, w, t, kv_ready=False):
    poison_new_rows(w, t)
    tf, tu = clone(t), clone(t)
    fused = D.ResidentDecode(w, tf, fused=True, kv_ready=kv_ready)
    unfused = D.ResidentDecode(w, tu, fused=False)
    torch.cuda.synchronize()     # the clones' kernels are complete
    fused.step()
    unfused.step()
    torch.cuda.synchronize()
    return fused, unfused, tf, tu


def assert_same(fused, unfused, tf, tu):
    assert torch.equal(fused.o.tile_out, unfused.o.tile_out)
    assert torch.equal(fused.o.tile_lse, unfused.o.tile_lse)
    assert torch.equal(fused.o.out, unfused.o.out)
    assert torch.equal(fused.o.lse, unfused.o.lse)
    assert torch.equal(tf["pool"].view(torch.int16), tu["pool"].view(torch.int16))


def edge_workload():
    lengths = [1, 63, 64, 65, 150, 1000, 4097]
    tiles = [
        [(0, 1), (0, 0)],
        [(0, 63), (5, 6), (62, 63)],
        [(0, 64), (0, 32), (32, 64)],
        [(0, 65), (64, 65), (0, 64)],
        [(37, 101), (0, 150), (100, 150), (149, 150)],
        [(0, 1000), (0, 333), (333, 1000), (1, 999), (500, 500)],
        [(0, 4097), (4096, 4097), (63, 2049), (0, 4096)],
    ]
    return wl.custom(lengths, tiles, seed=21, n_spare=5, max_pages=70, n_layers=2)


def test_fused_equals_two_launches_on_edge_tiles(D):
    w = edge_workload()
    t = wl.materialize(w, "cuda")
    fused, unfused, tf, tu = run_both(D, w, t)
    assert fused.kernel_status() == 0 and unfused.kernel_status() == 0
    assert torch.isfinite(fused.o.out).all()
    assert_same(fused, unfused, tf, tu)
    for r in range(w.batch):
        ref = oracle_request(w, tf, 1, r)
        o = fused.o
        assert_close_to_oracle(o.tile_out[1, r], o.tile_lse[1, r], o.out[1, r], o.lse[1, r], ref,
                               w.tiles[r], f"fused request {r}")


@pytest.mark.parametrize("make", [wl.four_requests_31744, wl.ragged_window],
                         ids=["4x31744", "ragged-window"])
def test_fused_equals_two_launches_at_full_size(D, make):
    w = make(n_layers=2)
    t = wl.materialize(w, "cuda")
    fused, unfused, tf, tu = run_both(D, w, t)
    assert fused.kernel_status() == 0 and unfused.kernel_status() == 0
    assert_same(fused, unfused, tf, tu)
    del fused, unfused, tf, tu, t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kv_ready", [False, True], ids=["wait", "early-loads"])
def test_fused_over_several_launches(D, kv_ready):
    # 80 requests x 4 tiles x 4 kv heads = 1,280 units: the library issues two
    # launches, and only the first stores the new rows (the second may load
    # the pages the first writes early: it substitutes the rows anyway).
    rng = np.random.default_rng(4)
    lengths = rng.integers(1, 400, size=80)
    tiles = [[(0, int(L)), (0, int(L) // 2), (int(L) // 2, int(L)), (max(0, int(L) - 7), int(L))]
             for L in lengths]
    w = wl.custom(lengths, tiles, seed=8, n_spare=3)
    t = wl.materialize(w, "cuda")
    fused, unfused, tf, tu = run_both(D, w, t, kv_ready=kv_ready)
    assert fused.kernel_status() == 0 and unfused.kernel_status() == 0
    assert_same(fused, unfused, tf, tu)


def test_fused_bad_position_is_reported_and_not_stored(D):
    w = wl.custom([640, 200], [[(0, 640)], [(0, 200)]], seed=3, n_spare=2)
    t = wl.materialize(w, "cuda")
    t["positions"][0] = w.max_pages * w.geometry.page_tokens + 5
    before = t["pool"].clone()
    dec = D.ResidentDecode(w, t, fused=True)
    dec.layer(0)
    torch.cuda.synchronize()
    assert dec.kernel_status() & 4                      # PA_STATUS_BAD_ROW
    page = int(w.page_table[1, 199 // 64])
    changed = (t["pool"].view(torch.int16) != before.view(torch.int16)).any(dim=-1)
    assert changed.nonzero().tolist() == [[0, page, 199 % 64]]    # request 1's row only
    assert torch.isfinite(dec.o.out).all()


@pytest.mark.parametrize("make", [edge_workload, lambda: wl.four_requests_31744(n_layers=3)],
                         ids=["edge", "4x31744"])
def test_early_page_loads_change_no_bits(D, make):
    # PA_DECODE_KV_READY lets each launch load its first pages while the
    # previous kernel (the previous layer's merge) finishes; two steps back
    # to back must give the same bits as launches that wait first.
    w = make()
    t = wl.materialize(w, "cuda")
    runs = []
    for kv_ready in (True, False):
        tc = clone(t)
        dec = D.ResidentDecode(w, tc, kv_ready=kv_ready)
        torch.cuda.synchronize()     # the clone's kernels are complete
        dec.step()
        dec.step()
        torch.cuda.synchronize()
        assert dec.kernel_status() == 0
        runs.append((dec, tc))
    (a, ta), (b, tb) = runs
    assert_same(a, b, ta, tb)


def test_fused_merge_many_tiles_and_repeated_steps(D):
    # up to 20 tiles per request (some empty, some overlapping, one request
    # with a single tile): the in-kernel merge equals lse_merge bit for bit on
    # every one of three consecutive steps (its counters reset each time).
    rng = np.random.default_rng(12)
    lengths = [3000, 700, 64, 5000]
    tiles = []
    for L in lengths:
        cuts = sorted(rng.integers(0, L, size=18).tolist())
        t_req = [(0, cuts[0])] + [(a, b) for a, b in zip(cuts, cuts[1:])] + [(cuts[-1], L)]
        tiles.append(t_req[:20])
    tiles[2] = [(0, 64)]
    w = wl.custom(lengths, tiles, seed=17, n_spare=4, n_layers=2)
    t = wl.materialize(w, "cuda")
    poison_new_rows(w, t)
    tf, tu = clone(t), clone(t)
    fused = D.ResidentDecode(w, tf, fused=True)
    unfused = D.ResidentDecode(w, tu, fused=False)
    torch.cuda.synchronize()
    for _ in range(3):
        fused.step()
        unfused.step()
        torch.cuda.synchronize()
        assert fused.kernel_status() == 0 and unfused.kernel_status() == 0
        assert_same(fused, unfused, tf, tu)
