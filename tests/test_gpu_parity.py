"""GPU parity of the CUDA path against the fp64 oracle on small and edge cases.

Every call goes through the C-ABI library (ctypes binding).  Tolerances:
max-abs 2e-3 on outputs and 1e-4 on LSE against the oracle; 1e-5 between a
tiled+merged result and the single-tile result; bit equality where only the
physical placement of pages differs.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import (TOL_LSE, TOL_OUT, TOL_SPLIT, assert_close_to_oracle, bits, max_abs,
                          oracle_request)

pytestmark = pytest.mark.gpu

VARIANTS = [False, True]   # cuda_core flag: tensor-core kernel, CUDA-core kernel
VARIANT_IDS = ["tensor_core", "cuda_core"]


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding


@pytest.fixture(scope="module")
def D(B):
    from paged_decode_attention_attn_gb300 import decode
    return decode


def run_resident(D, w, t, cuda_core, tiles=None):
    dec = D.ResidentDecode(w, t, cuda_core=cuda_core, tiles=tiles)
    dec.step()
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    return dec


@pytest.mark.parametrize("cuda_core", VARIANTS, ids=VARIANT_IDS)
def test_tiny_decode_matches_oracle(B, D, cuda_core):
    w = wl.tiny_decode(seed=0)
    t = wl.materialize(w, "cuda")
    dec = run_resident(D, w, t, cuda_core)
    ref = oracle_request(w, t, 0, 0)
    o = dec.o
    assert torch.isfinite(o.tile_out).all() and torch.isfinite(o.out).all()
    assert_close_to_oracle(o.tile_out[0, 0], o.tile_lse[0, 0], o.out[0, 0], o.lse[0, 0], ref,
                           w.tiles[0], "tiny")
    # one tile over the whole history vs four tiles merged
    single = run_resident(D, w, t, cuda_core, tiles=np.array([[[0, 2048]]], dtype=np.int32))
    assert max_abs(single.o.tile_out[0, 0, 0].cpu(), o.out[0, 0].cpu()) <= TOL_SPLIT
    assert max_abs(single.o.tile_lse[0, 0, 0].cpu(), o.lse[0, 0].cpu()) <= TOL_SPLIT
    assert max_abs(single.o.tile_out[0, 0, 0].double().cpu(), ref["unsplit_out"]) <= TOL_OUT
    assert max_abs(single.o.tile_lse[0, 0, 0].double().cpu(), ref["unsplit_lse"]) <= TOL_LSE


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
    return wl.custom(lengths, tiles, seed=21, n_spare=5, max_pages=70)


@pytest.mark.parametrize("cuda_core", VARIANTS, ids=VARIANT_IDS)
def test_edge_cases_match_oracle(B, D, cuda_core):
    w = edge_workload()
    t = wl.materialize(w, "cuda")
    dec = run_resident(D, w, t, cuda_core)
    o = dec.o
    for r in range(w.batch):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(o.tile_out[0, r], o.tile_lse[0, r], o.out[0, r], o.lse[0, r],
                               ref, w.tiles[r], f"request {r}")


@pytest.mark.parametrize("cuda_core", VARIANTS, ids=VARIANT_IDS)
def test_physical_placement_does_not_change_bits(B, D, cuda_core):
    w = wl.custom([3000, 777, 64], [[(0, 3000), (100, 2000)], [(0, 777)], [(0, 64)]], seed=5,
                  n_spare=7)
    t = wl.materialize(w, "cuda")
    a = run_resident(D, w, t, cuda_core)
    # move every page to a new physical slot, rebuild the page table accordingly
    perm = np.random.default_rng(9).permutation(w.pool_pages)
    t2 = dict(t)
    pool2 = torch.empty_like(t["pool"])
    pool2[:, torch.as_tensor(perm, device="cuda")] = t["pool"]
    t2["pool"] = pool2
    table2 = w.page_table.copy()
    n_used = [w.pages_of(r) for r in range(w.batch)]
    for r in range(w.batch):
        table2[r, :n_used[r]] = perm[w.page_table[r, :n_used[r]]]
    w2 = wl.DecodeWorkload(w.name, w.seed, w.n_layers, w.lengths, w.tiles, table2, w.pool_pages,
                           perm[w.spare_pages], w.geometry)
    t2["page_table"] = torch.as_tensor(table2, device="cuda")
    b = run_resident(D, w2, t2, cuda_core)
    assert torch.equal(a.o.tile_out, b.o.tile_out)
    assert torch.equal(a.o.tile_lse, b.o.tile_lse)
    assert torch.equal(a.o.out, b.o.out) and torch.equal(a.o.lse, b.o.lse)


def test_pages_past_4_gib_of_pool(B, D):
    """The same pages placed at the top of a 5.4 GB pool (byte offsets past
    2^32, row coordinates past 2^24): bits unchanged, new rows stored there."""
    w = wl.custom([3000, 777], [[(0, 3000), (100, 2000)], [(0, 777)]], seed=6, n_spare=2)
    t = wl.materialize(w, "cuda")
    a = run_resident(D, w, t, False)
    big = 20480                                    # pages of 256 KiB: 5.37 GB
    top = np.arange(big - w.pool_pages, big)       # the old pool's pages, in order, at the top
    pool2 = torch.zeros((1, big) + tuple(t["pool"].shape[2:]), dtype=t["pool"].dtype,
                        device="cuda")
    pool2[:, big - w.pool_pages:] = t["pool"]
    table2 = w.page_table.copy()
    for r in range(w.batch):
        n = w.pages_of(r)
        table2[r, :n] = top[w.page_table[r, :n]]
    w2 = wl.DecodeWorkload(w.name, w.seed, w.n_layers, w.lengths, w.tiles, table2, big,
                           top[w.spare_pages], w.geometry)
    nan = torch.tensor(float("nan"), dtype=pool2.dtype, device="cuda")
    for r in range(w.batch):                       # the new rows must be stored again
        pos = int(w.lengths[r]) - 1
        pool2[0, int(table2[r, pos // 64]), pos % 64] = nan
    t2 = dict(t)
    t2["pool"] = pool2
    t2["page_table"] = torch.as_tensor(table2, device="cuda")
    b = run_resident(D, w2, t2, False)
    assert torch.equal(a.o.tile_out, b.o.tile_out) and torch.equal(a.o.tile_lse, b.o.tile_lse)
    assert torch.equal(a.o.out, b.o.out) and torch.equal(a.o.lse, b.o.lse)
    for r in range(w.batch):                       # the fused tail write landed up there
        pos = int(w.lengths[r]) - 1
        page = int(table2[r, pos // 64])
        assert page * 262144 > (1 << 32)
        assert torch.equal(pool2[0, page, pos % 64].view(torch.int16),
                           t["new_rows"][0, r].view(torch.int16))
    del pool2, t2
    torch.cuda.empty_cache()


# The tensor-core kernel carries each probability as a bf16 hi + lo pair
# (relative error <= 2^-18); the CUDA-core kernel keeps fp32.  Their outputs
# can differ by up to 2^-18 * max|v - out| (~4e-6 * 10 for N(0,1) values), so
# the two are held to 1e-4 here, well inside the 2e-3 bound both meet against
# the oracle.  LSEs do not depend on that rounding.
TOL_VARIANTS_OUT = 1e-4


def test_variants_agree(B, D):
    w = edge_workload()
    t = wl.materialize(w, "cuda")
    a = run_resident(D, w, t, False)
    b = run_resident(D, w, t, True)
    assert max_abs(a.o.out.cpu(), b.o.out.cpu()) <= TOL_VARIANTS_OUT
    assert max_abs(a.o.lse.cpu(), b.o.lse.cpu()) <= 2 * TOL_SPLIT


@pytest.mark.parametrize("cuda_core", VARIANTS, ids=VARIANT_IDS)
def test_bad_page_id_is_reported_not_read(B, D, cuda_core):
    w = wl.custom([640, 640], [[(0, 320), (320, 640)], [(0, 640), (0, 0)]], seed=3, n_spare=2)
    t = wl.materialize(w, "cuda")
    t["page_table"][0, 7] = w.pool_pages + 1000     # page 7 = tokens [448, 512)
    dec = D.ResidentDecode(w, t, cuda_core=cuda_core)
    dec.layer(0)
    torch.cuda.synchronize()
    assert dec.kernel_status() & B.PA_STATUS_BAD_PAGE
    o = dec.o
    assert torch.isnan(o.tile_out[0, 0, 1]).all() and torch.isnan(o.tile_lse[0, 0, 1]).all()
    assert torch.isfinite(o.tile_out[0, 0, 0]).all()        # tile 0 never touches page 7
    assert torch.isfinite(o.tile_out[0, 1]).all()
    ref = oracle_request(w, t, 0, 1)
    assert_close_to_oracle(o.tile_out[0, 1], o.tile_lse[0, 1], None, None, ref, w.tiles[1])


def test_append_rows_writes_exact_bytes(B):
    w = wl.custom([100, 64, 3], [[(0, 100)], [(0, 64)], [(0, 3)]], seed=4, n_spare=1)
    t = wl.materialize(w, "cuda")
    pool = t["pool"][0]
    before = pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_append_rows(pool, t["page_table"], t["positions"], t["new_rows"][0], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    changed = (pool.view(torch.int16) != before.view(torch.int16)).any(dim=-1)
    for r in range(w.batch):
        pos = int(w.lengths[r]) - 1
        page, row = int(w.page_table[r, pos // 64]), pos % 64
        assert torch.equal(pool[page, row].view(torch.int16), t["new_rows"][0, r].view(torch.int16))
        changed[page, row] = False
    assert not changed.any()                        # nothing else was written
    bad = torch.tensor([5000, 1, 2], dtype=torch.int32, device="cuda")
    before = pool.clone()
    B.kv_append_rows(pool, t["page_table"], bad, t["new_rows"][0], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & B.PA_STATUS_BAD_ROW
    # request 0 (position past its page table) is skipped; 1 and 2 land at rows 1 and 2
    changed = (pool.view(torch.int16) != before.view(torch.int16)).any(dim=-1)
    for r, pos in ((1, 1), (2, 2)):
        page = int(w.page_table[r, 0])
        assert torch.equal(pool[page, pos].view(torch.int16), t["new_rows"][0, r].view(torch.int16))
        changed[page, pos] = False
    assert not changed.any()


def merge_inputs_from_oracle(case, requests):
    outs, lses, offsets, targets = [], [], [0], []
    for r in requests:
        o, l, t_out, t_lse = oracle.merge_stress_partials(case.tile_logits[r], case.tile_values[r],
                                                          case.tile_bias[r])
        outs.append(o)
        lses.append(l)
        offsets.append(offsets[-1] + o.shape[0])
        targets.append((t_out, t_lse))
    return (np.concatenate(outs), np.concatenate(lses), np.array(offsets, dtype=np.int32),
            targets)


def test_lse_merge_stress_matches_unsplit_softmax(B):
    case = wl.merge_stress(seed=5)
    outs, lses, offsets, targets = merge_inputs_from_oracle(case, range(len(case.tile_logits)))
    assert np.ptp(lses) > 100                         # the +-80 spread is there
    dev = "cuda"
    op = torch.as_tensor(outs, dtype=torch.float32, device=dev)
    lp = torch.as_tensor(lses, dtype=torch.float32, device=dev)
    off = torch.as_tensor(offsets, device=dev)
    nb = len(targets)
    out = torch.empty((nb, case.n_heads, case.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((nb, case.n_heads), dtype=torch.float32, device=dev)
    B.lse_merge(op, lp, off, out, lse)
    torch.cuda.synchronize()
    worst_o = worst_l = 0.0
    for r, (t_out, t_lse) in enumerate(targets):
        worst_o = max(worst_o, max_abs(out[r].double().cpu(), t_out))
        worst_l = max(worst_l, max_abs(lse[r].double().cpu(), t_lse))
    assert worst_o <= TOL_OUT and worst_l <= TOL_LSE, (worst_o, worst_l)
    # the same partials through the oracle's own merge (fp32 inputs) agree too
    o32 = op.double().cpu().numpy()
    l32 = lp.double().cpu().numpy()
    for r in (0, nb // 2, nb - 1):
        mo, ml = oracle.lse_merge(o32[offsets[r]:offsets[r + 1]], l32[offsets[r]:offsets[r + 1]])
        assert max_abs(out[r].double().cpu(), mo) <= 1e-5
        assert max_abs(lse[r].double().cpu(), ml) <= 1e-4


@pytest.mark.parametrize("D", [4, 12, 128, 132, 256, 260, 520])
def test_lse_merge_head_dims_and_partial_counts(B, D):
    """Rows of any width (one or several 64-column passes, a ragged last one)
    and partial counts on both sides of the kernel's twelve-partial stages and
    of the eight-partial stages it had, against the oracle's fp64 merge of the
    same fp32 partials."""
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(D)
    H = 3
    counts = [1, 2, 7, 8, 9, 11, 12, 13, 15, 16, 17, 23, 24, 25, 33, 64]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    P = int(offsets[-1])
    parts = torch.randn((P, H, D), generator=g, device=dev)
    lses = (torch.rand((P, H), generator=g, device=dev) * 2 - 1) * 80
    out = torch.full((len(counts), H, D), 7.0, device=dev)
    lse = torch.full((len(counts), H), 7.0, device=dev)
    B.lse_merge(parts, lses, torch.as_tensor(offsets, device=dev), out, lse)
    torch.cuda.synchronize()
    o64 = parts.double().cpu().numpy()
    l64 = lses.double().cpu().numpy()
    for r in range(len(counts)):
        mo, ml = oracle.lse_merge(o64[offsets[r]:offsets[r + 1]], l64[offsets[r]:offsets[r + 1]])
        assert max_abs(out[r].double().cpu(), mo) <= 1e-5, (D, counts[r])
        assert max_abs(lse[r].double().cpu(), ml) <= 1e-4, (D, counts[r])
    assert torch.equal(out[0], parts[0]) and torch.equal(lse[0], lses[0])


def test_lse_merge_identity_and_edges(B):
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(1)
    H, D = 24, 256
    parts = torch.randn((4, H, D), generator=g, device=dev)
    lses = torch.randn((4, H), generator=g, device=dev) * 40
    lses[2] = -float("inf")                    # request 2: all -inf
    lses[3, 5] = float("nan")                  # request 3: one NaN head
    # requests: 0 -> [0,1) single; 1 -> [1,1) none; 2 -> [2,3) all -inf; 3 -> [3,4) nan
    off = torch.tensor([0, 1, 1, 2, 3, 4], dtype=torch.int32, device=dev)
    nb = 5
    out = torch.full((nb, H, D), 7.0, device=dev)
    lse = torch.full((nb, H), 7.0, device=dev)
    parts5 = torch.cat([parts[0:1], parts[2:3], parts[1:2], parts[3:4]])
    lses5 = torch.cat([lses[0:1], lses[2:3], lses[1:2], lses[3:4]])
    B.lse_merge(parts5, lses5, off, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out[0], parts5[0]) and torch.equal(lse[0], lses5[0])   # bitwise identity
    assert torch.all(out[1] == 0) and torch.all(lse[1] == -float("inf"))      # no partials
    assert torch.all(out[2] == 0) and torch.all(lse[2] == -float("inf"))      # all -inf
    assert torch.equal(out[3], parts5[2]) and torch.equal(lse[3], lses5[2])
    assert torch.isnan(lse[4, 5]) and torch.isnan(out[4, 5]).all()
    assert torch.isfinite(out[4, :5]).all()


GEOMETRIES = [(8, 8), (8, 1), (32, 4), (16, 2), (12, 6), (7, 7)]


@pytest.mark.parametrize("hq,hkv", GEOMETRIES, ids=[f"{a}q{b}kv" for a, b in GEOMETRIES])
def test_other_head_geometries_match_oracle(B, D, hq, hkv):
    # group sizes 1..8 and kv-head counts 1..8: every request's tiles and the
    # fused tail write and merge against the oracle, and the fused route
    # against the three-launch route bit for bit
    geo = wl.Geometry(n_q_heads=hq, n_kv_heads=hkv)
    w = wl.custom([700, 3000, 65], [[(0, 700), (100, 350)], [(0, 1500), (1500, 3000)],
                                     [(0, 65), (64, 65)]], seed=33, n_spare=3, geometry=geo)
    t = wl.materialize(w, "cuda")
    fused = D.ResidentDecode(w, {k: v.clone() for k, v in t.items()}, fused=True)
    split = D.ResidentDecode(w, {k: v.clone() for k, v in t.items()}, fused=False)
    torch.cuda.synchronize()
    fused.step()
    split.step()
    torch.cuda.synchronize()
    assert fused.kernel_status() == 0 and split.kernel_status() == 0
    assert torch.equal(fused.o.out, split.o.out) and torch.equal(fused.o.lse, split.o.lse)
    assert torch.equal(fused.o.tile_out, split.o.tile_out)
    for r in range(w.batch):
        ref = oracle_request(w, t, 0, r)
        o = fused.o
        assert_close_to_oracle(o.tile_out[0, r], o.tile_lse[0, r], o.out[0, r], o.lse[0, r],
                               ref, w.tiles[r], f"{hq}q/{hkv}kv request {r}")


def split_counts(lengths, tiles, n_kv_heads, sms, charge=6, page=64):
    """CTAs covering each (request, tile, kv head) unit when a launch's pages,
    each non-empty unit preceded by `charge` pages of bookkeeping, are cut
    into equal shares, one per CTA (the decode launch's work split; a launch
    of at least 32 pages per SM runs on 90% of the SMs; the grid is rounded
    down to a multiple of the kv-head count)."""
    units = [(s, e) for _ in range(n_kv_heads) for tl in tiles for (s, e) in tl]
    spans, total = [], 0
    for s, e in units:
        n = -(-e // page) - s // page if e > s else 0
        if n:
            total += charge
            spans.append((total, n))
        total += n
    grid = sms * 90 // 100 if total >= 32 * sms else min(sms, total)
    if grid >= n_kv_heads:
        grid -= grid % n_kv_heads
    cta = lambda p: ((p + 1) * grid - 1) // total
    return [cta(f + n - 1) - cta(f) + 1 for f, n in spans]


SPLIT_CASES = [(1, 24, 4), (2, 24, 4), (3, 24, 4), (1, 8, 1)]   # (requests, hq, hkv)


@pytest.mark.parametrize("cuda_core", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("batch,hq,hkv", SPLIT_CASES,
                         ids=[f"{b}x-{q}q{k}kv" for b, q, k in SPLIT_CASES])
def test_units_split_over_many_ctas(B, D, cuda_core, batch, hq, hkv):
    """One tile per request of a few thousand tokens spreads each (request,
    kv head) unit over 11-36 CTAs (107 with one kv head), whose partials the
    last of them merges: more than one register batch of partials, and more
    than one and more than two warps' worth of statistics.  The result must
    match the oracle, agree with the same history cut into two tiles and
    merged, and keep its bits when the pages move."""
    rng = np.random.default_rng(40 + batch)
    lengths = [int(x) for x in rng.integers(2500, 9000, size=batch)]
    one = [[(0, L)] for L in lengths]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    counts = split_counts(lengths, one, hkv, sms)
    assert max(counts) >= 13, counts
    geo = wl.Geometry(n_q_heads=hq, n_kv_heads=hkv)
    w = wl.custom(lengths, one, seed=60 + batch, n_spare=3, geometry=geo)
    t = wl.materialize(w, "cuda")
    a = run_resident(D, w, t, cuda_core)
    cut = [[(0, L // 3), (L // 3, L)] for L in lengths]
    b = run_resident(D, w, t, cuda_core, tiles=wl._pad_tiles([list(c) for c in cut]))
    for r in range(batch):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(a.o.tile_out[0, r], a.o.tile_lse[0, r], a.o.out[0, r],
                               a.o.lse[0, r], ref, w.tiles[r], f"request {r} of {batch}")
        assert max_abs(b.o.out[0, r].cpu(), a.o.tile_out[0, r, 0].cpu()) <= TOL_SPLIT
        assert max_abs(b.o.lse[0, r].cpu(), a.o.tile_lse[0, r, 0].cpu()) <= TOL_SPLIT
    # placement: reverse the physical order of the pool's pages
    perm = np.arange(w.pool_pages)[::-1].copy()
    pool2 = torch.empty_like(t["pool"])
    pool2[:, torch.as_tensor(perm, device="cuda")] = t["pool"]
    table2 = w.page_table.copy()
    for r in range(batch):
        n = w.pages_of(r)
        table2[r, :n] = perm[w.page_table[r, :n]]
    w2 = wl.DecodeWorkload(w.name, w.seed, w.n_layers, w.lengths, w.tiles, table2,
                           w.pool_pages, perm[w.spare_pages], w.geometry)
    t2 = dict(t, pool=pool2, page_table=torch.as_tensor(table2, device="cuda"))
    c = run_resident(D, w2, t2, cuda_core)
    assert torch.equal(a.o.tile_out, c.o.tile_out) and torch.equal(a.o.tile_lse, c.o.tile_lse)
    assert torch.equal(a.o.out, c.o.out) and torch.equal(a.o.lse, c.o.lse)
