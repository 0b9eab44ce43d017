"""The decode kernel's split-unit merge on the GPU, both ways it can run.

A unit (tile, kv head) split over several CTAs is merged in slices of its
output by the unit's own CTAs once the last one has arrived; a CTA that sees
no arrival for a while leaves its slice to the last CTA instead (the path a
grid that is not resident all at once takes).  A test hook shortens that wait
to zero, so most waiting CTAs leave at once: the outputs must be the same
bits as with the normal wait, the leavers must be counted in the workspace's
diagnostic word, and the workspace must be left ready for the next call.
"""

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


def leavers(dec):
    return int(dec.workspace[4:8].view(torch.int32).item())


CASES = {
    # one tile: each of the 4 units spans ~38 CTAs (16 merge slices)
    "1x32768": lambda: wl.uniform(1, 32768, n_layers=2),
    # several tiles per request, merged inside the launch (slices count toward
    # the per-(request, kv head) tile count)
    "tiles": lambda: wl.custom([70000, 5000], [[(0, 32768), (32768, 65536), (65536, 70000)],
                                               [(0, 2000), (2000, 5000)]], seed=23, n_layers=2),
    # ~10 CTAs per unit
    "4x8192": lambda: wl.uniform(4, 8192, n_layers=2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_leaving_the_merge_to_the_last_cta_gives_the_same_bits(mods, name):
    B, D = mods
    w = CASES[name]()
    t = wl.materialize(w, "cuda")
    ref = D.ResidentDecode(w, {k: v.clone() for k, v in t.items()})
    ref.step()
    torch.cuda.synchronize()
    assert ref.kernel_status() == 0 and leavers(ref) == 0
    dec = D.ResidentDecode(w, {k: v.clone() for k, v in t.items()})
    for i in range(w.n_layers):
        B.test_slice_wait(0)
        dec.layer(i)
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    assert leavers(dec) > 0
    for a, b in ((dec.o.tile_out, ref.o.tile_out), (dec.o.tile_lse, ref.o.tile_lse),
                 (dec.o.out, ref.o.out), (dec.o.lse, ref.o.lse)):
        assert torch.equal(a, b)
    # the same workspace is ready for the next call: a normal step on it
    # gives the same bits again (the tail rows it stores are the same rows)
    n0 = leavers(dec)
    dec.step()
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    assert torch.equal(dec.o.out, ref.o.out) and torch.equal(dec.o.lse, ref.o.lse)
    assert torch.equal(dec.o.tile_out, ref.o.tile_out)
    assert leavers(dec) - n0 >= 0


def test_split_units_match_the_oracle_when_merged_by_the_last_cta(mods):
    """The slices merged only by the last CTA still agree with the fp64 oracle."""
    from parity_utils import assert_close_to_oracle, oracle_request
    B, D = mods
    w = wl.uniform(1, 32768, n_layers=1)
    t = wl.materialize(w, "cuda")
    dec = D.ResidentDecode(w, t)
    B.test_slice_wait(0)
    dec.layer(0)
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0 and leavers(dec) > 0
    ref = oracle_request(w, t, 0, 0, gather_on_device=True)
    assert_close_to_oracle(dec.o.tile_out[0, 0], dec.o.tile_lse[0, 0], dec.o.out[0, 0],
                           dec.o.lse[0, 0], ref, w.tiles[0], "1x32768 leavers")


@pytest.mark.parametrize("leave", [False, True], ids=["merged-by-slices", "left-to-last-cta"])
def test_one_unit_split_over_every_cta(mods, leave):
    """One kv head, eight query heads, one 131,072-token tile: the single unit
    spans every CTA of the grid (as many partials as a split unit can have),
    merged in slices or by the last CTA alone, against the fp64 oracle."""
    from parity_utils import assert_close_to_oracle, oracle_request
    B, D = mods
    geo = wl.Geometry(n_q_heads=8, n_kv_heads=1)
    w = wl.custom([131072], [[(0, 131072)]], seed=29, n_layers=1, geometry=geo)
    t = wl.materialize(w, "cuda")
    dec = D.ResidentDecode(w, t)
    if leave:
        B.test_slice_wait(0)
    dec.layer(0)
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    assert (leavers(dec) > 0) == leave
    ref = oracle_request(w, t, 0, 0, gather_on_device=True)
    assert_close_to_oracle(dec.o.tile_out[0, 0], dec.o.tile_lse[0, 0], dec.o.out[0, 0],
                           dec.o.lse[0, 0], ref, w.tiles[0], "1 kv head x 131072")
