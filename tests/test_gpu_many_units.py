"""Calls with more (tile, kv head) units than one launch takes (1,024): the
library cuts them into several launches that share the workspace, and a
(request, kv head) pair's tiles can fall into two launches, so the fused
tile merge's count must span both.  Checked against the three-launch route
bit for bit, against the oracle on sampled requests, and for the merge
slices' leave path."""

import numpy as np
import pytest
import torch

from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import assert_close_to_oracle, oracle_request

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding, decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding, decode


def many_units(seed=31):
    """64 requests x 5 tiles x 4 kv heads = 1,280 units (two launches); lengths
    2,000-12,000 tokens, so long tiles split over several CTAs; uneven tiles,
    one empty."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(2000, 12001, size=64).tolist()
    tiles = []
    for L in lengths:
        cuts = sorted(rng.integers(1, L, size=4).tolist())
        t_req = [(0, cuts[0])] + [(a, b) for a, b in zip(cuts, cuts[1:])] + [(cuts[-1], L)]
        tiles.append(t_req)
    tiles[7][2] = (tiles[7][2][0], tiles[7][2][0])      # an empty tile
    return wl.custom(lengths, tiles, seed=seed, n_layers=1)


def clone(t):
    return {k: v.clone() for k, v in t.items()}


def test_two_launch_call_matches_three_launch_route_and_oracle(mods):
    B, D = mods
    w = many_units()
    assert w.batch * w.n_tiles * w.geometry.n_kv_heads > 1024
    t = wl.materialize(w, "cuda")
    tf, tu = clone(t), clone(t)
    fused = D.ResidentDecode(w, tf, fused=True)
    unfused = D.ResidentDecode(w, tu, fused=False)
    torch.cuda.synchronize()
    for _ in range(2):           # twice: the counters are left ready for the next call
        fused.step()
        unfused.step()
        torch.cuda.synchronize()
        assert fused.kernel_status() == 0 and unfused.kernel_status() == 0
        assert torch.equal(fused.o.tile_out, unfused.o.tile_out)
        assert torch.equal(fused.o.tile_lse, unfused.o.tile_lse)
        assert torch.equal(fused.o.out, unfused.o.out)
        assert torch.equal(fused.o.lse, unfused.o.lse)
    # requests whose kv head 3 tiles straddle the two launches (units
    # 960 + 5 b + tile: b = 12 holds units 1020..1024) and a few others
    for r in (0, 7, 12, 13, 63):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(fused.o.tile_out[0, r], fused.o.tile_lse[0, r], fused.o.out[0, r],
                               fused.o.lse[0, r], ref, w.tiles[r], f"request {r}")


def test_two_launch_call_with_merge_slices_left_to_the_last_cta(mods):
    B, D = mods
    w = many_units(seed=32)
    t = wl.materialize(w, "cuda")
    ref = D.ResidentDecode(w, clone(t))
    ref.step()
    dec = D.ResidentDecode(w, clone(t))
    B.test_slice_wait(0)
    dec.layer(0)
    torch.cuda.synchronize()
    assert ref.kernel_status() == 0 and dec.kernel_status() == 0
    assert torch.equal(dec.o.out, ref.o.out) and torch.equal(dec.o.lse, ref.o.lse)
    assert torch.equal(dec.o.tile_out, ref.o.tile_out)
