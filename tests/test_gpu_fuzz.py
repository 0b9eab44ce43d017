"""Seeded random decode cases on the GPU: random request counts, lengths, tiles
(overlapping, empty, not page aligned, new token inside or outside them) and
head geometries.  The fused launch (tail write, attention, tile merge; with
and without early page loads) must equal the three-launch route bit for bit,
and every request must match the oracle."""

import numpy as np
import pytest
import torch

from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import assert_close_to_oracle, oracle_request

pytestmark = pytest.mark.gpu

GEOS = [(24, 4), (8, 8), (16, 2), (32, 4), (6, 3), (8, 1)]


@pytest.fixture(scope="module")
def D():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return decode


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    hq, hkv = GEOS[seed % len(GEOS)]
    batch = int(rng.integers(1, 7))
    lengths = [int(rng.integers(1, 3000)) for _ in range(batch)]
    tiles = []
    for L in lengths:
        t = []
        for _ in range(int(rng.integers(1, 6))):
            a = int(rng.integers(0, L + 1))
            b = int(rng.integers(a, L + 1))
            t.append((a, b))
        if rng.random() < 0.5:
            t.append((0, L))                      # one tile holds the whole history
        tiles.append(t)
    geo = wl.Geometry(n_q_heads=hq, n_kv_heads=hkv)
    return wl.custom(lengths, tiles, seed=2000 + seed, n_spare=int(rng.integers(0, 5)),
                     n_layers=1, geometry=geo)


@pytest.mark.parametrize("seed", range(12))
def test_random_cases(D, seed):
    w = random_case(seed)
    t = wl.materialize(w, "cuda")
    runs = {}
    for name, kw in (("fused", dict(fused=True)), ("early", dict(fused=True, kv_ready=True)),
                     ("three", dict(fused=False))):
        tc = {k: v.clone() for k, v in t.items()}
        dec = D.ResidentDecode(w, tc, **kw)
        torch.cuda.synchronize()
        dec.step()
        torch.cuda.synchronize()
        assert dec.kernel_status() == 0, name
        runs[name] = dec
    for name in ("fused", "early"):
        assert torch.equal(runs[name].o.tile_out, runs["three"].o.tile_out), name
        assert torch.equal(runs[name].o.tile_lse, runs["three"].o.tile_lse), name
        assert torch.equal(runs[name].o.out, runs["three"].o.out), name
        assert torch.equal(runs[name].o.lse, runs["three"].o.lse), name
    o = runs["fused"].o
    for r in range(w.batch):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(o.tile_out[0, r], o.tile_lse[0, r], o.out[0, r], o.lse[0, r], ref,
                               w.tiles[r], f"seed {seed} request {r}")


def test_sixty_four_tiles_per_request(D):
    """64 tiles per request (the merge-stress partial count): uneven, empty
    and single-token tiles cut from histories of 1 to 9,000 tokens."""
    rng = np.random.default_rng(64)
    lengths = [9000, 1, 4097]
    tiles = []
    for L in lengths:
        cuts = np.sort(rng.integers(0, L + 1, size=63))
        edges = np.concatenate([[0], cuts, [L]])
        tiles.append([(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])])
    w = wl.custom(lengths, tiles, seed=640, n_spare=3, n_layers=1)
    assert w.n_tiles == 64
    t = wl.materialize(w, "cuda")
    runs = {}
    for name, kw in (("fused", dict(fused=True)), ("three", dict(fused=False))):
        tc = {k: v.clone() for k, v in t.items()}
        dec = D.ResidentDecode(w, tc, **kw)
        torch.cuda.synchronize()
        dec.step()
        torch.cuda.synchronize()
        assert dec.kernel_status() == 0, name
        runs[name] = dec
    a, b = runs["fused"].o, runs["three"].o
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)
    assert torch.equal(a.tile_out, b.tile_out) and torch.equal(a.tile_lse, b.tile_lse)
    for r in range(w.batch):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(a.tile_out[0, r], a.tile_lse[0, r], a.out[0, r], a.lse[0, r], ref,
                               w.tiles[r], f"request {r}")


@pytest.mark.parametrize("scale", [1.0, 0.3, 0.01, 0.125])
@pytest.mark.parametrize("cuda_core", [False, True], ids=["tensor", "cuda-core"])
def test_softmax_scale_is_applied(D, scale, cuda_core):
    """Scales other than 1/16 (peakier and flatter softmaxes) match the oracle
    on both kernel variants."""
    geo = wl.Geometry(scale=scale)
    w = wl.custom([700, 2049], [[(0, 300), (300, 700)], [(0, 2049)]], seed=31, n_spare=2,
                  geometry=geo)
    t = wl.materialize(w, "cuda")
    dec = D.ResidentDecode(w, t, cuda_core=cuda_core, fused=not cuda_core)
    torch.cuda.synchronize()
    dec.step()
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    o = dec.o
    for r in range(w.batch):
        ref = oracle_request(w, t, 0, r)
        assert_close_to_oracle(o.tile_out[0, r], o.tile_lse[0, r], o.out[0, r], o.lse[0, r], ref,
                               w.tiles[r], f"scale {scale} request {r}")
