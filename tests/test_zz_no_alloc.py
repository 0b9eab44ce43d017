"""The decode entry point that allocates nothing, against the regular one.

Some callers fix their device-memory budget before serving and forbid any
allocation afterwards, or cannot afford cudaMalloc's possible device-wide
synchronisation in their hot loop; ``paged_decode_attn_lse_noalloc`` serves
them from a fixed scratch array inside the library instead of a caller
workspace.  This file is named to be collected last, so that a failure here
does not hide any other test in a run that stops at the first failure.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import assert_close_to_oracle, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding


def _run_regular(B, w, t, tiles):
    geo = w.geometry
    T = tiles.shape[1]
    out = torch.empty((w.batch, T, geo.n_q_heads, geo.head_dim), device="cuda")
    lse = torch.empty((w.batch, T, geo.n_q_heads), device="cuda")
    ws = B.alloc_workspace(w.batch, T, geo.n_q_heads, geo.n_kv_heads, geo.head_dim)
    B.paged_decode_attn_lse(t["q"][0], t["pool"][0], t["page_table"], tiles, geo.scale, out,
                            lse, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    return out, lse


def _run_noalloc(B, w, t, tiles):
    geo = w.geometry
    T = tiles.shape[1]
    out = torch.full((w.batch, T, geo.n_q_heads, geo.head_dim), float("nan"), device="cuda")
    lse = torch.full((w.batch, T, geo.n_q_heads), float("nan"), device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.paged_decode_attn_lse_noalloc(t["q"][0], t["pool"][0], t["page_table"], tiles, geo.scale,
                                    out, lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


@pytest.mark.parametrize("case", ["ragged-tiles", "4x31744-one-layer"])
def test_noalloc_matches_regular_entry_point_twice_in_a_row(B, case):
    if case == "ragged-tiles":
        w = wl.custom([1, 700, 4097, 150], [[(0, 1)], [(0, 700), (5, 333)],
                                            [(0, 4097), (63, 2049), (4096, 4097)],
                                            [(37, 101), (0, 0)]], seed=17, n_spare=3)
    else:
        w = wl.four_requests_31744(n_layers=1)
    t = wl.materialize(w, "cuda")
    tiles = np.ascontiguousarray(w.tiles, dtype=np.int32)
    ref_out, ref_lse = _run_regular(B, w, t, tiles)
    for _ in range(2):      # the scratch array keeps the previous call's contents
        out, lse = _run_noalloc(B, w, t, tiles)
        # Same kernel, same inputs, same split of the work over the CTAs: the
        # two entry points must agree bit for bit.  Any difference would be
        # state left over in the shared scratch array.
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
    if case == "ragged-tiles":
        # and one request straight against the fp64 oracle (the pool row of
        # the last token is the one attended: no new row is substituted)
        geo = w.geometry
        r = 2
        ref = oracle.decode_layer(bits(t["q"][0, r]), bits(t["pool"][0]), w.page_table[r],
                                  int(w.lengths[r]), w.tiles[r], geo.scale, geo.n_kv_heads,
                                  geo.head_dim)
        assert_close_to_oracle(out[r], lse[r], None, None, ref, w.tiles[r], "noalloc")


def test_noalloc_refuses_more_scratch_than_it_holds(B):
    # 300 requests x 4 tiles x 4 kv heads = 4,800 units: more partial slots than
    # the fixed scratch array holds.  Refused on the host, before any launch.
    n_req, n_tiles = 300, 4
    tiles = np.zeros((n_req, n_tiles, 2), dtype=np.int32)
    tiles[:, :, 1] = 64
    q = torch.zeros((n_req, 24, 256), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, 64, 2048), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((n_req, 1), dtype=torch.int32, device="cuda")
    out = torch.zeros((n_req, n_tiles, 24, 256), device="cuda")
    lse = torch.zeros((n_req, n_tiles, 24), device="cuda")
    with pytest.raises(B.PagedAttnError) as e:
        B.paged_decode_attn_lse_noalloc(q, pool, table, tiles, 0.0625, out, lse)
    assert e.value.code == B.PA_ERR_INVALID
    assert "scratch" in str(e.value)
