"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (one attention launch per layer, persistent grid of one CTA per
SM), and bit-identity of the host-staged route against the resident route.

The oracle checks sampled (layer, request) pairs one by one; properties that
hold at any size (finite outputs, status word clear, tiled+merged equal to the
single-tile result within 1e-5, staged equal to resident bit for bit, tail
write-back equal to the new row bit for bit) are checked on every output.
"""

import gc

import numpy as np
import pytest
import torch

from paged_decode_attention_attn_gb300 import workloads as wl
from parity_utils import TOL_SPLIT, assert_close_to_oracle, max_abs, oracle_request

pytestmark = pytest.mark.gpu

FULL = {
    "4x31744": (wl.four_requests_31744, [(0, 1), (15, 3)]),
    "1x262144": (wl.one_request_262144, [(7, 0), (15, 0)]),
    "ragged-window": (wl.ragged_window, [(3, "longest"), (12, "shortest")]),
    "1x32768": (lambda n_layers=16: wl.uniform(1, 32768, 32768, n_layers=n_layers),
                [(0, 0), (9, 0)]),
}


@pytest.fixture(scope="module")
def D():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import decode
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return decode


def _free():
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_resident_matches_oracle(D, name):
    make, samples = FULL[name]
    w = make()
    t = wl.materialize(w, "cuda")
    dec = D.ResidentDecode(w, t)
    dec.step()
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    o = dec.o
    real = torch.as_tensor(w.tiles[:, :, 1] > w.tiles[:, :, 0], device="cuda")
    assert torch.isfinite(o.out).all() and torch.isfinite(o.lse).all()
    assert torch.isfinite(o.tile_out[:, real]).all()
    for i, r in samples:
        if r == "longest":
            r = int(np.argmax(w.lengths))
        elif r == "shortest":
            r = int(np.argmin(w.lengths))
        ref = oracle_request(w, t, i, r, gather_on_device=True)
        assert_close_to_oracle(o.tile_out[i, r], o.tile_lse[i, r], o.out[i, r], o.lse[i, r], ref,
                               w.tiles[r], f"{name} layer {i} request {r}")
    if w.n_tiles > 1:
        single = np.zeros((w.batch, 1, 2), dtype=np.int32)
        single[:, 0, 1] = w.lengths
        one = D.ResidentDecode(w, t, tiles=single)
        for i in range(w.n_layers):
            one.layer(i, attention_only=True)
        torch.cuda.synchronize()
        assert max_abs(one.o.tile_out[:, :, 0].cpu(), o.out.cpu()) <= TOL_SPLIT
        assert max_abs(one.o.tile_lse[:, :, 0].cpu(), o.lse.cpu()) <= TOL_SPLIT
        del one
    del dec, t, o
    _free()


@pytest.mark.parametrize("name,n_slots,leases", [("4x31744", 2, False), ("4x31744", 1, False),
                                                 ("1x262144", 2, False),
                                                 ("ragged-window", 2, False),
                                                 ("4x31744", 2, True), ("ragged-window", 1, True)])
def test_staged_route_is_bit_identical_to_resident(D, name, n_slots, leases):
    make, _ = FULL[name]
    w = make(n_layers=3)
    t = wl.materialize(w, "cuda")
    host = D.HostHistory(w, t)
    staged = D.StagedDecode(w, t, host, n_slots=n_slots, leases=leases)
    res = D.ResidentDecode(w, t)
    res.step()
    torch.cuda.synchronize()
    staged.step()
    staged.drain()
    torch.cuda.synchronize()
    assert res.kernel_status() == 0 and staged.kernel_status() == 0
    assert torch.equal(staged.o.tile_out, res.o.tile_out)
    assert torch.equal(staged.o.tile_lse, res.o.tile_lse)
    assert torch.equal(staged.o.out, res.o.out)
    assert torch.equal(staged.o.lse, res.o.lse)
    for i in range(w.n_layers):
        for r in range(w.batch):
            row = host.row(i, r, int(w.lengths[r]) - 1)
            assert torch.equal(row.view(torch.int16), t["new_rows"][i, r].cpu().view(torch.int16))
    st = staged.handle.stats()
    assert st.stage_generation == w.n_layers and st.quarantined == 0
    assert st.written_back_bytes == w.n_layers * w.batch * w.geometry.row_bytes
    # the resident window came from the pinned host rows: the sink page and
    # the newest pages up to (not including) the new token's row
    window_rows = 0
    if w.window:
        sink, recent = w.window
        for r in range(w.batch):
            n, L = w.pages_of(r), int(w.lengths[r])
            if n > sink + recent:
                window_rows += sink * 64 + (L - 1) - (n - recent) * 64
    assert st.loaded_bytes == w.n_layers * window_rows * w.geometry.row_bytes
    if leases:
        assert [r.layer for r in staged.receipts] == list(range(w.n_layers))
        assert sum(r.staged_bytes for r in staged.receipts) == st.staged_bytes
        assert all(r.written_back_bytes == w.batch * w.geometry.row_bytes
                   for r in staged.receipts)
        for r in range(w.batch):
            assert staged.handle.host_generation((0 << 32) | r)[1] == 0   # tickets released
    staged.close()
    host.close()
    del staged, res, host, t
    _free()


@pytest.mark.parametrize("make", [lambda: wl.one_request_262144(n_layers=2),
                                  lambda: wl.four_requests_31744(n_layers=2),
                                  lambda: wl.custom([5000, 70000], [[(0, 2000), (2000, 5000)],
                                                                   [(0, 32768), (32768, 65536),
                                                                    (65536, 70000)]],
                                                    seed=19, n_layers=2)],
                         ids=["1x262144", "4x31744", "uneven-tiles"])
def test_tile_staged_route_is_bit_identical_to_resident_tile_launches(D, make):
    """Staging per 32K-token tile into two tile slots gives the bits of the
    resident route with the same per-tile launches, writes every new row back
    exactly, and keeps the arena at two tiles."""
    w = make()
    t = wl.materialize(w, "cuda")
    host = D.HostHistory(w, t)
    staged = D.TiledStagedDecode(w, t, host, n_slots=2)
    staged.step()
    staged.drain()
    torch.cuda.synchronize()
    ref = D._Outputs(w, w.n_layers, "cuda")
    geo = w.geometry
    ws = D.B.alloc_workspace(1, 1, geo.n_q_heads, geo.n_kv_heads, geo.head_dim)
    D.resident_tiled_step(w, t, ref, ws)
    torch.cuda.synchronize()
    assert int(staged.workspace[:4].view(torch.int32).item()) == 0
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert torch.equal(staged.o.tile_out, ref.tile_out)
    assert torch.equal(staged.o.tile_lse, ref.tile_lse)
    assert torch.equal(staged.o.out, ref.out) and torch.equal(staged.o.lse, ref.lse)
    for i in range(w.n_layers):
        for r in range(w.batch):
            row = host.row(i, r, int(w.lengths[r]) - 1)
            assert torch.equal(row.view(torch.int16), t["new_rows"][i, r].cpu().view(torch.int16))
    # and the tiled results agree with the one-launch-per-layer route to rounding
    res = D.ResidentDecode(w, t)
    res.step()
    torch.cuda.synchronize()
    assert max_abs(staged.o.out.cpu(), res.o.out.cpu()) <= TOL_SPLIT
    assert staged.arena_bytes() <= 2 * 512 * 64 * geo.row_bytes     # two 32K-token tiles
    staged.close()
    host.close()
    del staged, host, t, res
    _free()


def test_bench_launch_configuration_matches_oracle(D):
    """The bench's configuration (fused launches with early page loads,
    replayed as a CUDA graph) returns the eager route's bits at full size,
    and sampled (layer, request) pairs match the oracle."""
    w = wl.four_requests_31744(n_layers=4)
    t = wl.materialize(w, "cuda")
    eager = D.ResidentDecode(w, {k: v.clone() for k, v in t.items()})
    torch.cuda.synchronize()
    eager.step()
    torch.cuda.synchronize()
    dec = D.ResidentDecode(w, t, kv_ready=True)
    torch.cuda.synchronize()
    dec.step()                                   # warm-up (also stores the new rows)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    dec.stream = cap
    with torch.cuda.graph(graph, stream=cap):
        dec.step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert dec.kernel_status() == 0
    assert torch.equal(dec.o.out, eager.o.out) and torch.equal(dec.o.lse, eager.o.lse)
    for i, r in [(0, 0), (3, 2)]:
        ref = oracle_request(w, t, i, r, gather_on_device=True)
        o = dec.o
        assert_close_to_oracle(o.tile_out[i, r], o.tile_lse[i, r], o.out[i, r], o.lse[i, r], ref,
                               w.tiles[r], f"graph layer {i} request {r}")
    del dec, eager, graph, t
    _free()


@pytest.mark.parametrize("n_slots", [1, 2])
def test_staged_route_over_many_steps(D, n_slots):
    """Eight consecutive steps of the staged route, with no host wait between
    them (slots refilled while earlier layers' attention and write-back may
    still run): every step's outputs equal the resident route's bit for bit."""
    make, _ = FULL["4x31744"]
    w = make(n_layers=3)
    t = wl.materialize(w, "cuda")
    host = D.HostHistory(w, t)
    staged = D.StagedDecode(w, t, host, n_slots=n_slots)
    res = D.ResidentDecode(w, t)
    res.step()
    torch.cuda.synchronize()
    outs = []
    for _ in range(8):
        staged.step()
        outs.append(tuple(x.clone() for x in (staged.o.tile_out, staged.o.tile_lse,
                                              staged.o.out, staged.o.lse)))
    staged.drain()
    torch.cuda.synchronize()
    assert res.kernel_status() == 0 and staged.kernel_status() == 0
    ref = (res.o.tile_out, res.o.tile_lse, res.o.out, res.o.lse)
    for k, o in enumerate(outs):
        assert all(torch.equal(a, b) for a, b in zip(o, ref)), f"step {k}"
    st = staged.handle.stats()
    assert st.stage_generation == 8 * w.n_layers and st.quarantined == 0
    staged.close()
    host.close()
    del staged, res, host, t
    _free()
