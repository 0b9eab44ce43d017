"""Failure detection on the GPU without a fault: a bounded device wait that
runs out is reported in the status word and leaves the context usable.

The test hook leaves one of CTA 0's page loads unarmed, so the consumers'
wait for that page never completes; with a 50 ms limit the kernel sets
PA_STATUS_TIMEOUT, the producer lets its issued loads land, every CTA returns,
and a following call on a fresh workspace is correct again.  No fault, trap
or endless loop is involved: every device wait in the kernel is bounded.
"""

import time

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


@pytest.mark.parametrize("iteration", [0, 2, 5])
def test_a_wait_that_runs_out_is_reported_and_the_context_survives(mods, iteration):
    B, D = mods
    # one 128,000-token tile: CTA 0's share holds ~45 real pages
    w = wl.custom([128000], [[(0, 128000)]], seed=41, n_spare=2)
    t = wl.materialize(w, "cuda")
    before = D.ResidentDecode(w, t)
    before.layer(0, attention_only=True)
    torch.cuda.synchronize()
    assert before.kernel_status() == 0
    dec = D.ResidentDecode(w, t)
    torch.cuda.synchronize()
    B.test_stall(iteration, 50_000_000)
    t0 = time.perf_counter()
    dec.layer(0, attention_only=True)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert dec.kernel_status() & B.PA_STATUS_TIMEOUT
    assert elapsed < 1.5                               # bounded by the 50 ms limit, not 2 s
    # the context is usable: a fresh decode on a fresh workspace returns the
    # same bits as the one before the stall
    after = D.ResidentDecode(w, t)
    after.layer(0, attention_only=True)
    torch.cuda.synchronize()
    assert after.kernel_status() == 0
    assert torch.equal(after.o.tile_out, before.o.tile_out)
    assert torch.equal(after.o.tile_lse, before.o.tile_lse)
