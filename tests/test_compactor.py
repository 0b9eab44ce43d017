"""Compact older pages on the host: the converter against the oracle, bit for bit.

"KV-cache engineering", sections "Exact recent pages, compact older pages" and
"What the hybrid tier buys": a page is converted only after it is fully
written in every layer, by background threads, with a CRC, and published;
until then it is served exact.  The format is this library's reading (the
pages name none), defined once in ``oracle/compact_pages.py`` and
``include/pagedattn.h``.
"""

import zlib

import numpy as np
import pytest
import torch

from oracle import compact_pages as oc

HKV, D, PT = 4, 256, 64
ROW = 2 * HKV * D


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    return binding


def bits_of(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def random_rows(rng, n, scale=1.0):
    x = torch.tensor(rng.standard_normal((n, ROW)).astype(np.float32) * scale)
    return x.to(torch.bfloat16)


def special_page(rng):
    rows = random_rows(rng, PT)
    rows[3, :D] = 0                                         # a zero slice
    rows[5, D:2 * D] = torch.tensor(np.r_[127.0, np.arange(-127, 128)[:D - 1] + 0.5],
                                    dtype=torch.float32).to(torch.bfloat16)   # halfway ratios
    rows[7, 2 * D:3 * D] *= 1e-38                          # subnormal territory
    rows[9] *= 8                                            # a scaled key row
    return rows


def test_crc32_matches_zlib(B):
    rng = np.random.default_rng(0)
    for n in (0, 1, 3, 8, 9, 1000, 133120):
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert B.crc32(data) == zlib.crc32(data)
    assert B.crc32(b"page", B.crc32(b"compact ")) == zlib.crc32(b"compact page")


@pytest.mark.parametrize("case", ["normal", "special", "large"])
def test_convert_page_matches_oracle(B, case):
    rng = np.random.default_rng({"normal": 1, "special": 2, "large": 3}[case])
    rows = {"normal": lambda: random_rows(rng, PT), "special": lambda: special_page(rng),
            "large": lambda: random_rows(rng, PT, 3e4)}[case]()
    data, crc = B.compact_convert_page(rows, HKV, D)
    ref = oc.convert_page(bits_of(rows), HKV, D)
    assert len(data) == B.compact_page_bytes(HKV, D) == len(ref["bytes"])
    assert data == ref["bytes"]
    assert crc == ref["crc"] == zlib.crc32(data)


def test_non_finite_page_is_not_convertible(B):
    rows = random_rows(np.random.default_rng(4), PT)
    rows[10, 77] = float("nan")
    with pytest.raises(B.PagedAttnError) as e:
        B.compact_convert_page(rows, HKV, D)
    assert e.value.code == B.PA_ERR_INVALID


class History:
    """Host exact history [layers][requests] segments and a compact store."""

    def __init__(self, B, lengths, n_layers=2, max_pages=None, seed=5):
        rng = np.random.default_rng(seed)
        self.lengths = lengths
        self.max_pages = max_pages or max(-(-L // PT) for L in lengths)
        self.rows = [[random_rows(rng, L) for L in lengths] for _ in range(n_layers)]
        cp = B.compact_page_bytes(HKV, D)
        self.cp = cp
        self.store = [[torch.zeros(self.max_pages * cp, dtype=torch.uint8) for _ in lengths]
                      for _ in range(n_layers)]
        exact = [self.rows[l][r].data_ptr() for l in range(n_layers) for r in range(len(lengths))]
        comp = [self.store[l][r].data_ptr() for l in range(n_layers) for r in range(len(lengths))]
        self.n_layers = n_layers

        def make(threads=3):
            return B.Compactor(n_layers, len(lengths), HKV, D, self.max_pages, exact, comp,
                               n_threads=threads)
        self.make = make

    def compact_bytes(self, l, r, p):
        return self.store[l][r][p * self.cp:(p + 1) * self.cp].numpy().tobytes()

    def oracle_page(self, l, r, p):
        return oc.convert_page(bits_of(self.rows[l][r][p * PT:(p + 1) * PT]), HKV, D)


def test_background_conversion_publishes_exact_oracle_bytes(B):
    h = History(B, [640, 200, 64 * 3 + 5])
    c = h.make()
    full = [L // PT for L in h.lengths]
    for r, f in enumerate(full):
        c.mark_written(r, f)
    c.wait_idle()
    for r, f in enumerate(full):
        st = c.states(r)
        assert st[:f] == [B.PA_PAGE_PUBLISHED] * f
        assert all(s == B.PA_PAGE_EXACT for s in st[f:])       # the partial page stays exact
        for p in range(f):
            c.verify(r, p)
            for l in range(h.n_layers):
                ref = h.oracle_page(l, r, p)
                assert h.compact_bytes(l, r, p) == ref["bytes"]
                assert c.crc(l, r, p) == ref["crc"]
    cnt = c.counters()
    assert cnt["published_pages"] == sum(full) and cnt["queued_pages"] == 0
    assert cnt["compact_bytes"] == sum(full) * h.n_layers * h.cp
    c.close()


def test_served_exact_until_published(B):
    h = History(B, [640])
    c = h.make()
    c.hold(True)
    c.mark_written(0, 10)
    assert c.states(0)[:10] == [B.PA_PAGE_QUEUED] * 10
    with pytest.raises(B.PagedAttnError) as e:
        c.crc(0, 0, 0)
    assert e.value.code == B.PA_ERR_ORDER
    with pytest.raises(B.PagedAttnError) as e:
        c.wait_idle(50)
    assert e.value.code == B.PA_ERR_ORDER                        # held with pages queued
    c.hold(False)
    c.wait_idle()
    assert c.states(0) == [B.PA_PAGE_PUBLISHED] * 10
    c.close()


def test_only_new_pages_are_queued_and_marking_is_monotone(B):
    h = History(B, [64 * 8])
    c = h.make(threads=1)
    c.mark_written(0, 3)
    c.wait_idle()
    c.mark_written(0, 2)                                         # nothing new
    c.mark_written(0, 5)                                         # pages 3, 4 only
    c.wait_idle()
    assert c.states(0) == [B.PA_PAGE_PUBLISHED] * 5 + [B.PA_PAGE_EXACT] * 3
    assert c.counters()["published_pages"] == 5
    with pytest.raises(B.PagedAttnError):
        c.mark_written(0, 9)                                     # beyond max_pages
    c.close()


def test_non_finite_page_in_any_layer_stays_exact(B):
    h = History(B, [64 * 4])
    h.rows[1][0][64 + 17, 3] = float("inf")                      # layer 1, page 1
    c = h.make()
    c.mark_written(0, 4)
    c.wait_idle()
    assert c.states(0) == [B.PA_PAGE_PUBLISHED, B.PA_PAGE_NOT_CONVERTIBLE,
                           B.PA_PAGE_PUBLISHED, B.PA_PAGE_PUBLISHED]
    assert c.counters()["not_convertible_pages"] == 1
    c.close()


def test_corruption_is_caught_by_the_crc(B):
    h = History(B, [64 * 2])
    c = h.make()
    c.mark_written(0, 2)
    c.wait_idle()
    c.verify(0, 1)
    h.store[1][0][h.cp + 1000] ^= 1                             # flip a bit of layer 1, page 1
    with pytest.raises(B.PagedAttnError) as e:
        c.verify(0, 1)
    assert e.value.code == B.PA_ERR_CRC
    c.verify(0, 0)
    c.close()


def test_thread_count_does_not_change_the_bytes(B):
    outs = []
    for threads in (1, 8):
        h = History(B, [64 * 12, 64 * 7 + 3], seed=9)
        c = h.make(threads=threads)
        for r, L in enumerate(h.lengths):
            c.mark_written(r, L // PT)
        c.wait_idle()
        outs.append([h.store[l][r].numpy().tobytes() for l in range(2) for r in range(2)])
        c.close()
    assert outs[0] == outs[1]


def test_hold_during_conversion_ends_an_idle_wait_promptly(B):
    # one converter thread, many queued pages: holding it while a page is in
    # progress leaves the rest queued, and a waiter for idleness returns as
    # soon as that page is done (held counts as idle) instead of at its timeout
    import time
    h = History(B, [64 * 40], n_layers=32)     # ~tens of ms per page (32 layers each)
    c = h.make(threads=1)
    c.mark_written(0, 40)
    time.sleep(0.005)                            # the thread is inside its first page
    c.hold(True)
    t0 = time.perf_counter()
    with pytest.raises(B.PagedAttnError) as e:
        c.wait_idle(20000)
    assert e.value.code == B.PA_ERR_ORDER
    assert time.perf_counter() - t0 < 5.0
    st = c.states(0)
    assert B.PA_PAGE_QUEUED in st                       # the hold stopped the queue
    c.hold(False)
    c.wait_idle()
    assert c.states(0) == [B.PA_PAGE_PUBLISHED] * 40
    c.close()
