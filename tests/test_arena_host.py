"""Host-side tests of the staging arena's ordering, refusal and quarantine rules.

The arena runs in record-only mode: every CUDA submission it would make is
appended to a log instead, so the device-side ordering rules of "Staging
without a stall" (sections "Two copy queues and device-side ordering" and
"Leases instead of buffers") can be checked without a GPU:
  * the compute stream waits on the copy event of the layer's stage;
  * a slot is refilled only after waits on its previous attention and
    write-back events, issued on the H2D stream before the copy;
  * write-back waits on the attention event and goes only to the staged owner;
  * a failed submission quarantines the arena until a drain succeeds.
"""

import pytest

PAGE = 64
ROW = 4096
BASE = 1 << 32
TABLES = 1 << 33


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    return binding


def make_arena(B, n_slots=2, slot_pages=8, window_pages=4, max_requests=4, max_pages=16,
               device_pages=None):
    pages = device_pages if device_pages is not None else window_pages + n_slots * slot_pages
    return B.Arena(BASE, pages * PAGE * ROW, ROW, n_slots, window_pages, slot_pages, TABLES,
                   max_requests, max_pages, compute_stream=1, h2d_stream=2, d2h_stream=3,
                   record_only=True)


def staged(lp, n, host, rows=None):
    return dict(logical_page=lp, n_pages=n, n_rows=n * PAGE if rows is None else rows,
                host_rows=host)


def resident(lp, n, page):
    return dict(logical_page=lp, n_pages=n, resident_page=page)


def full_layer(B, a, layer, reqs, tails):
    a.stage_layer(layer, reqs)
    a.mark_attention_done(layer)
    a.writeback_tail(layer, tails)


def test_first_stage_orders_compute_after_copy(B):
    a = make_arena(B)
    slot, table = a.stage_layer(0, [(0, 7, [staged(0, 3, 0x1000, rows=150)]),
                                    (2, 9, [staged(0, 2, 0x9000)])])
    assert slot == 0 and table == TABLES
    log = a.call_log()
    assert log == [
        "h2d copy h2d bytes=614400 page=4 row=0",
        "h2d copy h2d bytes=524288 page=7 row=0",
        "h2d table slot=0 runs=2 0:0+3->4 2:0+2->7",
        "h2d record copy[0]",
        "compute wait copy[0]",
    ]


def test_slot_reuse_waits_on_previous_readers_before_copy(B):
    a = make_arena(B, n_slots=2)
    req = lambda host: [(0, 1, [staged(0, 2, host, rows=100)])]
    tail = [(0, 99, 0x5000, 1)]
    full_layer(B, a, 0, req(0x1000), tail)
    full_layer(B, a, 1, req(0x2000), tail)
    n_before = len(a.call_log())
    slot, table = a.stage_layer(2, req(0x3000))
    assert slot == 0 and table == TABLES
    log = a.call_log()[n_before:]
    assert log[0] == "h2d wait attn[0]"
    assert log[1] == "h2d wait wb[0]"
    assert log[2].startswith("h2d copy h2d")
    assert a.stats().slot_reuses == 1
    # slot 1 is next; its readers are waited on too
    a.mark_attention_done(2)
    n_before = len(a.call_log())
    a.stage_layer(3, req(0x4000))
    log = a.call_log()[n_before:]
    assert log[:2] == ["h2d wait attn[1]", "h2d wait wb[1]"]


def test_reuse_without_writeback_waits_only_on_attention(B):
    a = make_arena(B, n_slots=1)
    a.stage_layer(0, [(0, 1, [staged(0, 1, 0x1000)])])
    a.mark_attention_done(0)
    n_before = len(a.call_log())
    a.stage_layer(1, [(0, 1, [staged(0, 1, 0x2000)])])
    log = a.call_log()[n_before:]
    assert log[0] == "h2d wait attn[0]"
    assert not any("wait wb" in line for line in log)


def test_stage_refused_while_slot_awaits_attention(B):
    a = make_arena(B, n_slots=1)
    a.stage_layer(0, [(0, 1, [staged(0, 1, 0x1000)])])
    n = len(a.call_log())
    with pytest.raises(B.PagedAttnError) as e:
        a.stage_layer(1, [(0, 1, [staged(0, 1, 0x2000)])])
    assert e.value.code == B.PA_ERR_ORDER
    assert len(a.call_log()) == n          # nothing submitted


def test_writeback_requires_attention_and_the_staged_owner(B):
    a = make_arena(B)
    a.stage_layer(0, [(1, 42, [staged(0, 2, 0x1000)])])
    with pytest.raises(B.PagedAttnError) as e:
        a.writeback_tail(0, [(1, 5, 0x7000, 42)])
    assert e.value.code == B.PA_ERR_ORDER
    a.mark_attention_done(0)
    n = len(a.call_log())
    with pytest.raises(B.PagedAttnError) as e:
        a.writeback_tail(0, [(1, 5, 0x7000, 43)])
    assert e.value.code == B.PA_ERR_OWNER
    assert len(a.call_log()) == n          # nothing submitted for a refused owner
    a.writeback_tail(0, [(1, 70, 0x7000, 42)])
    log = a.call_log()[n:]
    # row 70 = logical page 1, row 6 -> slot 0's second page (window 4 + 1)
    assert log == ["d2h wait attn[0]", "d2h copy d2h bytes=4096 page=5 row=6",
                   "d2h record wb[0]"]


def test_resident_window_runs_map_to_their_pages(B):
    a = make_arena(B, window_pages=4, max_pages=16)
    runs = [resident(0, 1, 0), staged(1, 5, 0x1000), resident(6, 3, 1)]
    a.stage_layer(3, [(0, 5, runs)])
    log = a.call_log()
    assert log[0] == "h2d copy h2d bytes=1310720 page=4 row=0"
    assert log[1] == "h2d table slot=0 runs=3 0:0+1->0 0:1+5->4 0:6+3->1"
    a.mark_attention_done(3)
    n = len(a.call_log())
    a.writeback_tail(3, [(0, 8 * PAGE + 17, 0x8000, 5)])   # page 8 is resident page 1 + 2
    assert a.call_log()[n + 1] == "d2h copy d2h bytes=4096 page=3 row=17"


def test_generation_is_strictly_increasing(B):
    a = make_arena(B, n_slots=2)
    gens = []
    for layer in range(5):
        a.stage_layer(layer, [(0, 1, [staged(0, 1, 0x1000)])])
        gens.append(a.stats().stage_generation)
        a.mark_attention_done(layer)
    assert gens == [1, 2, 3, 4, 5]


@pytest.mark.parametrize("fail_at", range(0, 9))
def test_injected_failure_quarantines_until_drain(B, fail_at):
    a = make_arena(B, n_slots=2)
    a.fail_after(fail_at)
    codes = []
    for layer in range(3):
        for call in (lambda: a.stage_layer(layer, [(0, 1, [staged(0, 1, 0x1000)])]),
                     lambda: a.mark_attention_done(layer),
                     lambda: a.writeback_tail(layer, [(0, 3, 0x2000, 1)])):
            try:
                call()
                codes.append(0)
            except B.PagedAttnError as e:
                codes.append(e.code)
    assert B.PA_ERR_CUDA in codes
    first = codes.index(B.PA_ERR_CUDA)
    assert all(c == 0 for c in codes[:first])
    assert all(c == B.PA_ERR_QUARANTINED for c in codes[first + 1:])
    assert a.stats().quarantined == 1
    a.drain()
    assert a.stats().quarantined == 0
    slot, _ = a.stage_layer(7, [(0, 1, [staged(0, 1, 0x1000)])])   # usable again
    assert "drain" in a.call_log()


def test_failed_drain_keeps_quarantine(B):
    a = make_arena(B)
    a.fail_after(0)
    with pytest.raises(B.PagedAttnError):
        a.stage_layer(0, [(0, 1, [staged(0, 1, 0x1000)])])
    a.fail_after(0)
    with pytest.raises(B.PagedAttnError) as e:
        a.drain()
    assert e.value.code == B.PA_ERR_CUDA
    assert a.stats().quarantined == 1
    with pytest.raises(B.PagedAttnError) as e:
        a.mark_attention_done(0)
    assert e.value.code == B.PA_ERR_QUARANTINED


def test_validation(B):
    with pytest.raises(B.PagedAttnError):
        make_arena(B, device_pages=10)          # 4 + 2*8 pages do not fit in 10
    a = make_arena(B)
    bad = [
        [(0, 1, [staged(15, 2, 0x1000)])],                      # past max_pages
        [(0, 1, [staged(0, 9, 0x1000)])],                       # more pages than a slot
        [(0, 1, [staged(0, 1, 0x1000, rows=65)])],              # rows do not fit the run
        [(4, 1, [staged(0, 1, 0x1000)])],                       # request >= max_requests
        [(0, 1, [staged(0, 1, 0x1000)]), (0, 2, [staged(1, 1, 0x2000)])],  # request twice
        [(0, 1, [resident(0, 2, 19)])],                         # resident past the arena
        [(0, 1, [resident(0, 2, 3)])],                          # resident into slot 0
        [(0, 1, [resident(0, 1, 12)])],                         # resident inside slot 1
    ]
    for reqs in bad:
        with pytest.raises(B.PagedAttnError) as e:
            a.stage_layer(0, reqs)
        assert e.value.code == B.PA_ERR_INVALID
    assert a.call_log() == []
    assert a.stats().stage_generation == 0


CPAGE = 133120          # compact page bytes at 4 kv heads x 256


def compact(lp, n, host):
    return dict(logical_page=lp, n_pages=n, n_rows=n * PAGE, host_compact=host)


def make_compact_arena(B, n_slots=2, slot_pages=8, window_pages=4, landing_pages=4):
    page_end = (window_pages + n_slots * slot_pages) * PAGE * ROW
    landing = landing_pages * CPAGE
    return B.Arena(BASE, page_end + n_slots * landing, ROW, n_slots, window_pages, slot_pages,
                   TABLES, 4, 16, compute_stream=1, h2d_stream=2, d2h_stream=3,
                   record_only=True, compact_head_dim=256, landing_offset=page_end,
                   landing_bytes=landing)


def test_compact_runs_land_then_expand_on_the_compute_stream(B):
    a = make_compact_arena(B)
    a.stage_layer(0, [(0, 7, [compact(0, 3, 0x1000), staged(3, 2, 0x9000, rows=100)]),
                      (1, 9, [compact(0, 1, 0x5000), resident(1, 1, 2)])])
    assert a.call_log() == [
        "h2d copy h2d bytes=399360 page=4 row=-1",
        "h2d copy h2d bytes=409600 page=7 row=0",
        "h2d copy h2d bytes=133120 page=9 row=-1",
        "h2d table slot=0 runs=4 0:0+3->4 0:3+2->7 1:0+1->9 1:1+1->2",
        "h2d record copy[0]",
        "compute wait copy[0]",
        "compute expand slot=0 runs=2 +0:3->4 +399360:1->9",
    ]
    assert a.stats().staged_bytes == 399360 + 409600 + 133120
    # slot 1's landing area follows slot 0's
    a.mark_attention_done(0)
    a.stage_layer(1, [(0, 7, [compact(0, 2, 0x1000)])])
    assert a.call_log()[-1] == "compute expand slot=1 runs=1 +0:2->12"


def test_compact_runs_are_checked(B):
    a = make_compact_arena(B, landing_pages=4)
    with pytest.raises(B.PagedAttnError) as e:                   # landing holds 4 pages
        a.stage_layer(0, [(0, 7, [compact(0, 5, 0x1000)])])
    assert e.value.code == B.PA_ERR_INVALID and "landing" in str(e.value)
    with pytest.raises(B.PagedAttnError) as e:                   # not fully written
        a.stage_layer(0, [(0, 7, [dict(logical_page=0, n_pages=2, n_rows=100,
                                       host_compact=0x1000)])])
    assert "fully written" in str(e.value)
    with pytest.raises(B.PagedAttnError):
        a.stage_layer(0, [(0, 7, [dict(logical_page=0, n_pages=1, n_rows=64, host_rows=0x10,
                                       host_compact=0x1000)])])
    assert a.call_log() == []
    plain = make_arena(B)
    with pytest.raises(B.PagedAttnError) as e:
        plain.stage_layer(0, [(0, 7, [compact(0, 1, 0x1000)])])
    assert "landing" in str(e.value)


def test_landing_geometry_is_checked(B):
    with pytest.raises(B.PagedAttnError):          # landing overlaps the pages
        B.Arena(BASE, 40 * PAGE * ROW, ROW, 2, 4, 8, TABLES, 4, 16, record_only=True,
                compact_head_dim=256, landing_offset=10 * PAGE * ROW, landing_bytes=CPAGE)
    with pytest.raises(B.PagedAttnError):          # smaller than one compact page
        B.Arena(BASE, 40 * PAGE * ROW, ROW, 2, 4, 8, TABLES, 4, 16, record_only=True,
                compact_head_dim=256, landing_offset=20 * PAGE * ROW, landing_bytes=CPAGE - 16)
    with pytest.raises(B.PagedAttnError):          # head_dim does not divide the row
        B.Arena(BASE, 40 * PAGE * ROW, ROW, 2, 4, 8, TABLES, 4, 16, record_only=True,
                compact_head_dim=96, landing_offset=20 * PAGE * ROW, landing_bytes=CPAGE)


# ---- copy-in of resident pages ("Staging without a stall", section
# "Admission that does arithmetic"; "GPU memory management", section "Pages
# held by right, borrowed or free": a page that turns hot is copied in once) ----

def test_load_resident_orders_compute_after_the_copies(B):
    a = make_arena(B, window_pages=4)
    a.load_resident([(0, 64, 0x1000), (3, 17, 0x9000)])
    assert a.call_log() == [
        "h2d copy h2d bytes=262144 page=0 row=0",
        "h2d copy h2d bytes=69632 page=3 row=0",
        "h2d record load[0]",
        "compute wait load[0]",
    ]
    assert a.stats().loaded_bytes == (64 + 17) * ROW and a.stats().staged_bytes == 0


def test_load_resident_waits_on_the_latest_readers(B):
    a = make_arena(B, n_slots=2, window_pages=4)
    full_layer(B, a, 0, [(0, 1, [resident(0, 1, 0), staged(1, 1, 0x1000, rows=10)])],
               [(0, 73, 0x5000, 1)])
    a.stage_layer(1, [(0, 1, [resident(0, 1, 0), staged(1, 1, 0x2000, rows=10)])])
    a.mark_attention_done(1)            # layer 1: attention, no write-back yet
    n = len(a.call_log())
    a.load_resident([(0, 64, 0x3000)])
    assert a.call_log()[n:] == [
        "h2d wait attn[1]",             # the latest attention (covers layer 0's)
        "h2d wait wb[0]",               # the latest write-back
        "h2d copy h2d bytes=262144 page=0 row=0",
        "h2d record load[0]",
        "compute wait load[0]",
    ]
    a.drain()
    n = len(a.call_log())
    a.load_resident([(1, 64, 0x3000)])  # after a drain nothing is pending
    assert a.call_log()[n:][0] == "h2d copy h2d bytes=262144 page=1 row=0"


def test_load_resident_is_checked_before_anything_is_enqueued(B):
    a = make_arena(B, n_slots=2, slot_pages=8, window_pages=4)
    bad = [
        [(4, 64, 0x1000)],                # slot 0's first page
        [(19, 1, 0x1000)],                # inside slot 1
        [(20, 1, 0x1000)],                # past the arena
        [(-1, 1, 0x1000)],
        [(0, 0, 0x1000)],                 # no rows
        [(0, 65, 0x1000)],                # more rows than a page
        [(0, 64, 0)],                     # null host rows
        [(0, 64, 0x1000), (5, 64, 0x2000)],  # one bad load refuses the call
    ]
    for loads in bad:
        with pytest.raises(B.PagedAttnError) as e:
            a.load_resident(loads)
        assert e.value.code == B.PA_ERR_INVALID
    assert a.call_log() == []
    assert a.stats().loaded_bytes == 0


@pytest.mark.parametrize("fail_at", range(0, 4))
def test_load_resident_failure_quarantines(B, fail_at):
    a = make_arena(B)
    a.fail_after(fail_at)
    with pytest.raises(B.PagedAttnError) as e:
        a.load_resident([(0, 64, 0x1000), (1, 64, 0x2000)])
    assert e.value.code == B.PA_ERR_CUDA
    with pytest.raises(B.PagedAttnError) as e:
        a.load_resident([(0, 64, 0x1000)])
    assert e.value.code == B.PA_ERR_QUARANTINED
    a.drain()
    a.load_resident([(0, 64, 0x1000)])
