"""Race checks of the staging arena's device ordering, on the CPU.

Record-only arenas are driven through seeded random stage, lease and
planner sessions (staged, resident and compact runs, copy-ins of resident
pages, one to three slots, write-back or not), the way the decode routes
drive them; the happens-before checker in
``event_order.py`` replays each log against the CUDA stream and event rules
and must find no race.  The checker is pinned first by hand-written logs and
then by planted mistakes: every wait, and every copy record, dropped from a
correct log on the CPU, must be flagged.  This is the mutation check of
"Staging without a stall" (a too-early slot reuse gives plausible wrong
output, so the gate must be shown to catch it) without breaking any GPU code.
"""

import numpy as np
import pytest

import event_order as E

PAGE = 64
ROW = 4096
BASE = 1 << 32
TABLES = 1 << 33
CPAGE = 133120          # compact page bytes at 4 kv heads x 256
SLOT_PAGES = 8
LANDING_PAGES = 4


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    return binding


def make_arena(B, n_slots, window_pages, compact):
    page_end = (window_pages + n_slots * SLOT_PAGES) * PAGE * ROW
    kw = {}
    extra = 0
    if compact:
        kw = dict(compact_head_dim=256, landing_offset=page_end,
                  landing_bytes=LANDING_PAGES * CPAGE)
        extra = n_slots * LANDING_PAGES * CPAGE
    return B.Arena(BASE, page_end + extra, ROW, n_slots, window_pages, SLOT_PAGES, TABLES, 4, 16,
                   compute_stream=1, h2d_stream=2, d2h_stream=3, record_only=True, **kw)


def random_layer(rng, layer, n_req, compact):
    """Requests and tail rows of one layer: per request an optional compact
    run, a staged run (last page possibly partial) and optionally a resident
    window page of its own (distinct per layer and request)."""
    reqs, tails = [], []
    for r in range(n_req):
        owner = 100 + r
        host = 0x10000000 * (layer + 1) + 0x1000000 * r
        runs, lp = [], 0
        if compact and rng.random() < 0.6:
            n = int(rng.integers(1, 3))
            runs.append(dict(logical_page=lp, n_pages=n, n_rows=n * PAGE, host_compact=host))
            lp += n
        n = int(rng.integers(1, 3))
        window = rng.random() < 0.4
        rows = n * PAGE if window else int(rng.integers((n - 1) * PAGE + 1, n * PAGE + 1))
        runs.append(dict(logical_page=lp, n_pages=n, n_rows=rows, host_rows=host + 0x800000))
        if window:
            lp += n
            runs.append(dict(logical_page=lp, n_pages=1, resident_page=layer * n_req + r))
            tail = lp * PAGE + int(rng.integers(0, PAGE))
        else:
            tail = lp * PAGE + rows - 1
        reqs.append((r, owner, runs))
        tails.append((r, tail, 0x7000000 + 0x10000 * layer + r, owner))
    return reqs, tails


def stage_session(B, seed, n_slots, compact, n_layers=4, steps=3, n_req=2, wb_prob=0.8):
    rng = np.random.default_rng(seed)
    a = make_arena(B, n_slots, n_layers * n_req, compact)
    for _ in range(steps):
        for layer in range(n_layers):
            reqs, tails = random_layer(rng, layer, n_req, compact)
            a.stage_layer(layer, reqs)
            a.mark_attention_done(layer)
            if rng.random() < wb_prob:
                a.writeback_tail(layer, tails)
    return a.call_log()


def lease_session(B, seed, n_slots, compact, n_layers=4, steps=3, n_req=2):
    rng = np.random.default_rng(seed)
    a = make_arena(B, n_slots, n_layers * n_req, compact)
    for step in range(steps):
        live = []
        for layer in range(n_layers):
            reqs, tails = random_layer(rng, layer, n_req, compact)
            lease = a.lease_begin(layer, step, reqs)
            att = a.lease_attention_done(lease.lease_id)
            wb = a.lease_writeback(lease.lease_id, tails) if rng.random() < 0.8 else 0
            a.lease_seal(lease.lease_id, att, wb)
            live.append(lease.lease_id)
        for lid in live:
            a.lease_retire(lid)
    return a.call_log()


# ---- the checker, pinned on hand-written logs ----

GOOD = [
    "h2d copy h2d bytes=524288 page=4 row=0",
    "h2d table slot=0 runs=1 0:0+2->4",
    "h2d record copy[0]",
    "compute wait copy[0]",
    "compute record attn[0]",
    "d2h wait attn[0]",
    "d2h copy d2h bytes=4096 page=5 row=63",
    "d2h record wb[0]",
    "h2d wait attn[0]",
    "h2d wait wb[0]",
    "h2d copy h2d bytes=524288 page=4 row=0",
    "h2d table slot=0 runs=1 0:0+2->4",
    "h2d record copy[0]",
    "compute wait copy[0]",
    "compute record attn[0]",
]


def test_checker_accepts_an_ordered_log():
    assert E.races(GOOD) == []


def test_checker_flags_a_wait_issued_before_its_record():
    # the second stage's attention waits before that stage's copy is recorded:
    # it sees the first copy's record and reads the refill unordered
    bad = GOOD[:12] + ["compute wait copy[0]", "h2d record copy[0]", "compute record attn[0]"]
    found = E.races(bad)
    assert any(r[0] == 10 and r[3] == "attention" for r in found)


def test_checker_flags_a_wait_on_an_event_never_recorded():
    bad = [line.replace("compute wait copy[0]", "compute wait copy[1]") for line in GOOD[:5]]
    assert E.races(bad)


def test_checker_orders_through_host_waits():
    refill = GOOD[10:]
    with_host = GOOD[:8] + ["host wait attn[0]", "host wait wb[0]"] + refill
    assert E.races(with_host) == []
    assert E.races(GOOD[:8] + refill)          # no wait of any kind: the refill races
    assert E.races(GOOD[:8] + ["host wait attn[0]"] + refill)   # the write-back still reads


def test_checker_flags_overlapping_rows_only():
    # another slot (its own pages and page table) needs no wait on slot 0's
    # readers; the same pages under another slot's table still do
    other = [GOOD[10].replace("page=4", "page=12"), "h2d table slot=1 runs=1 0:0+2->12",
             "h2d record copy[1]", "compute wait copy[1]", "compute record attn[1]"]
    assert E.races(GOOD[:8] + other) == []
    same_pages = [GOOD[10]] + other[1:]
    assert E.races(GOOD[:8] + same_pages)


def test_checker_covers_compact_landing_and_expand():
    log = [
        "h2d copy h2d bytes=266240 page=4 row=-1",
        "h2d table slot=0 runs=1 0:0+2->4",
        "h2d record copy[0]",
        "compute wait copy[0]",
        "compute expand slot=0 runs=1 +0:2->4",
        "compute record attn[0]",
        "h2d wait attn[0]",
        "h2d copy h2d bytes=266240 page=4 row=-1",
        "h2d table slot=0 runs=1 0:0+2->4",
        "h2d record copy[0]",
        "compute wait copy[0]",
        "compute expand slot=0 runs=1 +0:2->4",
        "compute record attn[0]",
    ]
    assert E.races(log) == []
    found = E.races(log[:6] + log[7:])          # landing refilled before the expand ran
    assert any(r[2] == log[4] and r[1] == 6 for r in found)


# ---- the arena's own logs ----

@pytest.mark.parametrize("n_slots", [1, 2, 3])
@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("seed", range(4))
def test_stage_sessions_have_no_race(B, seed, n_slots, compact):
    log = stage_session(B, seed, n_slots, compact)
    assert any("wait attn" in line for line in log) or n_slots >= 4
    assert E.races(log) == []


@pytest.mark.parametrize("n_slots", [1, 2, 3])
@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("seed", range(3))
def test_lease_sessions_have_no_race(B, seed, n_slots, compact):
    assert E.races(lease_session(B, seed, n_slots, compact)) == []


# ---- planted mistakes in correct logs ----

def fixed_session(B, compact, n_slots=2, n_layers=4, steps=3, n_req=2, wb_layers=(0, 2)):
    """Every stage of a slot fills the same pages (per request a compact page
    or not, then a staged page holding the tail row), so each wait the arena
    issues guards bytes: the checker must flag its loss."""
    a = make_arena(B, n_slots, 1, compact)
    for step in range(steps):
        for layer in range(n_layers):
            reqs, tails = [], []
            for r in range(n_req):
                host = 0x10000000 * (layer + 1) + 0x1000000 * r
                runs = []
                if compact:
                    runs.append(dict(logical_page=0, n_pages=1, n_rows=PAGE, host_compact=host))
                lp = len(runs)
                runs.append(dict(logical_page=lp, n_pages=1, n_rows=40, host_rows=host + 0x800000))
                reqs.append((r, 100 + r, runs))
                tails.append((r, lp * PAGE + 39, 0x7000000 + 0x10000 * layer + r, 100 + r))
            a.stage_layer(layer, reqs)
            a.mark_attention_done(layer)
            if layer in wb_layers:
                a.writeback_tail(layer, tails)
    return a.call_log()


@pytest.mark.parametrize("compact", [False, True])
def test_every_dropped_wait_or_copy_record_is_flagged(B, compact):
    log = fixed_session(B, compact)
    assert E.races(log) == []
    seen = set()
    for i, line in enumerate(log):
        words = line.split()
        if not (" wait " in line or line.startswith("h2d record copy")):
            continue
        kind = words[0] + " " + words[2].split("[")[0]
        seen.add(kind)
        mutant = log[:i] + log[i + 1:]
        if kind == "h2d attn" and log[i + 1] == line.replace("attn", "wb"):
            # the slot's write-back event was recorded after a wait on its
            # attention, so the wait on it orders the refill after both:
            # the attention wait is implied; dropping both is flagged
            assert E.races(mutant) == []
            assert E.races(log[:i] + log[i + 2:]), f"dropping lines {i}, {i + 1} went unnoticed"
        else:
            assert E.races(mutant), f"dropping line {i} ({line}) went unnoticed"
    assert seen >= {"h2d attn", "h2d wb", "compute copy", "d2h attn", "h2d copy"}


def test_dropped_host_waits_are_flagged_when_they_order_a_refill(B):
    # leases: a slot whose lease was retired (host waits) is refilled without
    # device waits, so the host waits are what order the refill
    log = lease_session(B, 3, 2, False, n_layers=2, steps=3)
    assert E.races(log) == []
    host = [i for i, line in enumerate(log) if line.startswith("host wait")]
    flagged = 0
    for i in host:
        if E.races(log[:i] + log[i + 1:]):
            flagged += 1
    assert flagged >= 1
    stripped = [line for line in log if not line.startswith("host wait")]
    assert E.races(stripped)


# ---- copy-in of resident pages (the planner's hot pages, a static window) ----

def planner_session(B, seed, n_slots, n_layers=3, steps=4, n_req=2, pool_pages=3):
    """Each step copies a random set of pool pages in (kv_load_resident), then
    stages every layer with runs mapping pool pages of its own region and a
    staged run, tails in either; write-backs on random layers."""
    rng = np.random.default_rng(seed)
    a = make_arena(B, n_slots, n_layers * pool_pages, False)
    for step in range(steps):
        loads = []
        for layer in range(n_layers):
            for p in range(pool_pages):
                if rng.random() < 0.5:
                    loads.append((layer * pool_pages + p, int(rng.integers(1, PAGE + 1)),
                                  0x20000000 + 0x100000 * (step * 16 + layer * pool_pages + p)))
        a.load_resident(loads)
        for layer in range(n_layers):
            reqs, tails = [], []
            for r in range(n_req):
                p = int(rng.integers(0, pool_pages))
                runs = [dict(logical_page=0, n_pages=1, resident_page=layer * pool_pages + p),
                        dict(logical_page=1, n_pages=1, n_rows=int(rng.integers(1, PAGE + 1)),
                             host_rows=0x10000000 * (layer + 1) + 0x1000000 * r)]
                tail = int(rng.integers(0, 2 * PAGE))
                reqs.append((r, 100 + r, runs))
                tails.append((r, tail, 0x7000000 + 0x10000 * layer + r, 100 + r))
            a.stage_layer(layer, reqs)
            a.mark_attention_done(layer)
            if rng.random() < 0.7:
                a.writeback_tail(layer, tails)
    return a.call_log()


@pytest.mark.parametrize("n_slots", [1, 2, 3])
@pytest.mark.parametrize("seed", range(4))
def test_planner_sessions_have_no_race(B, seed, n_slots):
    log = planner_session(B, seed, n_slots)
    assert any("record load" in line for line in log)
    assert E.races(log) == []


def fixed_load_session(B, steps=3):
    """Every step reloads pool page 0, which both layers map and whose row 10
    holds the new token (stored by the attention, read by the write-back),
    between layer 0's stage and its attention; only layer 0 writes back.
    Three slots, so some loads follow a stage that waited on nothing."""
    a = make_arena(B, 3, 1, False)
    for step in range(steps):
        for layer in range(2):
            runs = [dict(logical_page=0, n_pages=1, resident_page=0),
                    dict(logical_page=1, n_pages=1, n_rows=40,
                         host_rows=0x10000000 * (layer + 1))]
            a.stage_layer(layer, [(0, 100, runs)])
            if layer == 0:
                a.load_resident([(0, PAGE, 0x20000000 + 0x100000 * step)])
            a.mark_attention_done(layer)
            if layer == 0:
                a.writeback_tail(layer, [(0, 10, 0x7000000 + layer, 100)])
    return a.call_log()


def test_every_kind_of_load_wait_and_record_guards_bytes(B):
    log = fixed_load_session(B)
    assert E.races(log) == []
    loads = [i for i, line in enumerate(log) if line.startswith("h2d copy") and "page=0 " in line]
    assert len(loads) == 3
    flagged = set()
    for c in loads:
        # the load's own lines: the waits just before its copy, its record and
        # the compute wait just after it
        own = [c + 1, c + 2] + [j for j in (c - 1, c - 2) if log[j].startswith("h2d wait")]
        for i in own:
            if E.races(log[:i] + log[i + 1:]):
                flagged.add(log[i].split("[")[0])
    assert flagged == {"h2d record load", "compute wait load", "h2d wait attn", "h2d wait wb"}
