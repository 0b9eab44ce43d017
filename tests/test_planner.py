"""Admission planner (device window of each context), checked on the host.

Rules from "Staging without a stall", section "Admission that does
arithmetic", and "GPU memory management", sections "Pages held by right,
borrowed or free" and "A host pool that explains its own size": an explicit
whole-GiB pool; per context a target held by right, a burst borrowed while
pages are free, a floor of sink + 1; each step the sink and newest pages are
wanted hot and filled by reusing the context's own page, taking a free page,
reclaiming (borrowed pages, then pages above a target, then whole idle
contexts, least recently active first) or shrinking from the oldest page; a
context below its floor is refused; every decision is counted; the host pool
fit is min(limit, pool / history bytes) with its formula, refused or shrunk.
"""

import random

import pytest

PAGE = 64
MiB4 = 16 * PAGE * 4096          # one pool page: a 64-token page of all 16 layers


@pytest.fixture(scope="module")
def B():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    from paged_decode_attention_attn_gb300 import binding
    return binding


def planner(B, gib=1, **kw):
    return B.Planner(gib, **kw)


def pages(n):
    return n * PAGE


def test_pool_is_explicit_and_sized_from_its_gib(B):
    p = planner(B, 1)
    assert p.info()[0] == (1 << 30) // MiB4 == 256
    assert "256 pages" in p.formula
    with pytest.raises(B.PagedAttnError) as e:
        planner(B, 0)
    assert e.value.code == B.PA_ERR_INVALID and "automatic" in str(e.value)


def test_host_pool_fit_formula_refuse_and_shrink(B):
    hist = 16 * 131072 * 4096                       # one history: 8 GiB
    p = planner(B, host_pool_bytes=3 * hist + 123, max_contexts=2)
    assert p.info()[1] == 2
    assert "min(max_contexts=2" in p.formula and "= min(2, 3) = 2" in p.formula
    with pytest.raises(B.PagedAttnError) as e:
        planner(B, host_pool_bytes=3 * hist, max_contexts=8)        # refuse mode
    msg = str(e.value)
    assert e.value.code == B.PA_ERR_INVALID
    assert "host_pool_bytes" in msg and "max_contexts" in msg and "= min(8, 3) = 3" in msg
    s = planner(B, host_pool_bytes=3 * hist, max_contexts=8, shrink_mode=True)
    assert s.info()[1] == 3
    for c in range(3):
        s.admit(c, 4)
    with pytest.raises(B.PagedAttnError) as e:
        s.admit(99, 4)
    assert e.value.code == B.PA_ERR_REFUSED                          # the serving layer queues it
    s.release(0)
    s.admit(99, 4)


def test_window_is_sink_plus_newest_and_tail_reuses_own_page(B):
    p = planner(B)
    p.admit(1, target=4)
    assert p.step([(1, pages(10))]) == [True]
    assert sorted(p.resident(1)) == [0, 7, 8, 9]
    assert p.copied(1) == [0, 9, 8, 7]                              # sink, then newest first
    c0 = p.counters()
    assert c0["took_free"] == 4 and c0["copied_in"] == 4
    # the frontier moves by one page: the page that leaves the window is reused
    p.step([(1, pages(10) + 1)])
    res = p.resident(1)
    assert sorted(res) == [0, 8, 9, 10]
    assert p.copied(1) == [10]
    c1 = p.counters()
    assert c1["reused_own"] == 1 and c1["copied_in"] == 5 and c1["took_free"] == 4
    # a step within the same page changes nothing and copies nothing
    p.step([(1, pages(10) + 2)])
    assert p.resident(1) == res and p.copied(1) == []


def test_burst_is_borrowed_only_while_pages_are_free(B):
    p = planner(B)
    p.admit(1, target=2, burst=3)
    p.step([(1, pages(20))])
    assert sorted(p.resident(1)) == [0, 16, 17, 18, 19]             # target + burst


def test_reclamation_order_borrowed_then_above_target_then_idle(B):
    p = planner(B, 1)                                               # 256 pool pages
    p.admit(1, target=100, burst=100)                               # will borrow 100
    p.admit(2, target=50)
    p.step([(1, pages(300))])
    assert len(p.resident(1)) == 200 and p.counters()["free_pages"] == 56
    p.admit(3, target=100)
    p.step([(3, pages(100))])                                       # 56 free + 44 borrowed from 1
    c = p.counters()
    assert c["reclaimed_borrowed"] == 44 and len(p.resident(3)) == 100
    assert len(p.resident(1)) == 156
    # lower 1's target: its pages beyond the new target are "above target"
    p.set_target(1, target=20, burst=0)
    assert len(p.resident(1)) == 156                                # nothing moves between steps
    p.step([(2, pages(200))])                                       # 2 wants 50
    c = p.counters()
    assert c["reclaimed_borrowed"] == 44 + 50 and c["reclaimed_above_target"] == 0
    assert len(p.resident(2)) == 50
    # now idle contexts: 1 and 3 are not listed; 4 needs pages below target
    p.admit(4, target=150)
    p.step([(4, pages(150)), (2, pages(200))])
    c = p.counters()
    assert c["reclaimed_above_target"] + c["reclaimed_idle_contexts"] > 0
    assert len(p.resident(4)) == 150


def test_above_target_pages_are_reclaimed_before_idle_contexts(B):
    p = planner(B, 1)
    p.admit(1, target=200)
    p.admit(2, target=56)
    p.step([(1, pages(300)), (2, pages(300))])                      # 200 + 56: pool full
    assert p.counters()["free_pages"] == 0
    p.set_target(1, target=100)                                     # 1 now holds 100 above target
    p.admit(3, target=30)
    p.step([(2, pages(300)), (3, pages(30))])                       # 1 idle but above target first
    c = p.counters()
    assert c["reclaimed_above_target"] == 30 and c["reclaimed_idle_contexts"] == 0
    assert sorted(p.resident(1))[0] == 0                            # sink kept, oldest taken
    assert max(p.resident(1)) == 299                                # tail kept hot


def test_least_recently_active_context_is_reclaimed_first(B):
    p = planner(B, 1)
    for c in (1, 2):
        p.admit(c, target=10, burst=118)
    p.step([(1, pages(128))])                                       # step 1: ctx 1 (128 pages)
    p.step([(2, pages(128)), (1, pages(128))])                      # step 2: ctx 2 fills the rest
    p.admit(3, target=20)
    p.step([(2, pages(128)), (3, pages(20))])                       # 1 is least recently active
    assert len(p.resident(1)) == 108 and len(p.resident(2)) == 128


def test_shrink_keeps_the_tail_hot_and_refuses_below_the_floor(B):
    p = planner(B, 1)
    p.admit(1, target=256)
    p.step([(1, pages(256))])
    p.admit(2, target=10)
    ok = p.step([(1, pages(256)), (2, pages(10))])                  # 1 holds all at its target
    assert ok == [True, False]                                      # 2 gets nothing: refused
    c = p.counters()
    assert c["refused"] == 1 and c["shrunk_pages"] == 10
    p.set_target(1, target=250)
    ok = p.step([(2, pages(10)), (1, pages(256))])                  # 2 reclaims 1's 6 extra pages
    assert ok[0] and sorted(p.resident(2)) == [0, 5, 6, 7, 8, 9]     # sink + newest, oldest cold
    assert p.counters()["shrunk_pages"] == 10 + 4


def test_copied_pages_are_those_still_hot_at_the_step_boundary(B):
    p = planner(B, 1)                                               # 256 pool pages
    p.admit(1, target=100, burst=156)
    p.admit(2, target=100)
    ok = p.step([(1, pages(300)), (2, pages(100))])                 # 2 reclaims 1's borrowed pages
    assert ok == [True, True]
    res1 = p.resident(1)
    assert len(res1) == 156 and len(p.resident(2)) == 100
    assert sorted(p.copied(1)) == sorted(res1)                      # not the 100 taken back
    assert p.counters()["copied_in"] == 256


def test_release_returns_every_page(B):
    p = planner(B, 1)
    p.admit(1, target=40)
    p.step([(1, pages(40))])
    assert p.counters()["free_pages"] == 216
    p.release(1)
    assert p.counters()["free_pages"] == 256


def test_random_operations_conserve_pages(B):
    rng = random.Random(7)
    p = planner(B, 1, max_contexts=8)
    live, lengths = [], {}
    for step in range(300):
        op = rng.random()
        if op < 0.15 and len(live) < 8:
            c = rng.randrange(1 << 30)
            if c not in live:
                p.admit(c, rng.randrange(2, 80), rng.randrange(0, 40))
                live.append(c)
                lengths[c] = rng.randrange(1, 200 * PAGE)
        elif op < 0.2 and live:
            p.release(live.pop(rng.randrange(len(live))))
        elif op < 0.25 and live:
            p.set_target(rng.choice(live), rng.randrange(2, 80), rng.randrange(0, 40))
        elif live:
            chosen = rng.sample(live, rng.randrange(1, len(live) + 1))
            for c in chosen:
                lengths[c] += rng.randrange(0, 3 * PAGE)
            adm = p.step([(c, lengths[c]) for c in chosen])
            for c, ok in zip(chosen, adm):
                res = p.resident(c)
                n_pages = -(-lengths[c] // PAGE)
                if ok:
                    assert 0 in res or n_pages == 0                 # the sink is hot
                    assert n_pages - 1 in res                       # the newest page is hot
                assert all(0 <= lp < n_pages for lp in res)
        used = [pp for c in live for pp in p.resident(c).values()]
        assert len(used) == len(set(used))                          # no pool page twice
        assert len(used) + p.counters()["free_pages"] == 256


def test_same_inputs_give_the_same_plan(B):
    def run():
        p = planner(B, 1)
        for c in (5, 6, 7):
            p.admit(c, target=60, burst=40)
        for k in range(6):
            p.step([(5, pages(90 + k)), (6, pages(120)), (7, pages(70 + 3 * k))][: 1 + k % 3])
        return [p.resident(c) for c in (5, 6, 7)], p.counters()
    assert run() == run()
