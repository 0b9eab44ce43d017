"""Lease lifecycle of the staging arena, checked on the host (no GPU).

Rules from "Staging without a stall", section "Leases instead of buffers",
and "KV-cache engineering", section "Staging layers under a lease": every
staged layer is a lease with a strictly increasing stage generation; a new
lease begins only after the previous one is sealed or retired; a slot whose
previous lease is sealed but not retired is refilled only after that lease's
attention and write-back events; a lease is sealed only with its own recorded
attention event and current tail write-back; retirement waits on the host,
returns a receipt and releases the copy tickets, and a host page cannot be
recycled while a copy ticket holds it.  Any failure quarantines the arena.
The arena runs in record-only mode: submissions are logged, not made.
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


def arena(B, n_slots=2):
    return B.Arena(BASE, (4 + n_slots * 8) * PAGE * ROW, ROW, n_slots, 4, 8, TABLES, 4, 16,
                   compute_stream=1, h2d_stream=2, d2h_stream=3, record_only=True)


def reqs(owner=7, host=0x1000, pages=2):
    return [(0, owner, [dict(logical_page=0, n_pages=pages, n_rows=pages * PAGE - 1,
                             host_rows=host)])]


TAIL = [(0, 2 * PAGE - 1, 0x9000, 7)]


def full_lease(a, layer, step=0, owner=7, writeback=True):
    L = a.lease_begin(layer, step, reqs(owner))
    att = a.lease_attention_done(L.lease_id)
    wb = a.lease_writeback(L.lease_id, [(0, 2 * PAGE - 1, 0x9000, owner)]) if writeback else 0
    a.lease_seal(L.lease_id, att, wb)
    return L, att, wb


def test_full_lifecycle_and_receipt(B):
    a = arena(B)
    L = a.lease_begin(3, 11, reqs())
    assert L.lease_id == 1 and L.slot == 0 and L.page_table == TABLES
    att = a.lease_attention_done(L.lease_id)
    wb = a.lease_writeback(L.lease_id, TAIL)
    a.lease_seal(L.lease_id, att, wb)
    n = len(a.call_log())
    r = a.lease_retire(L.lease_id)
    assert a.call_log()[n:] == ["host wait copy[0]", "host wait attn[0]", "host wait wb[0]"]
    assert (r.lease_id, r.layer, r.step, r.n_requests) == (1, 3, 11, 1)
    assert r.staged_bytes == (2 * PAGE - 1) * ROW
    assert r.written_back_bytes == ROW
    assert r.tickets_released == 1


def test_stage_generation_strictly_increases(B):
    a = arena(B)
    ids = [full_lease(a, layer)[0].lease_id for layer in range(6)]
    assert ids == sorted(ids) and len(set(ids)) == 6


def test_new_lease_needs_the_previous_sealed_or_retired(B):
    a = arena(B)
    L = a.lease_begin(0, 0, reqs())
    n = len(a.call_log())
    with pytest.raises(B.PagedAttnError) as e:
        a.lease_begin(1, 0, reqs())
    assert e.value.code == B.PA_ERR_ORDER
    att = a.lease_attention_done(L.lease_id)
    with pytest.raises(B.PagedAttnError):
        a.lease_begin(1, 0, reqs())                   # attended but not sealed
    assert len(a.call_log()) == n + 1                 # only the attention event
    a.lease_seal(L.lease_id, att, 0)
    a.lease_begin(1, 0, reqs())                        # sealed: allowed


def test_sealed_not_retired_slot_waits_for_prior_readers(B):
    a = arena(B, n_slots=1)
    full_lease(a, 0)
    n = len(a.call_log())
    a.lease_begin(1, 0, reqs())
    log = a.call_log()[n:]
    assert log[:2] == ["h2d wait attn[0]", "h2d wait wb[0]"]


def test_retired_slot_is_refilled_without_device_waits(B):
    a = arena(B, n_slots=1)
    L, _, _ = full_lease(a, 0)
    a.lease_retire(L.lease_id)
    n = len(a.call_log())
    a.lease_begin(1, 0, reqs())
    assert not any(line.startswith("h2d wait") for line in a.call_log()[n:])


def test_seal_refuses_a_substituted_event(B):
    a = arena(B)
    L = a.lease_begin(0, 0, reqs())
    with pytest.raises(B.PagedAttnError) as e:
        a.lease_seal(L.lease_id, 1, 0)                 # no attention event yet
    assert e.value.code == B.PA_ERR_ORDER
    att = a.lease_attention_done(L.lease_id)
    wb = a.lease_writeback(L.lease_id, TAIL)
    for bad_att, bad_wb in ((att + 100, wb), (att, wb + 1), (att, 0)):
        with pytest.raises(B.PagedAttnError) as e:
            a.lease_seal(L.lease_id, bad_att, bad_wb)
        assert e.value.code == B.PA_ERR_ORDER
    with pytest.raises(B.PagedAttnError):
        a.lease_retire(L.lease_id)                     # still unsealed
    a.lease_seal(L.lease_id, att, wb)
    with pytest.raises(B.PagedAttnError):
        a.lease_seal(L.lease_id, att, wb)              # sealed once
    a.lease_retire(L.lease_id)
    with pytest.raises(B.PagedAttnError):
        a.lease_retire(L.lease_id)                     # retired once


def test_writeback_needs_attention_and_the_staged_owner(B):
    a = arena(B)
    L = a.lease_begin(0, 0, reqs(owner=7))
    with pytest.raises(B.PagedAttnError) as e:
        a.lease_writeback(L.lease_id, TAIL)
    assert e.value.code == B.PA_ERR_ORDER
    a.lease_attention_done(L.lease_id)
    with pytest.raises(B.PagedAttnError) as e:
        a.lease_writeback(L.lease_id, [(0, 5, 0x9000, 8)])
    assert e.value.code == B.PA_ERR_OWNER


def test_host_pages_are_not_recycled_under_a_ticket(B):
    a = arena(B)
    assert a.host_generation(7) == (1, 0)
    L, _, _ = full_lease(a, 0, owner=7)
    assert a.host_generation(7) == (1, 1)
    with pytest.raises(B.PagedAttnError) as e:
        a.host_recycle(7)
    assert e.value.code == B.PA_ERR_ORDER
    assert a.host_recycle(9) == 2                      # an owner with no tickets
    a.lease_retire(L.lease_id)
    assert a.host_generation(7) == (1, 0)
    assert a.host_recycle(7) == 2


def test_resident_only_lease_holds_no_ticket(B):
    a = arena(B)
    L = a.lease_begin(0, 0, [(0, 5, [dict(logical_page=0, n_pages=2, resident_page=0)])])
    assert a.host_generation(5) == (1, 0)
    att = a.lease_attention_done(L.lease_id)
    a.lease_seal(L.lease_id, att, 0)
    r = a.lease_retire(L.lease_id)
    assert r.tickets_released == 0 and r.staged_bytes == 0


def test_stage_and_lease_calls_do_not_mix(B):
    a = arena(B)
    a.lease_begin(0, 0, reqs())
    with pytest.raises(B.PagedAttnError) as e:
        a.stage_layer(1, reqs())
    assert e.value.code == B.PA_ERR_ORDER
    b = arena(B)
    b.stage_layer(0, reqs())
    with pytest.raises(B.PagedAttnError):
        b.lease_begin(1, 0, reqs())


@pytest.mark.parametrize("fail_at", range(0, 10))
def test_failure_quarantines_and_keeps_everything_until_drain(B, fail_at):
    a = arena(B)
    a.fail_after(fail_at)
    failed = False
    try:
        L, att, wb = full_lease(a, 0, owner=7)
        a.lease_retire(L.lease_id)
        L, att, wb = full_lease(a, 1, owner=7)
        a.lease_retire(L.lease_id)
    except B.PagedAttnError as e:
        failed = True
        assert e.code == B.PA_ERR_CUDA
    assert failed
    assert a.stats().quarantined == 1
    for call in (lambda: a.lease_begin(2, 0, reqs()), lambda: a.host_recycle(7)):
        with pytest.raises(B.PagedAttnError) as e:
            call()
        assert e.value.code == B.PA_ERR_QUARANTINED
    a.drain()
    # a drain that establishes completion drops the leases and their tickets
    assert a.host_generation(7)[1] == 0
    L, att, wb = full_lease(a, 2)
    a.lease_retire(L.lease_id)
