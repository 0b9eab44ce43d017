"""Happens-before checker for the staging arena's recorded submissions (test
infrastructure only).

The arena's record-only mode logs every submission it would make, one line
each (stream, verb, event or byte range).  This module replays such a log
against the CUDA stream and event rules, with nothing of the arena's own code:

  * work on one stream runs in submission order;
  * ``<stream> record E`` captures everything the stream has been ordered
    after so far; a later record of E replaces it;
  * ``<stream> wait E`` orders the stream's later work after what E captured
    at the time of the wait (nothing if E was never recorded);
  * ``host wait E`` returns once E's captured work is done, so every later
    submission on any stream is ordered after it.

Happens-before is tracked with one vector clock per stream.  Each submission
is turned into the device memory it touches:

  * ``h2d copy ... page=P row=R`` (R >= 0) writes pool rows [64 P + R, + bytes/row);
    with R = -1 (a compact run) it writes the landing area of the slot whose
    page table the stage fills next;
  * ``h2d table slot=S ...`` writes slot S's page table;
  * ``compute expand slot=S runs=...`` reads slot S's landing area and writes
    the listed pages;
  * ``compute record attn[S]`` stands for the caller's attention launch on the
    compute stream just before it: it reads slot S's page table and every page
    that table maps, and writes (the fused tail-row store) the rows that the
    write-back copies logged after it, up to the next attention, read;
  * ``d2h copy ... page=P row=R`` reads pool rows [64 P + R, + bytes/row).

Two accesses race when they overlap, come from different streams, at least
one writes, and the earlier is not ordered before the later.  The ordering
rules are those of "Staging without a stall" (sections "Two copy queues and
device-side ordering" and "Leases instead of buffers"): a slot is refilled
only after the attention and the write-back that read it, attention waits on
the copy, the write-back waits on the attention.
"""

from __future__ import annotations

import re
from dataclasses import dataclass, field

PAGE_TOKENS = 64
STREAMS = ("h2d", "compute", "d2h")


@dataclass
class Access:
    index: int          # log line
    stream: str
    resource: tuple     # ("rows", lo, hi) | ("table", slot) | ("landing", slot)
    write: bool
    clock: dict = field(default_factory=dict)
    what: str = ""


def _overlap(a: tuple, b: tuple) -> bool:
    if a[0] != b[0]:
        return False
    if a[0] == "rows":
        return a[1] < b[2] and b[1] < a[2]
    return a[1] == b[1]


def _join(a: dict, b: dict) -> dict:
    return {s: max(a.get(s, 0), b.get(s, 0)) for s in STREAMS}


def _row_range(line: str, row_bytes: int):
    nbytes = int(re.search(r"bytes=(\d+)", line).group(1))
    page = int(re.search(r"page=(-?\d+)", line).group(1))
    row = int(re.search(r"row=(-?\d+)", line).group(1))
    lo = page * PAGE_TOKENS + row
    return lo, lo + nbytes // row_bytes


_TABLE_RUN = re.compile(r"(\d+):(\d+)\+(\d+)->(\d+)")
_EXPAND_RUN = re.compile(r"\+(\d+):(\d+)->(\d+)")


def accesses(lines, row_bytes: int = 4096):
    """The log's device accesses, each with its stream's vector clock."""
    clock = {s: {t: 0 for t in STREAMS} for s in STREAMS}
    host = {t: 0 for t in STREAMS}
    events = {}
    tables = {}         # slot -> [(first_page, n_pages)] of its latest page table
    out = []

    # the slot of each compact landing copy: that of the next table line; the
    # tail rows each attention stores: those its layer's write-back reads
    landing_slot = {}
    tail_rows = {}
    pending = []
    last_attn = None
    for i, line in enumerate(lines):
        if line.startswith("h2d copy h2d") and line.endswith("row=-1"):
            pending.append(i)
        m = re.match(r"h2d table slot=(\d+)", line)
        if m:
            for j in pending:
                landing_slot[j] = int(m.group(1))
            pending = []
        if re.match(r"compute record attn\[", line):
            last_attn = i
            tail_rows[i] = []
        if line.startswith("d2h copy d2h") and last_attn is not None:
            tail_rows[last_attn].append(_row_range(line, row_bytes))

    def step(stream):
        c = _join(clock[stream], host)
        c[stream] += 1
        clock[stream] = c
        return dict(c)

    for i, line in enumerate(lines):
        words = line.split()
        if words[0] == "host":
            m = re.match(r"host wait (\w+\[\d+\])$", line)
            assert m, line
            host = _join(host, events.get(m.group(1), {}))
            continue
        stream, verb = words[0], words[1]
        assert stream in STREAMS, line
        if verb == "record":
            c = step(stream)
            events[words[2]] = c
            if words[2].startswith("attn["):
                slot = int(words[2][5:-1])
                # the caller's attention launch, just before the record
                out.append(Access(i, stream, ("table", slot), False, c, "attention"))
                for first, n in tables.get(slot, []):
                    out.append(Access(i, stream, ("rows", first * PAGE_TOKENS,
                                                  (first + n) * PAGE_TOKENS), False, c,
                                      "attention"))
                for lo, hi in tail_rows[i]:
                    out.append(Access(i, stream, ("rows", lo, hi), True, c, "attention tail"))
        elif verb == "wait":
            clock[stream] = _join(clock[stream], events.get(words[2], {}))
        elif verb == "copy":
            c = step(stream)
            if line.endswith("row=-1"):
                out.append(Access(i, stream, ("landing", landing_slot[i]), True, c, line))
            else:
                lo, hi = _row_range(line, row_bytes)
                out.append(Access(i, stream, ("rows", lo, hi), words[2] == "h2d", c, line))
        elif verb == "table":
            c = step(stream)
            slot = int(re.search(r"slot=(\d+)", line).group(1))
            tables[slot] = [(int(m.group(4)), int(m.group(3)))
                            for m in _TABLE_RUN.finditer(line)]
            out.append(Access(i, stream, ("table", slot), True, c, line))
        elif verb == "expand":
            c = step(stream)
            slot = int(re.search(r"slot=(\d+)", line).group(1))
            out.append(Access(i, stream, ("landing", slot), False, c, line))
            for m in _EXPAND_RUN.finditer(line):
                n, first = int(m.group(2)), int(m.group(3))
                out.append(Access(i, stream, ("rows", first * PAGE_TOKENS,
                                              (first + n) * PAGE_TOKENS), True, c, line))
        else:
            raise AssertionError(f"unknown log line: {line}")
    return out


def races(lines, row_bytes: int = 4096):
    """Pairs of log lines (earlier, later) whose accesses race."""
    acc = accesses(lines, row_bytes)
    found = []
    for k, b in enumerate(acc):
        for a in acc[:k]:
            if a.stream == b.stream or not (a.write or b.write):
                continue
            if not _overlap(a.resource, b.resource):
                continue
            if a.clock[a.stream] <= b.clock[a.stream]:
                continue            # a is ordered before b
            found.append((a.index, b.index, a.what or a.resource, b.what or b.resource))
    return found
