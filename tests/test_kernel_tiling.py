"""Host-side checks of the prefill kernels' work decomposition.

Chunk slots: both fast prefill kernels give block slot j to chunk k of
sequence i when j = floor(q_i / CHUNK) + i + k, and a block finds its
(sequence, chunk) with a warp-ballot search over query_start_loc.  A replay
of that search checks that every chunk of every sequence gets exactly one
slot below floor(total / CHUNK) + batch, including zero-length sequences.

Channel-first segments: fwd_cf_async_kernel streams a chunk's row as
256-token segments from an aligned start a0 and runs most of them without
per-lane checks: those segments are loaded with unchecked 16-byte copies and
stored with unchecked 16-byte stores.  A replay of the kernel's step order
(prologue issues, grouped lean steps, single lean steps, lean steps with a
checked issue, checked steps) for every row phase, width and a set of
sequence layouts, with the tiling constants read from the kernel source,
checks that:
- every unchecked load and store stays inside the chunk [cbeg, cend);
- every segment is issued once, after its ring slot was consumed, and
  consumed once, after it was issued;
- the segments cover the chunk and fit the chunk's segment budget;
- every segment starts on the 256-byte boundary the alignment promises.

Multi-row channel-first kernel: fwd_cf_rows_kernel runs one ring across a
warp's rows, with counters for the issue and consume positions; a replay of
those counters checks the ring's order, slots and commit groups and that
each row's outputs are stored once.  The channel-first streaming kernels
search with four candidates per lane in the final round.

Short problems: fwd_cl_short_kernel and fwd_cf_short_kernel find their chunk
with a search whose final round also fetches every candidate's end, state
line and flag; a replay checks that every chunk gets exactly one slot.  The
channel-first short kernel covers a chunk with a window of kShortSegs
256-token segments from the 16-byte boundary at or before its first token,
plus the vector before the window: a replay checks that the window and that
vector hold every input the chunk's outputs need, that each output token is
stored exactly once and that whole-vector stores stay inside the chunk.
"""
from __future__ import annotations

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_depthwise_conv1d_fwd_gb300", "csrc")


def _constants():
    src = open(os.path.join(CSRC, "ccv_fwd.cu")).read()
    common = open(os.path.join(CSRC, "ccv_common.cuh")).read()
    env = {"kMaxWidth": int(re.search(r"constexpr int kMaxWidth = (\d+);", common).group(1))}
    for name in ("kCfaSegs", "kCfaAlign", "kCfaSlots", "kCfaChunk", "kCfaChunkSplit", "kCfaPer",
                 "kCfrChunk", "kCfrRows", "kCfrRowsMid", "kCfrRowsShort", "kCfrAlign", "kCaThreads", "kCaWarps", "kCaRun", "kCaChunk",
                 "kShortRun", "kShortSegs", "kShortCfChunk"):
        expr = re.search(rf"constexpr int {name} = ([^;]+);", src).group(1)
        env[name] = int(eval(expr, {"__builtins__": {}}, dict(env)))
    return env


K = _constants()
SEG = 256


def replay(phase, cbeg, cend, chunk0, W):
    """Follow the kernel's steps for one row of one chunk; return the events."""
    S, A = K["kCfaSlots"], K["kCfaAlign"]
    need0 = cbeg - (W - 1)
    a0 = need0 - ((phase + need0) & (A - 1))
    nseg = (cend - a0 + SEG - 1) // SEG
    jin1 = max(1, (cend - a0) // SEG)
    issued, consumed = {}, {}
    unchecked_loads, unchecked_stores = [], []
    step = [0]  # index of the step being run; the prologue is step -1

    def issue(m, checked):
        if checked and m >= nseg:
            return  # the checked issue skips segments past the chunk
        assert m not in issued, f"segment {m} issued twice"
        issued[m] = step[0]
        if not checked:
            unchecked_loads.append(m)

    def consume(j, lean):
        assert j in issued, f"segment {j} consumed before it was issued"
        assert j not in consumed, f"segment {j} consumed twice"
        consumed[j] = step[0]
        if lean:
            unchecked_stores.append(j)

    step[0] = -1
    for m in range(1, S - 1):  # prologue: interior segments unchecked
        if m < jin1:
            issue(m, checked=False)
    issue(0, checked=True)
    for m in range(1, S - 1):
        if m >= jin1:
            issue(m, checked=True)

    def run(j, lean, issue_checked):
        step[0] = j
        consume(j, lean)
        issue(j + S - 1, checked=issue_checked)

    run(0, lean=False, issue_checked=True)
    j = 1
    while j + 2 * S - 2 < jin1:  # grouped lean steps
        for u in range(S):
            run(j + u, lean=True, issue_checked=False)
        j += S
    while j + S - 1 < jin1:  # single lean steps
        run(j, lean=True, issue_checked=False)
        j += 1
    while j < jin1:  # lean compute, checked issue
        run(j, lean=True, issue_checked=True)
        j += 1
    while j < nseg:  # checked steps
        run(j, lean=False, issue_checked=True)
        j += 1
    return dict(a0=a0, nseg=nseg, issued=issued, consumed=consumed,
                loads=unchecked_loads, stores=unchecked_stores)


def check(phase, cbeg, cend, chunk0, W):
    S, A = K["kCfaSlots"], K["kCfaAlign"]
    r = replay(phase, cbeg, cend, chunk0, W)
    a0, nseg = r["a0"], r["nseg"]
    assert 1 <= nseg <= K["kCfaSegs"], "the chunk must fit its segment budget"
    assert a0 <= cbeg - (W - 1), "segment 0 must hold the first token needed"
    assert (phase + a0) % A == 0, "segments start on the promised boundary"
    assert set(r["consumed"]) == set(range(nseg)), "every segment is consumed"
    assert a0 + nseg * SEG >= cend, "the segments cover the chunk"
    for m in r["loads"] + r["stores"]:
        lo_t, hi_t = a0 + m * SEG, a0 + (m + 1) * SEG
        assert cbeg <= lo_t and hi_t <= cend, f"unchecked segment {m} leaves the chunk"
    for m, when in r["issued"].items():
        if m in r["consumed"]:
            assert when < r["consumed"][m], f"segment {m} consumed before its copy"
        # the slot m % S was last read by segment m - S, at step m - S
        if m - S >= 0:
            assert r["consumed"][m - S] <= when, f"segment {m} overwrites a live slot"
        assert when >= m - (S - 1), f"segment {m} issued more than S-1 steps ahead"


LENGTHS = [1, 2, 3, 4, 5, 7, 8, 9, 200, 255, 256, 257, 300, 1000, 1790, 2047, 2048,
           2049, 4096, 4100]


@pytest.mark.parametrize("W", [2, 3, 4, 5])
def test_channel_first_segments_stay_inside_their_chunk(W):
    C = K["kCfaChunk"]
    lengths = LENGTHS + [C - 1, C, C + 1, 2 * C + 3]
    for phase in range(K["kCfaAlign"]):
        for start in (0, 1, 7, 8, 13, 128, 4096, 4099):
            for length in lengths:
                for chunk in range((length + C - 1) // C):
                    cbeg = start + chunk * C
                    cend = start + min(length, (chunk + 1) * C)
                    check(phase, cbeg, cend, chunk == 0, W)


def test_constants_are_the_kernels():
    """The replay uses the kernel's own constants."""
    assert K["kCfaChunk"] + K["kMaxWidth"] - 1 + K["kCfaAlign"] - 1 <= K["kCfaSegs"] * SEG
    assert K["kCfaAlign"] * 2 == 256  # tokens of 2 bytes on a 256-byte boundary


def locate(qsl, total, C, slot):
    """The kernels' chunk search, lane by lane: the largest sequence i with
    floor(qsl[i] / C) + i <= slot, by rounds of a 32-lane ballot."""
    lo, n = 0, len(qsl) - 1
    while n > 1:
        stride = (n + 31) >> 5
        mask = 0
        for lane in range(32):
            off = lane * stride
            if off < n and qsl[lo + off] // C + lo + off <= slot:
                mask |= 1 << lane
        if mask == 0:
            break
        top = mask.bit_length() - 1
        lo += top * stride
        n = min(stride, n - top * stride)
    start, end = qsl[lo], qsl[lo + 1]
    if start < 0 or end < start or end > total:
        return None
    k = slot - (start // C + lo)
    if k < 0 or k * C >= end - start:
        return None
    return lo, k


@pytest.mark.parametrize("C", ["kCaChunk"])
def test_chunk_slots_cover_every_chunk_once(C):
    import random

    C = K[C]
    rng = random.Random(7)
    for trial in range(60):
        batch = rng.choice([1, 2, 3, 31, 32, 33, 100, 1025])
        lens = [rng.choice([0, 1, 2, C - 1, C, C + 1, rng.randrange(0, 3 * C)])
                for _ in range(batch)]
        qsl = [0]
        for n in lens:
            qsl.append(qsl[-1] + n)
        total = qsl[-1] + rng.choice([0, 0, 5])  # tokens past the last sequence are skipped
        found = {}
        for slot in range(total // C + batch):
            r = locate(qsl, total, C, slot)
            if r is not None:
                assert r not in found, f"chunk {r} found by slots {found[r]} and {slot}"
                found[r] = slot
        want = {(i, k) for i, n in enumerate(lens) for k in range((n + C - 1) // C)}
        assert set(found) == want


def locate_short(qsl, total, C, slot, per=1):
    """The one-round-trip search (locate_seq): 32-wide narrowing rounds while
    more than 32 * per candidates remain, then one round in which lane l
    takes candidates per*l .. per*l+per-1 and the last candidate with
    floor(qsl[i] / C) + i <= slot of the highest such lane wins.  per = 1 in
    the short kernels, kCfaPer in the channel-first streaming kernels."""
    lo, n = 0, len(qsl) - 1
    while n > 32 * per:
        stride = (n + 31) >> 5
        mask = 0
        for lane in range(32):
            off = lane * stride
            if off < n and qsl[lo + off] // C + lo + off <= slot:
                mask |= 1 << lane
        if mask == 0:
            return None
        top = mask.bit_length() - 1
        lo += top * stride
        n = min(stride, n - top * stride)
    mask, pick = 0, [-1] * 32
    for lane in range(32):
        for k in range(per):
            i = per * lane + k
            if i < n and qsl[lo + i] // C + lo + i <= slot:
                pick[lane] = k
        if pick[lane] >= 0:
            mask |= 1 << lane
    if mask == 0:
        return None
    top = mask.bit_length() - 1
    seq = lo + per * top + pick[top]
    start, end = qsl[seq], qsl[seq + 1]
    if start < 0 or end < start or end > total:
        return None
    k = slot - (start // C + seq)
    if k < 0 or k * C >= end - start:
        return None
    return seq, k


@pytest.mark.parametrize("C, per", [("kShortRun", 1), ("kShortCfChunk", 1), ("kCfaChunk", "kCfaPer"),
                                    ("kCfaChunkSplit", "kCfaPer"), ("kCfrChunk", "kCfaPer")])
def test_short_chunk_slots_cover_every_chunk_once(C, per):
    import random

    C = K[C]
    per = K[per] if isinstance(per, str) else per
    rng = random.Random(11)
    for trial in range(60):
        batch = rng.choice([1, 2, 3, 31, 32, 33, 100, 127, 128, 129, 1025, 4200])
        lens = [rng.choice([0, 1, 2, C - 1, C, C + 1, rng.randrange(0, 3 * C)])
                for _ in range(batch)]
        qsl = [0]
        for n in lens:
            qsl.append(qsl[-1] + n)
        total = qsl[-1] + rng.choice([0, 0, 5])
        found = {}
        for slot in range(total // C + batch):
            r = locate_short(qsl, total, C, slot, per)
            if r is not None:
                assert r not in found, f"chunk {r} found by slots {found[r]} and {slot}"
                found[r] = slot
        want = {(i, k) for i, n in enumerate(lens) for k in range((n + C - 1) // C)}
        assert set(found) == want


@pytest.mark.parametrize("W", [2, 3, 4, 5])
def test_short_channel_first_window(W):
    """For every row phase and a set of chunk positions, the inputs the
    chunk's outputs read (tokens cbeg-(W-1) .. cend-1) lie in the window or
    the vector before it, and every output token is stored once, whole-vector
    stores only inside [cbeg, cend).  (Loads take a whole vector only when
    all 8 tokens lie inside the row, by the kernel's own test.)"""
    CH, SEGS = K["kShortCfChunk"], K["kShortSegs"]
    for total in (1, 7, 8, 300, CH - 1, CH, CH + 1, 3 * CH + 5):
        starts = sorted({0, 1, 3, 8, max(0, total - CH - 2), max(0, total - 1)})
        for start in starts:
            if start >= total:
                continue
            length = total - start
            for chunk in range((length + CH - 1) // CH):
                cbeg = start + chunk * CH
                cend = start + min(length, (chunk + 1) * CH)
                for phase in range(8):
                    a0 = cbeg - ((phase + cbeg) & 7)
                    assert (phase + a0) % 8 == 0 and cbeg - 8 < a0 <= cbeg
                    held = set(range(a0 - 8, a0 + 256 * SEGS))
                    need = set(range(cbeg - (W - 1), cend))
                    assert need <= held, (total, start, chunk, phase)
                    stored = []
                    for sg in range(SEGS):
                        for lane in range(32):
                            t0 = a0 + sg * 256 + lane * 8
                            if t0 + 8 <= cbeg or t0 >= cend:
                                continue
                            if t0 >= cbeg and t0 + 8 <= cend:
                                stored += range(t0, t0 + 8)
                            else:
                                stored += [t for t in range(t0, t0 + 8) if cbeg <= t < cend]
                    assert sorted(stored) == list(range(cbeg, cend)), (total, start, chunk, phase)


def replay_rows(phases, cbeg, cend, chunk0, W):
    """Follow one warp of fwd_cf_rows_kernel: rows with the given phases (in
    tokens mod kCfrAlign), one ring of kCfaSlots slots run across them with
    an issue counter and a consume counter, as in the kernel."""
    S, A = K["kCfaSlots"], K["kCfrAlign"]
    need0 = cbeg if chunk0 else cbeg - (W - 1)
    geo = []
    for ph in phases:
        a0 = need0 - ((ph + need0) & (A - 1))
        geo.append((a0, (cend - a0 + SEG - 1) // SEG))
    nr = len(phases)
    issues, st = [], dict(ir=0, ij=0, islot=0, groups=0)

    def issue_next(step):
        if st["ir"] < nr:
            issues.append((st["ir"], st["ij"], st["islot"], st["groups"], step))
            st["ij"] += 1
            if st["ij"] == geo[st["ir"]][1]:
                st["ij"], st["ir"] = 0, st["ir"] + 1
        st["islot"] = (st["islot"] + 1) & (S - 1)
        st["groups"] += 1  # one commit group per call, empty or not

    for _ in range(S - 1):
        issue_next(-1)
    cr = cj = cslot = step = 0
    consumes, stored = [], {r: [] for r in range(nr)}
    while cr < nr:
        complete = st["groups"] - (S - 2)  # groups 0 .. complete-1 have landed
        consumes.append((cr, cj, cslot, complete, step))
        cslot = (cslot + 1) & (S - 1)
        issue_next(step)
        a0 = geo[cr][0]
        for lane in range(32):
            t0 = a0 + cj * SEG + lane * 8
            stored[cr] += [t for t in range(t0, t0 + 8) if cbeg <= t < cend]
        cj += 1
        if cj == geo[cr][1]:
            cj, cr = 0, cr + 1
        step += 1
    return geo, issues, consumes, stored


@pytest.mark.parametrize("W", [2, 4, 5])
def test_rows_kernel_ring_runs_across_rows(W):
    """Every (row, segment) of a warp's rows is issued once and consumed once,
    in the same order and through the same slot, after its commit group has
    landed and before the slot is issued again; each row's segments start
    on the aligned boundary at or before its first token read (a first
    chunk's first token, a later chunk's first halo token), the inputs its
    outputs need lie in the segments or, for a first chunk, in the 4 tokens
    before them that the prior fills, and each output token is stored
    exactly once."""
    C, A, S = K["kCfrChunk"], K["kCfrAlign"], K["kCfaSlots"]
    per_warp = max(K["kCfrRows"], K["kCfrRowsMid"], K["kCfrRowsShort"]) // 8
    import random

    rng = random.Random(23)
    for trial in range(300):
        start = rng.choice([0, 1, 7, 8, 100, 4099])
        length = rng.choice([1, 2, 3, 5, 255, 256, 257, 1000, C - 1, C, C + 1, 2 * C + 3])
        nr = rng.randint(1, per_warp)
        stride = rng.choice([0, 1, 8, 13, 64])  # row-to-row phase step
        phase0 = rng.randrange(A)
        phases = [(phase0 + r * stride) % A for r in range(nr)]
        for chunk in range((length + C - 1) // C):
            cbeg = start + chunk * C
            cend = start + min(length, (chunk + 1) * C)
            chunk0 = chunk == 0
            geo, issues, consumes, stored = replay_rows(phases, cbeg, cend, chunk0, W)
            assert [i[:3] for i in issues] == [c[:3] for c in consumes]
            for m, (iss, con) in enumerate(zip(issues, consumes)):
                assert iss[3] < con[3], f"item {m} read before its group landed"
                if m + S < len(issues):
                    assert issues[m + S][4] >= con[4], f"slot of item {m} reissued before it was read"
            for r, (a0, nseg) in enumerate(geo):
                need0 = cbeg if chunk0 else cbeg - (W - 1)
                assert (phases[r] + a0) % A == 0 and need0 - A < a0 <= need0
                held_from = a0 - 4 if chunk0 else a0  # the prior fills a0-4 .. a0-1
                assert held_from <= cbeg - (W - 1) and a0 + nseg * SEG >= cend
                assert sorted(stored[r]) == list(range(cbeg, cend))
