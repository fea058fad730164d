"""Host-side check of the channel-first prefill kernel's segment arithmetic.

fwd_cf_async_kernel streams a chunk's row as 256-token segments from an
aligned start a0 and runs most of them without per-lane checks: those
segments are loaded with unchecked 16-byte copies and stored with unchecked
16-byte stores.  This test replays the kernel's step order (prologue issues,
grouped lean steps, single lean steps, lean steps with a checked issue,
checked steps) for every row phase, width and a set of sequence layouts, with
the tiling constants read from the kernel source, and checks that:
- every unchecked load and store stays inside the chunk [cbeg, cend);
- every segment is issued once, after its ring slot was consumed, and
  consumed once, after it was issued;
- the segments cover the chunk and fit the chunk's segment budget;
- every segment starts on the 256-byte boundary the alignment promises.
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
    for name in ("kCfaSegs", "kCfaAlign", "kCfaSlots", "kCfaChunk"):
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
