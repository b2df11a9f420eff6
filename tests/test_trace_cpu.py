"""The trace parser and summary (moe_ffn_expert_gb300/trace.py) on hand-made records, and the
host-side argument checks of mm_trace_set. No GPU: the summary's shares are checked against
values worked out by hand for a two-launch trace."""
import ctypes

import numpy as np
import pytest

from moe_ffn_expert_gb300 import _abi
from moe_ffn_expert_gb300 import build as mm_build
from moe_ffn_expert_gb300 import trace

NAMES = [f"stage{i}" for i in range(16)]
CTA, ML, EP = _abi.MM_TRACE_CTA, _abi.MM_TRACE_MAINLOOP, _abi.MM_TRACE_EPILOGUE


def recs(rows):
    """rows: (stage, role, sm, rank, unit, launch, t0, t1)"""
    a = np.zeros(len(rows), trace.RECORD_DTYPE)
    for i, r in enumerate(rows):
        a[i] = r
    return a


def buffer_bytes(records, offered, capacity):
    b = np.zeros((capacity + 1) * 32, np.uint8)
    b[:4] = np.frombuffer(np.uint32(offered).tobytes(), np.uint8)
    raw = records.tobytes()
    b[32:32 + len(raw)] = np.frombuffer(raw, np.uint8)
    return b


def test_record_layout_matches_header():
    # mm_trace_record: stage, role, sm, rank (uint16), unit (int32), launch (uint32), t0, t1
    assert trace.RECORD_DTYPE.itemsize == 32
    assert [trace.RECORD_DTYPE.fields[k][1] for k in ("unit", "launch", "t0", "t1")] == [8, 12, 16, 24]
    text = open(_abi.HEADER_PATH).read()
    for name in ("uint16_t stage", "uint16_t role", "uint16_t sm", "uint16_t rank", "int32_t unit",
                 "uint32_t launch", "uint64_t t0, t1"):
        assert name in text


def test_parse_counts_dropped_records():
    r = recs([(3, CTA, 0, 0, 0, 0, 10, 20), (3, CTA, 1, 0, 1, 0, 12, 25)])
    got, offered = trace.parse(buffer_bytes(r, offered=5, capacity=2))
    assert offered == 5 and got.size == 2
    assert got["t1"].tolist() == [20, 25] and got["sm"].tolist() == [0, 1]
    got, offered = trace.parse(buffer_bytes(r[:1], offered=1, capacity=4))
    assert offered == 1 and got.size == 1
    with pytest.raises(ValueError):
        trace.parse(np.zeros(32, np.uint8))


def test_union_and_cover():
    s, e = np.array([0, 5, 20]), np.array([10, 15, 30])
    assert trace._union_length(s, e) == 25
    assert trace._union_length(np.array([]), np.array([])) == 0
    # [0, 15) u [20, 30) inside [8, 22): 7 + 2
    assert trace._covered(s, e, np.array([8]), np.array([22])) == 9


def two_launch_trace():
    # launch 0: a pair unit schedule on SMs 0 (rank 0, issues the MMAs) and 1 (rank 1):
    # mainloops [0, 40) and [40, 80) on SM 0; each unit's epilogue on both SMs right after it
    # launch 1: one CTA on SM 5, [50, 150), concurrent with launch 0 for 50 ns
    return recs([
        (4, CTA, 0, 0, 0, 0, 0, 100), (4, CTA, 1, 1, 1, 0, 0, 100),
        (4, ML, 0, 0, 0, 0, 0, 40), (4, ML, 0, 0, 1, 0, 40, 80),
        (4, EP, 0, 0, 0, 0, 40, 60), (4, EP, 1, 1, 0, 0, 40, 60),
        (4, EP, 0, 0, 1, 0, 80, 100), (4, EP, 1, 1, 1, 0, 80, 100),
        (12, CTA, 5, 0, 0, 1, 50, 150),
    ])


def test_summary_shares_by_hand():
    s = trace.summarize(two_launch_trace(), NAMES)
    a, b = s["launches"]
    assert (a["stage"], a["ctas"], a["sms"]) == ("stage4", 2, 2)
    assert a["dur_us"] == pytest.approx(0.1) and b["start_us"] == pytest.approx(0.05)
    # SM-time 2 x 100; the issuer's 80 ns of mainloop keep both SMs of the pair busy
    assert a["mainloop_busy"] == pytest.approx(160 / 200)
    # 2 x 40 ns of epilogue; [40, 60) lies under the second mainloop, [80, 100) under none
    assert a["epilogue_busy"] == pytest.approx(80 / 200)
    assert a["epilogue_hidden"] == pytest.approx(0.5)
    assert a["mainloop_units"] == 2 and a["epilogue_records"] == 4
    assert "mainloop_busy" not in b
    assert s["concurrent"] == [{"a": 0, "b": 1, "overlap_us": pytest.approx(0.05)}]


def test_summary_planted_mistake_changes_shares():
    # a mistake a summary could make: counting a pair unit for one SM only. With the rank-1
    # epilogue records moved to the issuer's SM (no partner), mainloop_busy halves.
    r = two_launch_trace()
    r["sm"][(r["role"] == EP) & (r["rank"] == 1)] = 0
    r = r[~((r["role"] == CTA) & (r["sm"] == 1))]
    s = trace.summarize(r, NAMES)
    assert s["launches"][0]["mainloop_busy"] == pytest.approx(80 / 100)


def test_timeline_and_report_text():
    s = trace.summarize(two_launch_trace(), NAMES)
    t = trace.timeline(s, width=40)
    lines = t.splitlines()
    assert len(lines) == 3
    bars = [ln[ln.index("|") + 1:ln.rindex("|")] for ln in lines[1:]]
    assert all(len(b) == 40 for b in bars)
    assert bars[0].startswith("#") and bars[1].startswith(".") and bars[1].endswith("#")
    md = trace.report(s, "two launches")
    assert "stage12 (#1)" in md and "80 %" in md and "50 %" in md
    assert trace.summarize(np.zeros(0, trace.RECORD_DTYPE), NAMES)["launches"] == []


def test_trace_set_host_checks():
    # host-side checks only: no kernel is launched while the (host) buffer is set
    mm_build.build()
    buf = (ctypes.c_uint8 * 256)()
    base = ctypes.addressof(buf)
    aligned = (base + 31) // 32 * 32
    try:
        assert _abi.mm_trace_set(aligned + 4, 128) == _abi.MM_ERR_INVALID_ARG
        assert _abi.mm_trace_set(aligned, 32) == _abi.MM_ERR_INVALID_ARG
        assert _abi.mm_trace_set(aligned, 64) == _abi.MM_OK
    finally:
        assert _abi.mm_trace_set(0, 0) == _abi.MM_OK
