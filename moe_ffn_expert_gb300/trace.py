"""Per-tile trace of the layer's kernels: capture, parsing and a timeline summary.

While a trace buffer is set (mm_trace_set, include/mm.h), every kernel of mm_forward /
mm_backward writes 32-byte records: one per CTA (MM_TRACE_CTA), and for the grouped GEMMs one per
tile for the tensor-core mainloop (MM_TRACE_MAINLOOP, the MMA-issuing thread) and one per tile
and CTA for the epilogue (MM_TRACE_EPILOGUE). The RFC "HyperParallel Multicore HyperMegaMoE
fused forward/backward operator" (§8, performance acceptance) asks for the concurrency and
utilisation of the matrix and vector units over time; here the mainloop is the matrix unit's
work and the epilogue warps do the vector work, so `summarize` reports, per launch, how busy
each side was and how much of the epilogue ran hidden under the mainloop, and which launches ran
concurrently (the backward's Combine(dX) beside W1Grad).

Capture (device memory, one thread):

    buf = TraceBuffer(capacity=1 << 20)
    buf.start()
    ... mm_forward / mm_backward ...
    records = buf.stop()          # numpy structured array, RECORD_DTYPE
    text = timeline(summarize(records))
"""
from __future__ import annotations

import numpy as np

from . import _abi

# mm_trace_record (include/mm.h), little-endian
RECORD_DTYPE = np.dtype([("stage", "<u2"), ("role", "<u2"), ("sm", "<u2"), ("rank", "<u2"),
                         ("unit", "<i4"), ("launch", "<u4"), ("t0", "<u8"), ("t1", "<u8")])
assert RECORD_DTYPE.itemsize == _abi.TRACE_RECORD_BYTES

ROLE_NAMES = {_abi.MM_TRACE_CTA: "cta", _abi.MM_TRACE_MAINLOOP: "mainloop",
              _abi.MM_TRACE_EPILOGUE: "epilogue"}


def parse(raw: bytes | np.ndarray) -> tuple[np.ndarray, int]:
    """(records, offered) from the bytes of a trace buffer: the header's count of records
    offered, and the records actually stored (min(offered, capacity))."""
    b = np.frombuffer(bytes(raw) if not isinstance(raw, np.ndarray) else raw.tobytes(), np.uint8)
    if b.size < 2 * RECORD_DTYPE.itemsize:
        raise ValueError("a trace buffer holds a 32-byte header and at least one record")
    offered = int(b[:4].view("<u4")[0])
    cap = b.size // RECORD_DTYPE.itemsize - 1
    n = min(offered, cap)
    recs = b[RECORD_DTYPE.itemsize:RECORD_DTYPE.itemsize * (n + 1)].view(RECORD_DTYPE)
    return recs.copy(), offered


class TraceBuffer:
    """A device buffer for `capacity` records, set as the library's trace buffer by start()."""

    def __init__(self, capacity: int = 1 << 20, device: str = "cuda"):
        import torch
        self.capacity = int(capacity)
        self.nbytes = (self.capacity + 1) * RECORD_DTYPE.itemsize
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        self.offered = 0

    def start(self) -> None:
        self.buf[:RECORD_DTYPE.itemsize].zero_()
        _abi.check(_abi.mm_trace_set(self.buf.data_ptr(), self.nbytes), "mm_trace_set")

    def stop(self) -> np.ndarray:
        """Clears the library's trace buffer, waits for the device and returns the records."""
        import torch
        _abi.check(_abi.mm_trace_set(0, 0), "mm_trace_set")
        torch.cuda.synchronize(self.buf.device)
        recs, self.offered = parse(self.buf.cpu().numpy())
        return recs

    @property
    def dropped(self) -> int:
        return max(0, self.offered - self.capacity)


def stage_names() -> list[str]:
    return [_abi._lib().mm_stage_name(i).decode() for i in range(_abi.MM_NUM_STAGES)]


def _union_length(starts: np.ndarray, ends: np.ndarray) -> int:
    """Total length covered by the intervals [starts[i], ends[i])."""
    if starts.size == 0:
        return 0
    order = np.argsort(starts, kind="stable")
    total, cur_s, cur_e = 0, int(starts[order[0]]), int(ends[order[0]])
    for i in order[1:]:
        s, e = int(starts[i]), int(ends[i])
        if s > cur_e:
            total += cur_e - cur_s
            cur_s, cur_e = s, e
        else:
            cur_e = max(cur_e, e)
    return total + cur_e - cur_s


def _covered(starts: np.ndarray, ends: np.ndarray, cs: np.ndarray, ce: np.ndarray) -> int:
    """Length of the union of [starts, ends) that lies inside the union of [cs, ce)."""
    if starts.size == 0 or cs.size == 0:
        return 0
    a = _union_length(starts, ends)
    b = _union_length(cs, ce)
    both = _union_length(np.concatenate([starts, cs]), np.concatenate([ends, ce]))
    return a + b - both


def summarize(records: np.ndarray, names: list[str] | None = None) -> dict:
    """Per launch (in launch order): stage, start / end / duration in us from the first record,
    CTAs, SMs; for grouped-GEMM launches also
      mainloop_busy   share of the launch's SM-time (SMs x duration) during which an MMA issuer
                      worked on a tile (a CTA-pair unit counts for both SMs of the pair),
      epilogue_busy   the same for the first epilogue warp of each CTA,
      epilogue_hidden share of the epilogue time during which the same SM's (or pair's) MMA
                      issuer was working on another tile (double-buffered accumulators);
    and `concurrent`: pairs of launches whose CTA spans overlap in time, with the overlap in us.
    """
    if names is None:
        names = stage_names()
    out = {"launches": [], "concurrent": [], "records": int(records.size)}
    if records.size == 0:
        return out
    t_base = int(records["t0"].min())
    spans = {}
    for lid in np.unique(records["launch"]):
        r = records[records["launch"] == lid]
        stage = int(r["stage"][0])
        cta = r[r["role"] == _abi.MM_TRACE_CTA]
        src = cta if cta.size else r
        t0, t1 = int(src["t0"].min()), int(src["t1"].max())
        spans[int(lid)] = (t0, t1)
        d = {"launch": int(lid), "stage": names[stage] if stage < len(names) else str(stage),
             "start_us": (t0 - t_base) / 1e3, "end_us": (t1 - t_base) / 1e3,
             "dur_us": (t1 - t0) / 1e3, "ctas": int(cta.size), "sms": int(np.unique(src["sm"]).size)}
        ml = r[r["role"] == _abi.MM_TRACE_MAINLOOP]
        ep = r[r["role"] == _abi.MM_TRACE_EPILOGUE]
        if ml.size:
            # SMs that a mainloop unit keeps busy: the issuer's, and for a pair unit the SM of
            # the other CTA whose epilogue received it
            unit_sms = {}
            for u, sm in zip(ep["unit"], ep["sm"]):
                unit_sms.setdefault(int(u), set()).add(int(sm))
            partner = {}
            for u, sm in zip(ml["unit"], ml["sm"]):
                for other in unit_sms.get(int(u), ()):
                    if other != int(sm):
                        partner[other] = int(sm)
            sm_time = max(1, d["sms"]) * max(1, t1 - t0)
            busy_ml = 0
            for sm in np.unique(ml["sm"]):
                m = ml[ml["sm"] == sm]
                n_sms = 1 + sum(1 for p, o in partner.items() if o == int(sm))
                busy_ml += n_sms * _union_length(m["t0"], m["t1"])
            busy_ep, hidden = 0, 0
            for sm in np.unique(ep["sm"]):
                e = ep[ep["sm"] == sm]
                issuer = partner.get(int(sm), int(sm))
                m = ml[ml["sm"] == issuer]
                busy_ep += _union_length(e["t0"], e["t1"])
                hidden += _covered(e["t0"], e["t1"], m["t0"], m["t1"])
            d.update(mainloop_units=int(ml.size), epilogue_records=int(ep.size),
                     mainloop_busy=busy_ml / sm_time, epilogue_busy=busy_ep / sm_time,
                     epilogue_hidden=hidden / busy_ep if busy_ep else 0.0)
        out["launches"].append(d)
    lids = sorted(spans)
    for i, a in enumerate(lids):
        for b in lids[i + 1:]:
            ov = min(spans[a][1], spans[b][1]) - max(spans[a][0], spans[b][0])
            if ov > 0:
                out["concurrent"].append({"a": a, "b": b, "overlap_us": ov / 1e3})
    return out


def timeline(summary: dict, width: int = 72) -> str:
    """A text chart: one row per launch over the traced interval, '#' while the launch ran."""
    ls = summary["launches"]
    if not ls:
        return "(no records)"
    t_end = max(d["end_us"] for d in ls) or 1.0
    lines = [f"{'launch':<18}{'start us':>10}{'us':>9}  |{'0':<{width - len(f'{t_end:.0f} us')}}"
             f"{t_end:.0f} us|"]
    for d in ls:
        a = int(d["start_us"] / t_end * width)
        b = max(a + 1, int(round(d["end_us"] / t_end * width)))
        bar = "." * a + "#" * (min(b, width) - a) + "." * max(0, width - b)
        lines.append(f"{d['launch']:>3} {d['stage']:<14}{d['start_us']:>10.1f}{d['dur_us']:>9.1f}  |"
                     f"{bar}|")
    return "\n".join(lines)


def report(summary: dict, title: str = "", notes: str = "") -> str:
    """Markdown: a title and notes, the per-launch table (mainloop / epilogue shares for the
    grouped GEMMs), the launches that ran concurrently, and the text timeline."""
    rows = ["| # | stage | start us | us | CTAs | SMs | mainloop busy | epilogue busy | "
            "epilogue hidden |", "|---|---|---|---|---|---|---|---|---|"]
    for d in summary["launches"]:
        g = ("mainloop_busy" in d)
        rows.append(f"| {d['launch']} | {d['stage']} | {d['start_us']:.1f} | {d['dur_us']:.1f} | "
                    f"{d['ctas']} | {d['sms']} | "
                    + (f"{100 * d['mainloop_busy']:.0f} % | {100 * d['epilogue_busy']:.0f} % | "
                       f"{100 * d['epilogue_hidden']:.0f} % |" if g else "| | |"))
    by_id = {d["launch"]: d["stage"] for d in summary["launches"]}
    conc = [f"- {by_id[c['a']]} (#{c['a']}) and {by_id[c['b']]} (#{c['b']}): "
            f"{c['overlap_us']:.1f} us" for c in summary["concurrent"]]
    parts = [f"# {title}" if title else "", notes, "\n".join(rows),
             "Launches whose CTA spans overlap:\n" + ("\n".join(conc) if conc else "- none"),
             "```\n" + timeline(summary) + "\n```"]
    return "\n\n".join(p for p in parts if p) + "\n"
