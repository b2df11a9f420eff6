"""The per-tile trace on a GB300: the records describe the schedule the layer runs (every launch,
one record per CTA, one mainloop record per GEMM unit and one epilogue record per unit and CTA),
their times are ordered as the streams order the launches, tracing changes no output bit, and a
buffer that is too small loses records without being overrun."""
import pytest
import torch

from layer_harness import export_routing, make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from moe_ffn_expert_gb300 import trace
from workloads import synth

pytestmark = pytest.mark.gpu

KEYS = ("y", "dx", "d_topk_weights", "dW_up", "dW_down")
FWD = ["route_count", "route_scan", "route_rank", "gather_x", "gemm1_swiglu", "gemm2", "combine_y"]
BWD = ["gather_dy", "act_grad", "w2_grad", "input_grad", "combine_dx", "w1_grad"]
# (a sum of split weight gradients, "wgrad_reduce", follows a weight gradient when its sizes let
# the routing split an expert's rows; d_topk_weights come from W2Grad's launch, and only a W2Grad
# grid too small for the slots leaves them to a "d_topk" kernel after it)
GEMMS = ["gemm1_swiglu", "gemm2", "act_grad", "w2_grad", "input_grad", "w1_grad"]
SLACK_NS = 2000  # timer granularity allowance when comparing times taken on different SMs


def cdiv(a, b):
    return -(-a // b)


def expected_units(counts, T, H, I, E, K, single):
    """Work units of each grouped GEMM with work (the schedule the kernels document): row tiles
    of 128 (pairs of them for the CTA-pair MMAs) x column tiles; the weight gradients: experts
    with rows x row tiles of the weight (pairs when the experts average >= 256 rows) x 256-column
    tiles."""
    tiles = [cdiv(int(c), 128) for c in counts]
    m = sum(tiles) if single else sum(cdiv(t, 2) for t in tiles)
    busy = sum(1 for c in counts if c > 0)
    wpair = not single and T * K >= 256 * E
    w2_rows = cdiv(I, 128) if not wpair else cdiv(cdiv(I, 128), 2)
    w1_rows = cdiv(2 * I, 128) if not wpair else cdiv(cdiv(2 * I, 128), 2)
    return {"gemm1_swiglu": m * cdiv(I, 128), "gemm2": m * cdiv(H, 256),
            "act_grad": m * cdiv(I, 256), "input_grad": m * cdiv(H, 256),
            "w2_grad": busy * w2_rows * cdiv(H, 256), "w1_grad": busy * w1_rows * cdiv(H, 256)}, wpair


def traced_step(inp, capacity=1 << 16, flags=0, bwd_flags=None):
    tb = trace.TraceBuffer(capacity)
    tb.start()
    out = run_layer(inp, flags=flags, bwd_flags=flags if bwd_flags is None else bwd_flags)
    recs = tb.stop()
    return out, recs, tb


@pytest.mark.parametrize("single", [False, True], ids=["pairs", "one_cta"])
def test_trace_describes_the_schedule(single):
    T, H, I, E, K = 2048, 256, 256, 8, 2
    inp = make_inputs(synth.small("trace", T, H, I, E, K, seed=91))
    flags = _abi.MM_FLAG_SINGLE_CTA_TILES if single else 0
    fwd = flags | _abi.MM_FLAG_SEPARATE_FORWARD_GEMMS  # GEMM1 and GEMM2 as two launches
    ref = run_layer(inp, flags=fwd, bwd_flags=flags)
    out, recs, tb = traced_step(inp, flags=fwd, bwd_flags=flags)
    assert out["status"] == _abi.MM_OK and tb.dropped == 0 and recs.size == tb.offered
    for k in KEYS:  # tracing changes nothing the layer computes
        assert torch.equal(out[k], ref[k]), k
    names = trace.stage_names()
    assert (recs["t1"] >= recs["t0"]).all()
    # every launch of the step, in enqueue order, one stage each
    launches = sorted(set(recs["launch"].tolist()))
    assert launches == list(range(len(launches)))
    stage_of = {}
    for lid in launches:
        st = set(recs["stage"][recs["launch"] == lid].tolist())
        assert len(st) == 1
        stage_of[lid] = names[st.pop()]
    seq = [stage_of[i] for i in launches]
    assert [x for x in seq if x != "wgrad_reduce"] == FWD + BWD
    assert all(seq[i - 1] in ("w2_grad", "w1_grad") for i, x in enumerate(seq) if x == "wgrad_reduce")
    lid_of = {v: k for k, v in stage_of.items()}
    counts, _, _ = export_routing(out, E, T * K)
    units, wpair = expected_units(counts.tolist(), T, H, I, E, K, single)
    for g in GEMMS:
        r = recs[recs["launch"] == lid_of[g]]
        ml = r[r["role"] == _abi.MM_TRACE_MAINLOOP]
        ep = r[r["role"] == _abi.MM_TRACE_EPILOGUE]
        ctas = r[r["role"] == _abi.MM_TRACE_CTA]
        u = sorted(ml["unit"].tolist())
        assert len(u) == units[g] and len(set(u)) == len(u), g
        if g not in ("w1_grad", "w2_grad"):
            assert u == list(range(units[g])), g
        pair = not single and (g not in ("w1_grad", "w2_grad") or wpair)
        assert ctas.size > 0 and (not pair or ctas.size % 2 == 0), g
        assert set(ml["rank"].tolist()) == {0}, g  # a pair's MMAs are issued by its even CTA
        # each unit's accumulator goes to one epilogue per CTA of its pair, after its mainloop
        # started, on the SM of the CTA that issued it or of that CTA's partner
        start = dict(zip(ml["unit"].tolist(), ml["t0"].tolist()))
        per_unit = {}
        for uu, rk, t0 in zip(ep["unit"].tolist(), ep["rank"].tolist(), ep["t0"].tolist()):
            per_unit.setdefault(uu, []).append(rk)
            assert t0 + SLACK_NS >= start[uu], g
        assert sorted(per_unit) == u, g
        assert all(sorted(v) == ([0, 1] if pair else [0]) for v in per_unit.values()), g
    # stream order: a launch's CTAs start after the previous launch of its stream has ended
    # (programmatic launches wait for the previous grid's completion before any work)
    span = {}
    for lid in launches:
        c = recs[(recs["launch"] == lid) & (recs["role"] == _abi.MM_TRACE_CTA)]
        span[lid] = (int(c["t0"].min()), int(c["t1"].max()))
    main = [lid for lid in launches if stage_of[lid] != "combine_dx"]
    for prev, nxt in zip(main, main[1:]):
        assert span[nxt][0] + SLACK_NS >= span[prev][1], (stage_of[prev], stage_of[nxt])
    # the side stream's Combine(dX) starts after input_grad, like W1Grad beside it
    assert span[lid_of["combine_dx"]][0] + SLACK_NS >= span[lid_of["input_grad"]][1]
    s = trace.summarize(recs, names)
    g1 = next(d for d in s["launches"] if d["stage"] == "gemm1_swiglu")
    assert 0.0 < g1["mainloop_busy"] <= 1.0 + 1e-9 and 0.0 < g1["epilogue_busy"] <= 1.0 + 1e-9
    assert "gemm2" in trace.report(s)


def test_trace_overflow_and_off():
    T, H, I, E, K = 1000, 128, 128, 4, 2
    inp = make_inputs(synth.small("trace_small", T, H, I, E, K, seed=92))
    _, full, tb_full = traced_step(inp)
    assert tb_full.dropped == 0
    # 16 record slots inside a larger allocation whose tail must stay untouched
    cap = 16
    nbytes = (cap + 1) * 32
    guard = 4096
    buf = torch.full((nbytes + guard,), 0xAB, dtype=torch.uint8, device="cuda")
    buf[:32].zero_()
    _abi.check(_abi.mm_trace_set(buf.data_ptr(), nbytes), "mm_trace_set")
    run_layer(inp)
    _abi.check(_abi.mm_trace_set(0, 0), "mm_trace_set")
    torch.cuda.synchronize()
    got, offered = trace.parse(buf[:nbytes].cpu().numpy())
    assert offered == full.size and got.size == cap
    assert (buf[nbytes:] == 0xAB).all()
    # tracing off: the same buffer receives nothing more
    head = buf[:4].clone()
    run_layer(inp)
    torch.cuda.synchronize()
    assert torch.equal(buf[:4], head)
    assert (buf[nbytes:] == 0xAB).all()


def test_trace_of_the_one_launch_forward_and_a_shared_expert():
    """The one-launch forward records one mainloop per GEMM1 and per GEMM2 unit in a single
    launch; a shared expert's seven launches (its tables and GEMMs) carry its stage."""
    T, H, I, E, K = 1500, 256, 256, 6, 2
    w = synth.small("trace_fused", T, H, I, E, K, seed=93)
    inp = make_inputs(w)
    names = trace.stage_names()
    tb = trace.TraceBuffer(1 << 16)
    tb.start()
    out = run_layer(inp, flags=_abi.MM_FLAG_FUSED_FORWARD_GEMMS, backward=False)
    recs = tb.stop()
    assert out["status"] == _abi.MM_OK and tb.dropped == 0
    stages = [names[int(recs["stage"][recs["launch"] == lid][0])]
              for lid in sorted(set(recs["launch"].tolist()))]
    assert stages == ["route_count", "route_scan", "route_rank", "gather_x", "gemm1_gemm2",
                      "combine_y"]
    counts, _, _ = export_routing(out, E, T * K)
    pairs = sum(cdiv(cdiv(int(c), 128), 2) for c in counts.tolist())
    fused = recs[recs["stage"] == names.index("gemm1_gemm2")]
    ml = fused[fused["role"] == _abi.MM_TRACE_MAINLOOP]
    assert sorted(ml["unit"].tolist()) == list(range(pairs * (cdiv(I, 128) + cdiv(H, 256))))

    su, sd = synth.shared_up(w, 384, device="cuda"), synth.shared_down(w, 384, device="cuda")
    tb.start()
    out = run_layer(inp, shared=(su, sd))
    recs = tb.stop()
    assert out["status"] == _abi.MM_OK and tb.dropped == 0
    shared = recs[recs["stage"] == names.index("shared_expert")]
    assert len(set(shared["launch"].tolist())) == 7
    # the shared expert's GEMMs are grouped GEMMs like the routed ones: mainloop records in six
    # of its seven launches (not in its routing tables)
    with_ml = {int(l) for l in shared["launch"][shared["role"] == _abi.MM_TRACE_MAINLOOP]}
    assert len(with_ml) == 6
