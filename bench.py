"""Benchmark of the fused MoE-FFN layer (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload qwen] [--impl reference]

A step is one forward + backward of the layer over one batch of the workload (default: the
Qwen-like layer T=16384, H=2048, I=768, E=128, K=8, uniform top-8 routing), inputs resident in
device memory. Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the layer on its own GPU ("replicas only": the path has no exchange
step on one GPU per layer instance); `value` is the tokens of all ranks / the slowest rank's time.

`--impl reference` times the float64 CPU oracle instead (the reference arm), on a bounded
sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-FFN fwd+bwd tokens/s and TFLOPS (% of GB300 BF16 dense peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# algorithmic FLOPs per slot of each GEMM stage (routed work only, no padding)
GEMM_FLOPS_PER_SLOT = {"gemm1_swiglu": 4, "gemm2": 2, "gemm1_gemm2": 6, "act_grad": 2,
                       "w2_grad": 2, "input_grad": 4, "w1_grad": 4}  # x H*I


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest():
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "moe_ffn_expert_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(stage, w):
    """DRAM bytes per launch of `stage` on workload `w`, from a committed ncu capture of one
    kernel on a smaller case with the same H, I, K and rows per expert (profiles/traffic.json),
    scaled by the ratio of slots (the same as the ratio of experts). None unless the capture was
    taken from the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("captures", {}).get(stage)
    if not e or e.get("source") != source_digest():
        return None
    c = e["case"]
    if (c["H"], c["I"], c["K"]) != (w.H, w.I, w.K) or c["T"] * c["K"] * w.E != w.T * w.K * c["E"]:
        return None
    return int(round((e["dram_read"] + e["dram_write"]) * w.E / c["E"]))


def workload_of(args):
    """The named workload, optionally with a smaller token count (profiling captures)."""
    import dataclasses

    from workloads import synth
    w = synth.BY_NAME[args.workload]
    if args.tokens:
        w = dataclasses.replace(w, T=int(args.tokens))
    if args.experts:
        w = dataclasses.replace(w, E=int(args.experts))
    return w


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_ms: float, units: float, device=None):
    """Max of the elapsed time and sum of the processed units over all ranks (identity at N=1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_ms, units
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("uuid,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[0] != self.uuid and not self.uuid.endswith(parts[0][4:]):
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[2]) for r in rows]
            smax = max(float(r[3]) for r in rows)
            power = [float(r[4]) for r in rows if r[4] not in ("[N/A]", "N/A")]
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
               "samples": len(rows)}
        if power:
            out["power_w_max"] = max(power)
        return out


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    import torch.distributed as dist

    from moe_ffn_expert_gb300 import _abi
    from moe_ffn_expert_gb300 import build as mm_build
    from workloads import synth

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the layer has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        mm_build.build()  # no-op when libmm.so is newer than its sources
    barrier(dev)

    w = workload_of(args)
    T, H, I, E, K = w.T, w.H, w.I, w.E, w.K
    S = T * K
    d = _abi.dims(T, H, I, E, K)
    I_s = args.shared_intermediate
    stream = torch.cuda.current_stream(dev)
    st = stream.cuda_stream

    ids = synth.routing(w).to(dev)
    tw = synth.topk_weights(w).to(dev)
    x = synth.x(w, device=dev)
    dy = synth.dy(w, device=dev)
    wu = synth.w_up(w, device=dev)
    wd = synth.w_down(w, device=dev)
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dtk = torch.empty(T, K, dtype=torch.float32, device=dev)
    du = torch.empty_like(wu)
    dd = torch.empty_like(wd)
    if I_s:  # a shared expert (always-on SwiGLU FFN of intermediate size I_s)
        su, sd = synth.shared_up(w, I_s, device=dev), synth.shared_down(w, I_s, device=dev)
        dsu, dsd = torch.empty_like(su), torch.empty_like(sd)
        se = _abi.shared_expert(I_s, su.data_ptr(), sd.data_ptr(), dsu.data_ptr(), dsd.data_ptr())
        opt = _abi.options(se)
    nbytes = _abi.mm_workspace_size_ex(d, opt) if I_s else _abi.mm_workspace_size(d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    bufs0 = dict(x=x, ids=ids, tw=tw, dy=dy, y=y, dx=dx, dtk=dtk)

    def fwd(bf=bufs0, extra_flags=0, s=None):
        args_f = (bf["x"].data_ptr(), bf["ids"].data_ptr(), bf["tw"].data_ptr(), wu.data_ptr(),
                  wd.data_ptr(), bf["y"].data_ptr(), ws.data_ptr(), nbytes, s or st,
                  args.fwd_flags | extra_flags)
        if I_s:
            _abi.check(_abi.mm_forward_ex(d, opt, *args_f), "fwd")
        else:
            _abi.check(_abi.mm_forward(d, *args_f), "fwd")

    def bwd(bf=bufs0, s=None):
        args_b = (bf["dy"].data_ptr(), bf["x"].data_ptr(), bf["ids"].data_ptr(),
                  bf["tw"].data_ptr(), wu.data_ptr(), wd.data_ptr(), ws.data_ptr(), nbytes,
                  bf["dx"].data_ptr(), bf["dtk"].data_ptr(), du.data_ptr(), dd.data_ptr(), s or st,
                  args.bwd_flags)
        if I_s:
            _abi.check(_abi.mm_backward_ex(d, opt, *args_b), "bwd")
        else:
            _abi.check(_abi.mm_backward(d, *args_b), "bwd")

    def step():
        fwd()
        bwd()

    def timed(fn, n):
        barrier(dev)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        return a.elapsed_time(b)

    first_ms = timed(step, 1)  # first call: attribute setup, descriptor fetch, cold caches
    status = _abi.mm_get_status(ws.data_ptr(), st)
    if status != _abi.MM_OK:
        raise SystemExit(f"device status after first step: {_abi.mm_status_string(status)}")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- main timed region: K steps, per-stage CUDA events on the library's stream
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else uuid).start()
    _abi.mm_timing_read()
    _abi.mm_timing_enable(True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    step_i = [0]

    def step_marked():  # one event per step boundary: the per-step median and minimum
        if step_i[0] == 0:
            step_ev[0].record(stream)
        step()
        step_i[0] += 1
        step_ev[step_i[0]].record(stream)

    elapsed = timed(step_marked, args.steps)
    _abi.mm_timing_enable(False)
    per_step = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps))
    stages = _abi.mm_timing_read()
    clocks = sampler.stop()
    if _abi.mm_get_status(ws.data_ptr(), st) != _abi.MM_OK:
        raise SystemExit("device status error in the timed region")
    elapsed_max, tokens_all = aggregate(elapsed, float(T * args.steps), dev)
    ms_per_step = elapsed_max / args.steps
    value = tokens_all / (elapsed_max / 1e3)

    # ---- forward alone and backward alone
    n_part = args.steps  # as many as the main region: the same clock and power state
    fwd_ms = timed(fwd, n_part) / n_part
    infer_ms = timed(lambda: fwd(extra_flags=_abi.MM_FLAG_FORWARD_ONLY), n_part) / n_part
    fwd()
    bwd_ms = timed(bwd, n_part) / n_part

    # ---- the same step captured once as a CUDA graph and replayed (no per-launch host work)
    graph = None
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):  # one eager step on the capture stream first
            fwd(s=gs.cuda_stream)
            bwd(s=gs.cuda_stream)
        gs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            fwd(s=gs.cuda_stream)
            bwd(s=gs.cuda_stream)
        g.replay()
        n_graph = args.steps
        graph_ms = timed(g.replay, n_graph) / n_graph
        if _abi.mm_get_status(ws.data_ptr(), st) != _abi.MM_OK:
            raise RuntimeError("device status error after the graph replays")
        graph = {"ms_per_step": round(graph_ms, 4), "tokens_per_s": round(T / (graph_ms / 1e3), 1),
                 "note": "one fwd+bwd step captured once as a CUDA graph, replayed "
                         f"{n_graph} times (per-stage timer off)"}
    except Exception as exc:  # reported, not fatal: the headline does not depend on it
        graph = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    # ---- end to end: host buffers in, results out, copies inside the timed region
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())  # noqa: E731
    hx, hids, htw, hdy = pin(x), pin(ids), pin(tw), pin(dy)
    hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    hdx = torch.empty(dx.shape, dtype=dx.dtype, pin_memory=True)
    hdt = torch.empty(dtk.shape, dtype=dtk.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, htw, hdy))
    d2h = sum(t.numel() * t.element_size() for t in (hy, hdx, hdt))

    # Two device buffer sets: while step i computes on one, step i+1's inputs are copied into
    # the other on a copy-in stream and step i-1's results leave on a copy-out stream (the way a
    # training loop prefetches its next batch). Every step still copies all of its inputs in and
    # its results out inside the timed region.
    bufs1 = {k: torch.empty_like(v) for k, v in bufs0.items()}
    sets = (bufs0, bufs1)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_start = torch.cuda.Event()

    def copy_in(i):
        bf = sets[i % 2]
        s_in.wait_event(ev_done[i % 2])  # step i-2 has finished reading this set
        with torch.cuda.stream(s_in):
            for k, h in (("x", hx), ("ids", hids), ("tw", htw), ("dy", hdy)):
                bf[k].copy_(h, non_blocking=True)
        ev_in[i % 2].record(s_in)

    def e2e_run(n):
        ev_start.record(stream)
        s_in.wait_event(ev_start)
        copy_in(0)
        for i in range(n):
            bf = sets[i % 2]
            stream.wait_event(ev_in[i % 2])
            stream.wait_event(ev_out[i % 2])  # step i-2's results have left this set
            fwd(bf)
            bwd(bf)
            ev_done[i % 2].record(stream)
            if i + 1 < n:
                copy_in(i + 1)
            s_out.wait_event(ev_done[i % 2])
            with torch.cuda.stream(s_out):
                hy.copy_(bf["y"], non_blocking=True)
                hdx.copy_(bf["dx"], non_blocking=True)
                hdt.copy_(bf["dtk"], non_blocking=True)
            ev_out[i % 2].record(s_out)
        stream.wait_event(ev_out[(n - 1) % 2])

    e2e_run(3)
    n_e2e = args.steps
    e2e_ms = timed(lambda: e2e_run(n_e2e), 1)
    e2e_max, e2e_tokens = aggregate(e2e_ms, float(T * n_e2e), dev)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return

    peaks, peak_src = load_peaks()
    hi = H * I
    flops = w.flops()
    if I_s:  # the shared expert adds one SwiGLU FFN over every token: 6*H*I_s fwd, 12 bwd
        flops = {k: v + m * H * I_s * T for (k, v), m in zip(flops.items(), (6, 12, 18))}
    total_flops_step = flops["total"]
    tflops = total_flops_step * args.steps * world / (elapsed_max / 1e3) / 1e12
    peak_burst = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak_burst)

    stage_ms = {k: v[0] / max(1, args.steps) for k, v in stages.items()}
    launches = int(sum(v[1] for v in stages.values()))
    gemm_stages = {k: v for k, v in stages.items() if k in GEMM_FLOPS_PER_SLOT and v[1] > 0}
    top = max(gemm_stages, key=lambda k: gemm_stages[k][0])
    top_ms, top_n = gemm_stages[top]
    avg_ms = top_ms / top_n
    top_flops = GEMM_FLOPS_PER_SLOT[top] * hi * S
    achieved = top_flops / (avg_ms / 1e3) / 1e12

    # HBM-bound stages: algorithmic bytes per launch (the least DRAM traffic the step's
    # definition needs: every input read once, every output written once, at the definition's
    # dtypes) / event-timed duration, against the measured copy bandwidth
    Hb = 2 * H
    algo_bytes = {
        # the token rows read once (the K reads of a row after the first hit L2), the slot rows
        # written once
        "gather_x": T * Hb + S * Hb, "gather_dy": T * Hb + S * Hb,
        # the slot rows, routing index and weight read, the token rows written
        "combine_y": S * Hb + T * Hb + 8 * S, "combine_dx": S * Hb + T * Hb + 4 * S,
        # in: dy slot rows, bf16 gate|up, W_down, routing weight; out: bf16 [d_gate|d_up] and
        # one fp32 <g,h> per slot (w*h, which W2Grad reads, is written by GEMM1's epilogue)
        "act_grad": S * (Hb + 4 * I + 4) + E * I * Hb + S * (4 * I + 4),
    }
    # what this build's act_grad moves by design: fp32 gate|up in, [d_gate|d_up] as bf16 hi + lo
    # planes out (the weight gradients' precision), plus one partial per column half
    impl_bytes = {"act_grad": S * (Hb + 8 * I + 4) + E * I * Hb
                  + S * (8 * I + 4 * 2 * ((I + 255) // 256))}
    hbm_peak = peaks["hbm_gbs"]
    hbm_stages = {}
    for k, nbytes_k in algo_bytes.items():
        ms_k, n_k = stages.get(k, (0.0, 0))
        if n_k:
            gbs = nbytes_k / (ms_k / n_k / 1e3) / 1e9
            hbm_stages[k] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 3),
                             "bytes_per_launch": int(nbytes_k)}
            if k in impl_bytes:
                gi = impl_bytes[k] / (ms_k / n_k / 1e3) / 1e9
                hbm_stages[k].update({"impl_bytes_per_launch": int(impl_bytes[k]),
                                      "impl_GB/s": round(gi, 1),
                                      "impl_frac": round(gi / hbm_peak, 3)})
    hbm_stages["note"] = ("algorithmic bytes (each input read once and each output written once, "
                          "at the layer definition's dtypes) / average launch time, against the "
                          "measured copy bandwidth; impl_*: the bytes this build's act_grad moves "
                          "by design (fp32 gate|up, bf16 hi + lo output pairs); combine_dx runs "
                          "beside w1_grad on a second stream")

    # CPU baseline: the oracle on a bounded sample of this workload
    cpu = (cpu_baseline(w, args.cpu_budget, (wu, wd)) if args.cpu_budget > 0 and not I_s
           else None)

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded counter-based generator; inputs larger than L2 (no flush)",
        "config": {"workload": f"{w.name} T={T} H={H} I={I} E={E} K={K}"
                               + (f" shared I_s={I_s}" if I_s else ""), "T": T, "H": H, "I": I,
                   "E": E, "K": K, "routing": w.routing, "seed": w.seed,
                   **({"shared_I": I_s} if I_s else {}),
                   **({"forward_flags": hex(args.fwd_flags)} if args.fwd_flags else {}),
                   **({"backward_flags": hex(args.bwd_flags)} if args.bwd_flags else {}),
                   "l2": "inputs larger than L2: 1.2 GB of expert weights and 0.6 GB of slot rows per step",
                   "parallelism": "single GPU" if world == 1 else f"{world} independent replicas"},
        "tflops": round(tflops, 2),
        "frac_of_bf16_peak": {"burst": round(tflops / peak_burst, 4),
                              "sustained": round(tflops / peak_sus, 4), "peaks": peak_src,
                              "note": "burst: the peak of a GEMM timed alone at full clock, the "
                                      "denominator for short timed regions; sustained: a "
                                      "seconds-long GEMM loop under the power cap"},
        "fwd": {"ms": round(fwd_ms, 4), "tokens_per_s": round(T / (fwd_ms / 1e3), 1),
                "tflops": round(flops["fwd"] / (fwd_ms / 1e3) / 1e12, 2)},
        "fwd_inference": {"ms": round(infer_ms, 4),
                          "tokens_per_s": round(T / (infer_ms / 1e3), 1),
                          "tflops": round(flops["fwd"] / (infer_ms / 1e3) / 1e12, 2),
                          "note": "mm_forward with MM_FLAG_FORWARD_ONLY (no gate|up kept)"},
        "bwd": {"ms": round(bwd_ms, 4), "tokens_per_s": round(T / (bwd_ms / 1e3), 1),
                "tflops": round(flops["bwd"] / (bwd_ms / 1e3) / 1e12, 2)},
        "graph": graph,
        "first_call_ms": round(first_ms, 3),
        "step_ms": {"median": round(per_step[len(per_step) // 2], 4), "min": round(per_step[0], 4),
                    "max": round(per_step[-1], 4)},
        "stages_ms_per_step": {k: round(v, 4) for k, v in stage_ms.items()},
        "hbm_stages": hbm_stages,
        "roofline": {"kernel": top, "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peak_burst, "unit": "TFLOP/s", "frac": round(achieved / peak_burst, 4),
                     "peak_kind": f"bf16 burst ({peak_src})",
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "flops_per_launch": int(top_flops),
                     "ms_per_launch": round(avg_ms, 4),
                     "traffic": profiled_traffic(top, w),
                     **({"executed_tflops": round(2 * achieved, 2),
                         "executed_frac": round(2 * achieved / peak_burst, 4),
                         "executed_frac_of_sustained": round(2 * achieved / peak_sus, 4),
                         "executed_note": "the weight gradients issue two MMAs per k-step (bf16 hi "
                                          "and lo planes of the split operand): twice the "
                                          "algorithmic FLOPs"}
                        if top in ("w1_grad", "w2_grad") else {})},
        "gpu_launches": launches,
        "e2e": {"value": round(e2e_tokens / (e2e_max / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "x, topk_ids, topk_weights, dy copied in from pinned host memory and y, dx, "
                        "d_topk_weights copied out every step, on two copy streams that overlap "
                        "the neighbouring steps' compute (two device buffer sets); expert weights "
                        "and their gradients stay resident"},
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if args.trace and rank == 0:  # one more step, traced, after every timed leg
        import numpy as np

        from moe_ffn_expert_gb300 import trace as mm_trace
        tb = mm_trace.TraceBuffer(capacity=1 << 21, device=dev)
        tb.start()
        step()
        recs = tb.stop()
        summ = mm_trace.summarize(recs)
        title = (f"Trace of one fwd+bwd step: {w.name} (T={T}, H={H}, I={I}, E={E}, K={K}), "
                 f"fwd flags 0x{args.fwd_flags:x}, bwd flags 0x{args.bwd_flags:x}")
        cmd = "python bench.py " + " ".join(sys.argv[1:])
        notes = (f"Made by `{cmd}`: one step after the timed legs, with the per-tile trace on "
                 f"({int(recs.size)} records). Times are %globaltimer ns from the first record; "
                 "tracing adds an atomic per record, so the step here runs a little longer than "
                 "untraced. mainloop busy: share of the launch's SM-time in which an MMA issuer "
                 "held a tile (from taking a free accumulator to its last commit, operand waits "
                 "included; a CTA-pair unit counts for both SMs). epilogue busy: the same for "
                 "the first epilogue warp of each CTA. epilogue hidden: share of that epilogue "
                 "time during which the same SM's (or pair's) MMA issuer held the next tile.")
        with open(args.trace, "w") as f:
            f.write(mm_trace.report(summ, title, notes))
        np.save(os.path.splitext(args.trace)[0] + ".npy", recs)  # the raw records beside it
        line["trace"] = {"file": args.trace, "records": int(recs.size), "dropped": tb.dropped}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ oracle (CPU) arm

def _oracle_tokens(w, n, inputs):
    """fwd+bwd of the float64 oracle over the first n tokens of the workload; returns seconds."""
    import oracle
    x, ids, tw, dy, wu, wd = inputs
    t0 = time.perf_counter()
    oracle.backward(x[:n], ids[:n], tw[:n], wu, wd, dy[:n])  # includes the forward recompute
    oracle.forward(x[:n], ids[:n], tw[:n], wu, wd)
    return time.perf_counter() - t0


def _oracle_inputs(w, n_max, device_weights=None):
    """Host copies of the first n_max tokens' inputs and of the expert weights they use
    (drawn on the host, or copied from the benchmark's device tensors when given)."""
    import torch

    from workloads import synth
    ids = synth.routing(w)[:n_max]
    tw = synth.topk_weights(w)[:n_max]
    x = synth.x(w, rows=range(n_max))
    dy = synth.dy(w, rows=range(n_max))
    if device_weights is not None:
        wu, wd = (t.cpu() for t in device_weights)
    else:
        wu = synth.LazyExperts(w, "up")
        wd = synth.LazyExperts(w, "down")
        for e in torch.unique(ids).tolist():  # draw them before any timing starts
            wu[e], wd[e]
    return x, ids, tw, dy, wu, wd


def _calibrate(w, inp, target_s, n_start=32):
    """Token count whose oracle fwd+bwd takes about target_s (doubling from n_start)."""
    n_max = inp[0].shape[0]
    n = min(n_start, n_max)
    t = _oracle_tokens(w, n, inp)
    while t < target_s / 2 and n < n_max:
        n = min(n_max, int(n * min(8.0, max(2.0, 0.8 * target_s / max(t, 1e-3)))))
        t = _oracle_tokens(w, n, inp)
    return n, t


def cpu_baseline(w, budget_s=15.0, device_weights=None):
    import torch
    torch.set_num_threads(os.cpu_count() or 1)
    inp = _oracle_inputs(w, w.T, device_weights)
    n, t = _calibrate(w, inp, budget_s)
    return {"value": round(n / t, 2), "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": f"float64 oracle fwd+bwd of the first {n} tokens of {w.name} "
                      f"(all experts they route to), {t:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch

    from workloads import synth
    torch.set_num_threads(os.cpu_count() or 1)
    w = workload_of(args)
    inp = _oracle_inputs(w, w.T)
    per_step_budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    n, _ = _calibrate(w, inp, per_step_budget, n_start=8)
    for _ in range(args.warmup):
        _oracle_tokens(w, n, inp)
    total = 0.0
    for _ in range(args.steps):
        total += _oracle_tokens(w, n, inp)
    value = n * args.steps / total
    sample = (f"float64 oracle fwd+bwd of the first {n} tokens of {w.name} per step "
              f"(all experts they route to)")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded counter-based generator",
        "config": {"workload": f"{w.name} T={w.T} H={w.H} I={w.I} E={w.E} K={w.K}", "T": w.T,
                   "H": w.H, "I": w.I, "E": w.E, "K": w.K, "routing": w.routing, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                         "cores": torch.get_num_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="qwen")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (smaller profiling cases)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the workload's expert count (profiling captures: fewer tokens "
                         "with the same rows per expert)")
    ap.add_argument("--fwd-flags", type=lambda v: int(v, 0), default=0,
                    help="mm_forward flags, e.g. 0x8 (one-launch forward GEMMs), 0x10 (combine in "
                         "GEMM2's epilogue), 0x100 (one CTA per tile instead of pair MMAs)")
    ap.add_argument("--bwd-flags", type=lambda v: int(v, 0), default=0,
                    help="mm_backward flags, e.g. 0x100 (one CTA per tile instead of pair MMAs)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--shared-intermediate", type=int, default=0,
                    help="add a shared expert of this intermediate size (0: none)")
    ap.add_argument("--trace", default="",
                    help="after the timed legs, trace one more step (per-tile records, see "
                         "moe_ffn_expert_gb300/trace.py) and write its timeline to this file")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample (0: skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference" and args.shared_intermediate:
        ap.error("the oracle arm times the routed layer only (no --shared-intermediate)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
