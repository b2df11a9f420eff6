"""Many seeded random shapes, bit for bit: the default launches twice (run-to-run determinism),
against the one-CTA launches, a forward with the fused combine and/or the one-launch GEMM1 ->
GEMM2 form, and a backward in another weight-gradient output form (fp32, and/or added into
zeroed outputs), whose bf16 rounding must equal the default bf16 gradients; every fourth shape
also runs with a shared expert of random size, default against one-CTA launches. Different schedules
of the same arithmetic must give the same bits, so a race or an unwritten read in any of them
shows up as a difference. The oracle bounds are checked on fewer shapes in
test_gpu_random_shapes.py. MM_SOAK_SHAPES sets the count (default 300, a few seconds) and
MM_SOAK_SEED the shape sequence (default 777)."""
import os
import random

import pytest
import torch

from layer_harness import make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu

KEYS = ("y", "dx", "d_topk_weights", "dW_up", "dW_down")


def test_soak_schedules_agree_bit_for_bit():
    n = int(os.environ.get("MM_SOAK_SHAPES", "300"))
    seed = int(os.environ.get("MM_SOAK_SEED", "777"))
    rng = random.Random(seed)
    rng_forms = random.Random(seed + 1)  # a stream of its own: the shapes stay those of `seed`
    f32, acc = _abi.MM_FLAG_FP32_WEIGHT_GRADS, _abi.MM_FLAG_ACCUMULATE_WEIGHT_GRADS
    single = _abi.MM_FLAG_SINGLE_CTA_TILES
    fused = (_abi.MM_FLAG_FUSED_COMBINE, _abi.MM_FLAG_FUSED_FORWARD_GEMMS,
             _abi.MM_FLAG_FUSED_COMBINE | _abi.MM_FLAG_FUSED_FORWARD_GEMMS)
    failures = []
    for i in range(n):
        E = rng.choice([1, 2, 3, 4, 6, 8, 13, 16, 32, 64, 96])
        K = rng.randint(1, min(8, E))
        T = rng.choice([1, 5, 64, 127, 128, 129, 255, 333, 777, 1000, 2048, 3001, 4096, 8192])
        H = 8 * rng.randint(1, 128)
        I = 8 * rng.randint(1, 64)
        kind = rng.choice(["uniform", "zipf"])
        ff = rng.choice(fused)
        shape = (T, H, I, E, K, kind)
        inp = make_inputs(synth.small("soak", T, H, I, E, K, routing_kind=kind,
                                      seed=5000 + i + 100003 * (seed - 777)))
        a = run_layer(inp)
        runs = {"again": run_layer(inp),
                "single": run_layer(inp, flags=single, bwd_flags=single)}
        f = run_layer(inp, flags=ff, backward=False)
        wf = rng_forms.choice([f32, acc, f32 | acc])
        gdt = torch.float32 if wf & f32 else torch.bfloat16
        g = run_layer(inp, bwd_flags=wf,
                      d_up=torch.zeros(inp["w_up"].shape, dtype=gdt, device="cuda"),
                      d_down=torch.zeros(inp["w_down"].shape, dtype=gdt, device="cuda"))
        if a["status"] != _abi.MM_OK or f["status"] != _abi.MM_OK or g["status"] != _abi.MM_OK or \
                any(r["status"] != _abi.MM_OK for r in runs.values()):
            failures.append((shape, "status"))
            continue
        diffs = [f"{name}:{k}" for name, r in runs.items() for k in KEYS if not torch.equal(a[k], r[k])]
        if not torch.equal(a["y"], f["y"]):
            diffs.append(f"fused 0x{ff:x}: y")
        for k in ("dW_up", "dW_down"):
            if not torch.equal(g[k].to(torch.bfloat16), a[k]):
                diffs.append(f"weight-gradient form 0x{wf:x}: {k}")
        if i % 4 == 3:  # a shared expert: its own sub-workspace, tables and seven launches
            I_s = 8 * rng_forms.randint(1, 64)
            w = synth.small("soak", T, H, I, E, K, routing_kind=kind,
                            seed=5000 + i + 100003 * (seed - 777))
            sh = (synth.shared_up(w, I_s, device="cuda"), synth.shared_down(w, I_s, device="cuda"))
            sa = run_layer(inp, shared=sh)
            sb = run_layer(inp, shared=sh, flags=single, bwd_flags=single)
            if sa["status"] != _abi.MM_OK or sb["status"] != _abi.MM_OK:
                diffs.append("shared: status")
            else:
                diffs += [f"shared I_s={I_s}: {k}" for k in KEYS + ("dS_up", "dS_down")
                          if not torch.equal(sa[k], sb[k])]
        if diffs:
            failures.append((shape, diffs))
    assert not failures, failures[:10]
