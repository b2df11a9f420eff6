"""Seeded random layer shapes (ragged T, H and I multiples of 8, expert counts from 1 to 96,
K up to 8, uniform and Zipf routing) through the C ABI: the default launches (CTA-pair MMAs,
paired weight gradients when experts average 256 rows or more) equal the one-CTA launches bit
for bit, and both meet the float64 oracle's bounds (routing bit-exact)."""
import random

import pytest
import torch

import oracle
from layer_harness import assert_close, assert_dtopk, export_routing, make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu


def _shapes(n=24, seed=2026):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        E = rng.choice([1, 2, 3, 5, 8, 13, 32, 96])
        K = rng.randint(1, min(8, E))
        T = rng.choice([1, 7, 129, 333, 1000, 2048, 3001])
        H = 8 * rng.randint(1, 80)
        I = 8 * rng.randint(1, 64)
        kind = rng.choice(["uniform", "zipf"])
        out.append((T, H, I, E, K, kind, 100 + i))
    return out


@pytest.mark.parametrize("T,H,I,E,K,kind,seed", _shapes())
def test_random_shape(T, H, I, E, K, kind, seed):
    w = synth.small("rand", T, H, I, E, K, routing_kind=kind, seed=seed)
    inp = make_inputs(w)
    single = _abi.MM_FLAG_SINGLE_CTA_TILES
    out = run_layer(inp)
    ref = run_layer(inp, flags=single, bwd_flags=single)
    assert out["status"] == _abi.MM_OK and ref["status"] == _abi.MM_OK
    for k in ("y", "dx", "d_topk_weights", "dW_up", "dW_down"):
        assert torch.equal(out[k], ref[k]), k
    h = {k: v.cpu() for k, v in inp.items()}
    counts, offsets, row_of_slot, _ = oracle.route(h["topk_ids"], E)
    g_counts, g_offsets, g_rows = export_routing(out, E, T * K)
    assert torch.equal(g_counts.long(), counts) and torch.equal(g_offsets.long(), offsets)
    assert torch.equal(g_rows.long(), row_of_slot)
    y = oracle.forward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"])
    g = oracle.backward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"], h["dy"])
    assert_close("y", out["y"], y)
    assert_close("dx", out["dx"], g["dx"])
    assert_dtopk(out["d_topk_weights"], g["d_topk_weights"])
    assert_close("dW_up", out["dW_up"], g["dW_up"])
    assert_close("dW_down", out["dW_down"], g["dW_down"])
