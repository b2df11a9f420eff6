"""Shared-expert fusion (RFC "HyperParallel Multicore HyperMegaMoE fused forward/backward operator",
§6.1) through the C ABI and the torch entry point, against the float64 oracle, with the same
tolerances as the routed layer."""
import pytest
import torch

import oracle
from layer_harness import assert_close, assert_dtopk, make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu


def _case(T, H, I, E, K, I_s, seed):
    w = synth.small("se", T, H, I, E, K, seed=seed)
    inp = make_inputs(w)
    return w, inp, synth.shared_up(w, I_s, device="cuda"), synth.shared_down(w, I_s, device="cuda")


@pytest.mark.parametrize("T,H,I,E,K,I_s", [(1024, 512, 128, 4, 2, 384),   # the tiny workload
                                           (333, 256, 128, 8, 3, 200),    # T and I_s off tiles
                                           (96, 136, 72, 5, 2, 72)])      # H, I, I_s not /64
def test_shared_expert_parity(T, H, I, E, K, I_s):
    w, inp, su, sd = _case(T, H, I, E, K, I_s, seed=21)
    out = run_layer(inp, shared=(su, sd))
    assert out["status"] == _abi.MM_OK
    h = {k: v.cpu() for k, v in inp.items()}
    sh = (su.cpu(), sd.cpu())
    y = oracle.forward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"], shared=sh)
    g = oracle.backward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"], h["dy"],
                        shared=sh)
    assert_close("y", out["y"], y)
    assert_close("dx", out["dx"], g["dx"])
    assert_dtopk(out["d_topk_weights"], g["d_topk_weights"])
    assert_close("dW_up", out["dW_up"], g["dW_up"])
    assert_close("dW_down", out["dW_down"], g["dW_down"])
    assert_close("dS_up", out["dS_up"], g["dS_up"])
    assert_close("dS_down", out["dS_down"], g["dS_down"])


def test_shared_expert_leaves_the_routed_gradients_unchanged():
    """The routed experts' weight gradients and d_topk do not depend on the shared expert."""
    w, inp, su, sd = _case(300, 256, 128, 6, 2, 256, seed=5)
    a = run_layer(inp)
    b = run_layer(inp, shared=(su, sd))
    for k in ("dW_up", "dW_down", "d_topk_weights"):
        assert torch.equal(a[k], b[k]), k


def test_shared_expert_torch_autograd():
    from moe_ffn_expert_gb300.torch_api import hyper_mega_moe
    w, inp, su, sd = _case(200, 256, 128, 5, 2, 192, seed=8)
    ref = run_layer(inp, shared=(su, sd))
    x = inp["x"].clone().requires_grad_(True)
    su_t, sd_t = su.clone().requires_grad_(True), sd.clone().requires_grad_(True)
    y = hyper_mega_moe(x, inp["topk_ids"], inp["topk_weights"], inp["w_up"], inp["w_down"],
                       shared_up_proj_weight=su_t, shared_down_proj_weight=sd_t)
    y.backward(inp["dy"])
    assert torch.equal(y.detach(), ref["y"]) and torch.equal(x.grad, ref["dx"])
    assert torch.equal(su_t.grad, ref["dS_up"]) and torch.equal(sd_t.grad, ref["dS_down"])


@pytest.mark.parametrize("T,H,I,E,K,I_s", [(1200, 256, 128, 4, 2, 320),   # 10 row tiles; paired weight
                                           # gradients with odd weight row tiles (320, 640 rows)
                                           (333, 256, 128, 8, 3, 200)])   # 3 row tiles: a lone last one
def test_shared_expert_pairs_equal_single_tiles(T, H, I, E, K, I_s):
    """The shared expert's GEMMs as pair MMAs (its T rows tiled like an expert's) equal the
    one-CTA launches bit for bit."""
    w, inp, su, sd = _case(T, H, I, E, K, I_s, seed=13)
    single = _abi.MM_FLAG_SINGLE_CTA_TILES
    ref = run_layer(inp, shared=(su, sd), flags=single, bwd_flags=single)
    out = run_layer(inp, shared=(su, sd))
    assert out["status"] == _abi.MM_OK and ref["status"] == _abi.MM_OK
    for k in ("y", "dx", "d_topk_weights", "dW_up", "dW_down", "dS_up", "dS_down"):
        assert torch.equal(out[k], ref[k]), k
