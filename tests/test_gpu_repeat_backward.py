"""Several backwards after one forward: mm_backward reads only what mm_forward kept in the
workspace (routing, dispatched x rows, gate|up), so a second call with another dy, and autograd's
retain_graph, give what a fresh forward + backward gives, bit for bit."""
import pytest
import torch

from layer_harness import make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu

GRADS = ("dx", "d_topk_weights", "dW_up", "dW_down")


def _other_dy(dy, seed):
    g = torch.Generator(device=dy.device).manual_seed(seed)
    return torch.randn(dy.shape, generator=g, device=dy.device).to(torch.bfloat16)


def _backward_only(inp, out, dy, shared=None):
    """One more mm_backward(_ex) on the workspace `out` was left with (by run_layer)."""
    x, ids, tw, wu, wd = inp["x"], inp["topk_ids"], inp["topk_weights"], inp["w_up"], inp["w_down"]
    res = dict(dx=torch.empty_like(x), d_topk_weights=torch.empty(ids.shape, dtype=torch.float32,
                                                                   device=x.device),
               dW_up=torch.empty_like(wu), dW_down=torch.empty_like(wd))
    ws = out["ws"]
    st = torch.cuda.current_stream().cuda_stream
    args = (dy.data_ptr(), x.data_ptr(), ids.data_ptr(), tw.data_ptr(), wu.data_ptr(),
            wd.data_ptr(), ws.data_ptr(), ws.numel(), res["dx"].data_ptr(),
            res["d_topk_weights"].data_ptr(), res["dW_up"].data_ptr(), res["dW_down"].data_ptr(),
            st, 0)
    if shared is None:
        _abi.check(_abi.mm_backward(out["dims"], *args), "mm_backward")
    else:
        su, sd = shared
        res.update(dS_up=torch.empty_like(su), dS_down=torch.empty_like(sd))
        se = _abi.shared_expert(sd.shape[0], su.data_ptr(), sd.data_ptr(),
                                res["dS_up"].data_ptr(), res["dS_down"].data_ptr())
        _abi.check(_abi.mm_backward_ex(out["dims"], _abi.options(se), *args), "mm_backward_ex")
    assert _abi.mm_get_status(ws.data_ptr(), st) == _abi.MM_OK
    return res


@pytest.mark.parametrize("T,H,I,E,K,I_s", [(700, 256, 128, 6, 2, 0),     # lone pair halves, tails
                                           (1536, 256, 128, 4, 2, 0),    # paired weight gradients
                                           (333, 256, 128, 8, 3, 200)])  # with a shared expert
def test_second_backward_equals_a_fresh_step(T, H, I, E, K, I_s):
    w = synth.small("rb", T, H, I, E, K, seed=17)
    inp = make_inputs(w)
    shared = (synth.shared_up(w, I_s, device="cuda"), synth.shared_down(w, I_s, device="cuda")) \
        if I_s else None
    inp2 = dict(inp, dy=_other_dy(inp["dy"], 3))
    ref1 = run_layer(inp, shared=shared)
    ref2 = run_layer(inp2, shared=shared)
    keys = GRADS + (("dS_up", "dS_down") if shared else ())
    out = run_layer(inp, shared=shared)  # forward + backward with dy, then two more backwards
    assert out["status"] == _abi.MM_OK
    again2 = _backward_only(inp, out, inp2["dy"], shared)
    again1 = _backward_only(inp, out, inp["dy"], shared)
    for k in keys:
        assert torch.equal(again2[k], ref2[k]), k
        assert torch.equal(again1[k], ref1[k]), k
    assert not torch.equal(ref1["dx"], ref2["dx"])


def test_autograd_retain_graph():
    """y.backward(dy1, retain_graph=True) then, with the gradients cleared, y.backward(dy2):
    each gives a fresh step's gradients; after the second the graph, workspace included, is
    freed and a third backward raises."""
    from moe_ffn_expert_gb300.torch_api import hyper_mega_moe
    w = synth.small("rg", 300, 256, 128, 6, 2, seed=9)
    inp = make_inputs(w)
    dy2 = _other_dy(inp["dy"], 4)
    ref1 = run_layer(inp)
    ref2 = run_layer(dict(inp, dy=dy2))
    x = inp["x"].clone().requires_grad_(True)
    tw = inp["topk_weights"].clone().requires_grad_(True)
    wu = inp["w_up"].clone().requires_grad_(True)
    wd = inp["w_down"].clone().requires_grad_(True)
    y = hyper_mega_moe(x, inp["topk_ids"], tw, wu, wd)
    y.backward(inp["dy"], retain_graph=True)
    first = {k: t.grad.clone() for k, t in (("dx", x), ("d_topk_weights", tw), ("dW_up", wu),
                                             ("dW_down", wd))}
    for k in GRADS:
        assert torch.equal(first[k], ref1[k]), k
    for t in (x, tw, wu, wd):
        t.grad = None
    y.backward(dy2)
    for k, t in (("dx", x), ("d_topk_weights", tw), ("dW_up", wu), ("dW_down", wd)):
        assert torch.equal(t.grad, ref2[k]), k
    with pytest.raises(RuntimeError):
        y.backward(inp["dy"])
