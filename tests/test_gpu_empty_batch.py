"""An empty batch (T = 0) through the C ABI and the torch entry point: the forward leaves empty
routing tables, the backward writes exact zeros into the weight gradients (or leaves them as
they are when accumulating), and a caller histogram must be all zero."""
import pytest
import torch

from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu


def _weights(H=256, I=128, E=6, I_s=0):
    w = synth.small("empty", 8, H, I, E, 2, seed=3)
    out = dict(wu=synth.w_up(w, device="cuda"), wd=synth.w_down(w, device="cuda"))
    if I_s:
        out.update(su=synth.shared_up(w, I_s, device="cuda"), sd=synth.shared_down(w, I_s, device="cuda"))
    return out


@pytest.mark.parametrize("flags", [0, _abi.MM_FLAG_FP32_WEIGHT_GRADS,
                                   _abi.MM_FLAG_ACCUMULATE_WEIGHT_GRADS])
@pytest.mark.parametrize("I_s", [0, 192])
def test_empty_batch_c_abi(flags, I_s):
    H, I, E, K = 256, 128, 6, 2
    wts = _weights(H, I, E, I_s)
    d = _abi.dims(0, H, I, E, K)
    se = _abi.shared_expert(I_s, wts["su"].data_ptr(), wts["sd"].data_ptr()) if I_s else None
    opt = _abi.options(se) if I_s else None
    n = _abi.mm_workspace_size_ex(d, opt)
    assert n > 0
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")  # poisoned
    st = torch.cuda.current_stream().cuda_stream
    wu, wd = wts["wu"], wts["wd"]
    assert _abi.mm_forward_ex(d, opt, 0, 0, 0, wu.data_ptr(), wd.data_ptr(), 0, ws.data_ptr(), n,
                              st, 0) == _abi.MM_OK
    assert _abi.mm_get_status(ws.data_ptr(), st) == _abi.MM_OK
    counts = torch.full((E,), -7, dtype=torch.int32)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32)
    assert _abi.mm_routing_export(d, ws.data_ptr(), counts.data_ptr(), offsets.data_ptr(),
                                  0, st) == _abi.MM_OK
    assert counts.eq(0).all() and offsets.eq(0).all()
    gdt = torch.float32 if flags & _abi.MM_FLAG_FP32_WEIGHT_GRADS else torch.bfloat16
    base = {k: torch.randn(t.shape, device="cuda").to(gdt) for k, t in wts.items()}
    grads = {k: v.clone() for k, v in base.items()}
    if I_s:
        se_b = _abi.shared_expert(I_s, wts["su"].data_ptr(), wts["sd"].data_ptr(),
                                  grads["su"].data_ptr(), grads["sd"].data_ptr())
        opt = _abi.options(se_b)
    assert _abi.mm_backward_ex(d, opt, 0, 0, 0, 0, wu.data_ptr(), wd.data_ptr(), ws.data_ptr(), n,
                               0, 0, grads["wu"].data_ptr(), grads["wd"].data_ptr(), st,
                               flags) == _abi.MM_OK
    torch.cuda.synchronize()
    for k in grads:
        if flags & _abi.MM_FLAG_ACCUMULATE_WEIGHT_GRADS:
            assert torch.equal(grads[k], base[k]), k
        else:
            assert grads[k].eq(0).all(), k


def test_empty_batch_tokens_per_expert():
    H, I, E, K = 256, 128, 6, 2
    wts = _weights(H, I, E)
    d = _abi.dims(0, H, I, E, K)
    st = torch.cuda.current_stream().cuda_stream
    for tpe, expect in ((torch.zeros(E, dtype=torch.int32, device="cuda"), _abi.MM_OK),
                        (torch.tensor([0, 0, 1, 0, 0, 0], dtype=torch.int32, device="cuda"),
                         _abi.MM_ERR_TOKENS_PER_EXPERT)):
        opt = _abi.options(None, tpe.data_ptr())
        n = _abi.mm_workspace_size_ex(d, opt)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        args = (d, opt, 0, 0, 0, wts["wu"].data_ptr(), wts["wd"].data_ptr(), 0, ws.data_ptr(), n, st)
        assert _abi.mm_forward_ex(*args, 0) == _abi.MM_OK
        assert _abi.mm_get_status(ws.data_ptr(), st) == expect
        assert _abi.mm_forward_ex(*args, _abi.MM_FLAG_VALIDATE_IDS) == expect


def test_empty_batch_backward_after_forward_only():
    """A backward on the workspace of a forward-only empty batch is refused through the status
    word, as it is for T > 0; after a training forward the same workspace is accepted again."""
    H, I, E, K = 256, 128, 6, 2
    wts = _weights(H, I, E)
    d = _abi.dims(0, H, I, E, K)
    n = _abi.mm_workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    wu, wd = wts["wu"], wts["wd"]
    du, dd = torch.empty_like(wu), torch.empty_like(wd)
    for fflags, expect in ((_abi.MM_FLAG_FORWARD_ONLY, _abi.MM_ERR_INVALID_ARG), (0, _abi.MM_OK)):
        for bflags in (0, _abi.MM_FLAG_ACCUMULATE_WEIGHT_GRADS):
            assert _abi.mm_forward(d, 0, 0, 0, wu.data_ptr(), wd.data_ptr(), 0, ws.data_ptr(), n,
                                   st, fflags) == _abi.MM_OK
            assert _abi.mm_backward(d, 0, 0, 0, 0, wu.data_ptr(), wd.data_ptr(), ws.data_ptr(), n,
                                    0, 0, du.data_ptr(), dd.data_ptr(), st, bflags) == _abi.MM_OK
            assert _abi.mm_get_status(ws.data_ptr(), st) == expect, (fflags, bflags)


def test_empty_batch_noalloc_routing():
    E = 5
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert _abi.mm_route_noalloc(_abi.dims(0, 64, 64, E, 2), 0, counts.data_ptr(),
                                 offsets.data_ptr(), 0, st) == _abi.MM_OK
    torch.cuda.synchronize()
    assert counts.eq(0).all() and offsets.eq(0).all()


def test_empty_batch_torch_autograd():
    from moe_ffn_expert_gb300.torch_api import hyper_mega_moe
    H, I, E, K = 256, 128, 6, 2
    wts = _weights(H, I, E)
    x = torch.empty(0, H, dtype=torch.bfloat16, device="cuda", requires_grad=True)
    ids = torch.empty(0, K, dtype=torch.int64, device="cuda")
    tw = torch.empty(0, K, dtype=torch.float32, device="cuda", requires_grad=True)
    wu = wts["wu"].clone().requires_grad_(True)
    wd = wts["wd"].clone().requires_grad_(True)
    y = hyper_mega_moe(x, ids, tw, wu, wd)
    assert y.shape == (0, H)
    y.backward(torch.empty(0, H, dtype=torch.bfloat16, device="cuda"))
    assert x.grad.shape == (0, H) and tw.grad.shape == (0, K)
    assert wu.grad.eq(0).all() and wd.grad.eq(0).all()
