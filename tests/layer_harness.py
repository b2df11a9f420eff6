"""Shared helpers of the GPU tests: build inputs, run the layer through the C ABI, compare
with the oracle under the stated tolerances."""
from __future__ import annotations

import torch

from moe_ffn_expert_gb300 import _abi
from workloads import synth

# |gpu - oracle| <= ATOL + RTOL * |oracle| for y, dx and the weight gradients;
# d_topk_weights: |gpu - oracle| <= DTOPK_REL * max(|oracle|, rms(oracle)).
ATOL = 1e-2
RTOL = 1e-2
DTOPK_REL = 2e-2


def make_inputs(w: synth.Workload, device="cuda", ids=None):
    """Seeded inputs of workload `w`, on `device` (routing drawn on the host)."""
    ids = synth.routing(w) if ids is None else ids
    return dict(
        x=synth.x(w, device=device),
        topk_ids=ids.to(device),
        topk_weights=synth.topk_weights(w).to(device),
        w_up=synth.w_up(w, device=device),
        w_down=synth.w_down(w, device=device),
        dy=synth.dy(w, device=device),
    )


def run_layer(inp, flags=0, ws=None, stream=None, backward=True, bwd_flags=0, d_up=None,
              d_down=None, shared=None, tokens_per_expert=None, ds_up=None, ds_down=None):
    """Forward (+ backward) through the C ABI; returns device tensors and the workspace.

    d_up/d_down (and ds_up/ds_down for a shared expert), when given, are the weight-gradient
    output buffers: their contents matter with MM_FLAG_ACCUMULATE_WEIGHT_GRADS, and they must be
    fp32 with MM_FLAG_FP32_WEIGHT_GRADS. `shared` = (shared_up [H, 2I_s], shared_down [I_s, H])
    and `tokens_per_expert` (device int32 [E]) go through mm_forward_ex / mm_backward_ex."""
    x, ids, tw = inp["x"], inp["topk_ids"], inp["topk_weights"]
    wu, wd = inp["w_up"], inp["w_down"]
    T, H = x.shape
    E, _, I2 = wu.shape
    K = ids.shape[1]
    d = _abi.dims(T, H, I2 // 2, E, K)
    gdt = torch.float32 if bwd_flags & _abi.MM_FLAG_FP32_WEIGHT_GRADS else torch.bfloat16
    ex = shared is not None or tokens_per_expert is not None
    se = opt = None
    if shared is not None:
        su, sd = shared
        ds_up = torch.empty(su.shape, dtype=gdt, device=x.device) if ds_up is None else ds_up
        ds_down = torch.empty(sd.shape, dtype=gdt, device=x.device) if ds_down is None else ds_down
        se = _abi.shared_expert(sd.shape[0], su.data_ptr(), sd.data_ptr(), ds_up.data_ptr(),
                                ds_down.data_ptr())
    if ex:
        opt = _abi.options(se, tokens_per_expert.data_ptr() if tokens_per_expert is not None else 0)
    nbytes = _abi.mm_workspace_size_ex(d, opt) if ex else _abi.mm_workspace_size(d)
    assert nbytes > 0
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    st = (stream or torch.cuda.current_stream()).cuda_stream
    y = torch.empty_like(x)
    fargs = (x.data_ptr(), ids.data_ptr(), tw.data_ptr(), wu.data_ptr(), wd.data_ptr(),
             y.data_ptr(), ws.data_ptr(), nbytes, st, flags)
    if ex:
        _abi.check(_abi.mm_forward_ex(d, opt, *fargs), "mm_forward_ex")
    else:
        _abi.check(_abi.mm_forward(d, *fargs), "mm_forward")
    out = dict(y=y, ws=ws, dims=d)
    if backward:
        dx = torch.empty_like(x)
        d_topk = torch.empty(T, K, dtype=torch.float32, device=x.device)
        d_up = torch.empty(wu.shape, dtype=gdt, device=x.device) if d_up is None else d_up
        d_down = torch.empty(wd.shape, dtype=gdt, device=x.device) if d_down is None else d_down
        bargs = (inp["dy"].data_ptr(), x.data_ptr(), ids.data_ptr(), tw.data_ptr(), wu.data_ptr(),
                 wd.data_ptr(), ws.data_ptr(), nbytes, dx.data_ptr(), d_topk.data_ptr(),
                 d_up.data_ptr(), d_down.data_ptr(), st, bwd_flags)
        if ex:
            _abi.check(_abi.mm_backward_ex(d, opt, *bargs), "mm_backward_ex")
        else:
            _abi.check(_abi.mm_backward(d, *bargs), "mm_backward")
        out.update(dx=dx, d_topk_weights=d_topk, dW_up=d_up, dW_down=d_down)
        if shared is not None:
            out.update(dS_up=ds_up, dS_down=ds_down)
    out["status"] = _abi.mm_get_status(ws.data_ptr(), st)
    return out


def export_routing(out, E, S):
    counts = torch.empty(E, dtype=torch.int32)
    offsets = torch.empty(E + 1, dtype=torch.int32)
    rows = torch.empty(S, dtype=torch.int32)
    _abi.check(_abi.mm_routing_export(out["dims"], out["ws"].data_ptr(), counts.data_ptr(),
                                      offsets.data_ptr(), rows.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream), "mm_routing_export")
    return counts, offsets, rows


def assert_close(name, got, ref, atol=ATOL, rtol=RTOL):
    got = got.detach().to("cpu", torch.float64)
    ref = ref.to(torch.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{name}: non-finite values"
    err = (got - ref).abs()
    bound = atol + rtol * ref.abs()
    bad = err > bound
    if bad.any():
        i = int(torch.argmax((err - bound).reshape(-1)))
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.numel()} elements outside |d| <= {atol} + {rtol}|ref|; "
            f"worst flat index {i}: got {got.reshape(-1)[i].item():.6g} ref {ref.reshape(-1)[i].item():.6g}; "
            f"max abs err {err.max().item():.3g}")


def assert_dtopk(got, ref, rel=DTOPK_REL):
    got = got.detach().to("cpu", torch.float64)
    ref = ref.to(torch.float64)
    rms = ref.pow(2).mean().sqrt()
    bound = rel * torch.maximum(ref.abs(), rms)
    err = (got - ref).abs()
    bad = err > bound
    assert not bad.any(), (f"d_topk_weights: {int(bad.sum())} of {bad.numel()} outside "
                           f"{rel}*max(|ref|, rms); max err {err.max().item():.3g}")
