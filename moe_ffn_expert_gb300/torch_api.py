"""PyTorch entry points over the C ABI: torch supplies device memory and the current stream.

`hyper_mega_moe(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)` follows the
public call of the RFC "HyperParallel Multicore HyperMegaMoE fused forward/backward operator"
(§3.1 Python API, §3.2 autograd semantics): it returns y[T,H] and its backward returns
gradients for x, topk_weights and both expert weights (None for topk_ids).
Argument marshalling only: int64 or non-contiguous inputs are converted (as the multicore
usage guide describes for tokens_per_expert/ids), everything else runs in libmm.so.
"""
from __future__ import annotations

import torch

from . import _abi


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def check_inputs(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight):
    if not x.is_cuda:
        raise ValueError("hyper_mega_moe runs on a CUDA device only (no CPU path)")
    if x.dim() != 2 or topk_ids.dim() != 2 or topk_weights.shape != topk_ids.shape:
        raise ValueError("expected x[T,H], topk_ids[T,K], topk_weights[T,K]")
    T, H = x.shape
    E, H2, I2 = up_proj_weight.shape
    if H2 != H or I2 % 2 or down_proj_weight.shape != (E, I2 // 2, H) or topk_ids.shape[0] != T:
        raise ValueError("expected up_proj_weight[E,H,2I] and down_proj_weight[E,I,H]")
    for name, t in (("x", x), ("up_proj_weight", up_proj_weight), ("down_proj_weight", down_proj_weight)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
    if not topk_weights.is_floating_point():
        raise TypeError("topk_weights must be floating point")
    if topk_ids.dtype not in (torch.int32, torch.int64):
        raise TypeError("topk_ids must be int32 or int64")
    return T, H, I2 // 2, E, topk_ids.shape[1]


class Workspace:
    """A caller-owned workspace buffer for one pending forward/backward pair (with room for a
    shared expert of intermediate size shared_I when given)."""

    def __init__(self, T, H, I, E, K, device, shared_I=0):
        self.dims = _abi.dims(T, H, I, E, K)
        self.nbytes = (_abi.mm_workspace_size_se(self.dims, shared_I) if shared_I
                       else _abi.mm_workspace_size(self.dims))
        if self.nbytes == 0:
            raise ValueError(f"unsupported sizes T={T} H={H} I={I} E={E} K={K}")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def forward(ws: Workspace, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y=None,
            flags: int = 0):
    if y is None:
        y = torch.empty_like(x)
    st = _abi.mm_forward(ws.dims, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(up_proj_weight),
                         _ptr(down_proj_weight), _ptr(y), ws.ptr, ws.nbytes, _stream(x.device), flags)
    _abi.check(st, "mm_forward")
    return y


def backward(ws: Workspace, dy, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
             dx=None, d_topk=None, d_up=None, d_down=None):
    dx = torch.empty_like(x) if dx is None else dx
    d_topk = torch.empty(topk_ids.shape, dtype=torch.float32, device=x.device) if d_topk is None else d_topk
    d_up = torch.empty_like(up_proj_weight) if d_up is None else d_up
    d_down = torch.empty_like(down_proj_weight) if d_down is None else d_down
    st = _abi.mm_backward(ws.dims, _ptr(dy), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                          _ptr(up_proj_weight), _ptr(down_proj_weight), ws.ptr, ws.nbytes, _ptr(dx),
                          _ptr(d_topk), _ptr(d_up), _ptr(d_down), _stream(x.device), 0)
    _abi.check(st, "mm_backward")
    return dx, d_topk, d_up, d_down


class HyperMegaMoESharedFunction(torch.autograd.Function):
    """The same with a shared expert (RFC §6.1): an always-on SwiGLU FFN merged at the combine."""

    @staticmethod
    def forward(ctx, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, shared_up,
                shared_down):
        T, H, I, E, K = check_inputs(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)
        I_s = shared_down.shape[0]
        if shared_up.shape != (H, 2 * I_s) or shared_down.shape != (I_s, H):
            raise ValueError("expected shared_up_proj_weight[H,2I_s], shared_down_proj_weight[I_s,H]")
        x = x.contiguous()
        ids = topk_ids.to(torch.int32).contiguous()
        w = topk_weights.to(torch.float32).contiguous()
        wu, wd = up_proj_weight.contiguous(), down_proj_weight.contiguous()
        su, sd = shared_up.contiguous(), shared_down.contiguous()
        ws = Workspace(T, H, I, E, K, x.device, shared_I=I_s)
        y = torch.empty_like(x)
        se = _abi.shared_expert(I_s, _ptr(su), _ptr(sd))
        _abi.check(_abi.mm_forward_se(ws.dims, se, _ptr(x), _ptr(ids), _ptr(w), _ptr(wu), _ptr(wd),
                                      _ptr(y), ws.ptr, ws.nbytes, _stream(x.device), 0),
                   "mm_forward_se")
        ctx.ws = ws
        ctx.wdtype = topk_weights.dtype
        ctx.save_for_backward(x, ids, w, wu, wd, su, sd)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, ids, w, wu, wd, su, sd = ctx.saved_tensors
        dy = dy.contiguous().to(torch.bfloat16)
        dx, d_topk = torch.empty_like(x), torch.empty(ids.shape, dtype=torch.float32, device=x.device)
        d_up, d_down = torch.empty_like(wu), torch.empty_like(wd)
        ds_up, ds_down = torch.empty_like(su), torch.empty_like(sd)
        se = _abi.shared_expert(sd.shape[0], _ptr(su), _ptr(sd), _ptr(ds_up), _ptr(ds_down))
        ws = ctx.ws
        _abi.check(_abi.mm_backward_se(ws.dims, se, _ptr(dy), _ptr(x), _ptr(ids), _ptr(w), _ptr(wu),
                                       _ptr(wd), ws.ptr, ws.nbytes, _ptr(dx), _ptr(d_topk),
                                       _ptr(d_up), _ptr(d_down), _stream(x.device), 0),
                   "mm_backward_se")
        ctx.ws = None
        return dx, None, d_topk.to(ctx.wdtype), d_up, d_down, ds_up, ds_down


class HyperMegaMoEFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight):
        T, H, I, E, K = check_inputs(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)
        x = x.contiguous()
        ids = topk_ids.to(torch.int32).contiguous()
        w = topk_weights.to(torch.float32).contiguous()
        wu, wd = up_proj_weight.contiguous(), down_proj_weight.contiguous()
        ws = Workspace(T, H, I, E, K, x.device)
        y = forward(ws, x, ids, w, wu, wd)
        ctx.ws = ws
        ctx.wdtype = topk_weights.dtype
        ctx.save_for_backward(x, ids, w, wu, wd)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, ids, w, wu, wd = ctx.saved_tensors
        dx, d_topk, d_up, d_down = backward(ctx.ws, dy.contiguous().to(torch.bfloat16), x, ids, w, wu, wd)
        ctx.ws = None
        return dx, None, d_topk.to(ctx.wdtype), d_up, d_down


def hyper_mega_moe(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, *,
                   shared_up_proj_weight=None, shared_down_proj_weight=None):
    """y[T,H] = sum_k topk_weights[t,k] * SwiGLU-FFN_{topk_ids[t,k]}(x[t])
    (+ SwiGLU-FFN_shared(x[t]) when the keyword-only shared-expert weights are given)."""
    if (shared_up_proj_weight is None) != (shared_down_proj_weight is None):
        raise ValueError("give both shared-expert weights or neither")
    if shared_up_proj_weight is not None:
        return HyperMegaMoESharedFunction.apply(x, topk_ids, topk_weights, up_proj_weight,
                                                down_proj_weight, shared_up_proj_weight,
                                                shared_down_proj_weight)
    return HyperMegaMoEFunction.apply(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)
