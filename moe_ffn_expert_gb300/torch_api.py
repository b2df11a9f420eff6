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
        opt = _abi.options(_abi.shared_expert(shared_I, 0, 0)) if shared_I else None
        self.nbytes = _abi.mm_workspace_size_ex(self.dims, opt)
        if self.nbytes == 0:
            raise ValueError(f"unsupported sizes T={T} H={H} I={I} E={E} K={K} I_s={shared_I}")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    @classmethod
    def wrap(cls, dims, buf: torch.Tensor) -> "Workspace":
        """A Workspace over an existing buffer (one that a forward has filled)."""
        ws = cls.__new__(cls)
        ws.dims, ws.buf, ws.nbytes = dims, buf, buf.numel()
        return ws

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def _options(shared=None, tokens_per_expert=None):
    """mm_options for (shared_up, shared_down[, d_shared_up, d_shared_down]) and a tokens_per_expert
    tensor (device int32 [E]), or None when neither is given."""
    if shared is None and tokens_per_expert is None:
        return None
    se = None
    if shared is not None:
        su, sd, *grads = shared
        dsu, dsd = grads if grads else (None, None)
        se = _abi.shared_expert(sd.shape[0], _ptr(su), _ptr(sd), _ptr(dsu) if dsu is not None else 0,
                                _ptr(dsd) if dsd is not None else 0)
    return _abi.options(se, _ptr(tokens_per_expert) if tokens_per_expert is not None else 0)


def forward(ws: Workspace, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y=None,
            flags: int = 0, shared=None, tokens_per_expert=None):
    """One mm_forward(_ex) on the current stream; `shared` = (shared_up, shared_down)."""
    if y is None:
        y = torch.empty_like(x)
    st = _abi.mm_forward_ex(ws.dims, _options(shared, tokens_per_expert), _ptr(x), _ptr(topk_ids),
                            _ptr(topk_weights), _ptr(up_proj_weight), _ptr(down_proj_weight), _ptr(y),
                            ws.ptr, ws.nbytes, _stream(x.device), flags)
    _abi.check(st, "mm_forward")
    return y


def backward(ws: Workspace, dy, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
             dx=None, d_topk=None, d_up=None, d_down=None, flags: int = 0, shared=None,
             d_shared=None):
    """One mm_backward(_ex). Returns dx, d_topk, d_up, d_down (+ d_shared_up, d_shared_down)."""
    gdt = torch.float32 if flags & _abi.MM_FLAG_FP32_WEIGHT_GRADS else torch.bfloat16
    dx = torch.empty_like(x) if dx is None else dx
    d_topk = torch.empty(topk_ids.shape, dtype=torch.float32, device=x.device) if d_topk is None else d_topk
    d_up = torch.empty(up_proj_weight.shape, dtype=gdt, device=x.device) if d_up is None else d_up
    d_down = torch.empty(down_proj_weight.shape, dtype=gdt, device=x.device) if d_down is None else d_down
    if shared is not None and d_shared is None:
        d_shared = tuple(torch.empty(t.shape, dtype=gdt, device=x.device) for t in shared)
    opt = _options((*shared, *d_shared) if shared is not None else None)
    st = _abi.mm_backward_ex(ws.dims, opt, _ptr(dy), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                             _ptr(up_proj_weight), _ptr(down_proj_weight), ws.ptr, ws.nbytes,
                             _ptr(dx), _ptr(d_topk), _ptr(d_up), _ptr(d_down), _stream(x.device),
                             flags)
    _abi.check(st, "mm_backward")
    if shared is not None:
        return dx, d_topk, d_up, d_down, d_shared[0], d_shared[1]
    return dx, d_topk, d_up, d_down


class HyperMegaMoEFunction(torch.autograd.Function):
    """Forward and backward of the layer (RFC §3.2); optional shared expert (RFC §6.1) and
    caller histogram (usage guide, tokens_per_expert)."""

    @staticmethod
    def forward(ctx, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, shared_up,
                shared_down, tokens_per_expert):
        T, H, I, E, K = check_inputs(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)
        shared = None
        I_s = 0
        if shared_up is not None:
            I_s = shared_down.shape[0]
            if shared_up.shape != (H, 2 * I_s) or shared_down.shape != (I_s, H):
                raise ValueError("expected shared_up_proj_weight[H,2I_s], shared_down_proj_weight[I_s,H]")
            if shared_up.dtype != torch.bfloat16 or shared_down.dtype != torch.bfloat16:
                raise TypeError("shared-expert weights must be bfloat16")
            shared = (shared_up.contiguous(), shared_down.contiguous())
        tpe = None
        if tokens_per_expert is not None:
            if tokens_per_expert.shape != (E,) or tokens_per_expert.device != x.device:
                raise ValueError("tokens_per_expert must be a [E] tensor on x's device")
            tpe = tokens_per_expert.to(torch.int32).contiguous()
        x = x.contiguous()
        ids = topk_ids.to(torch.int32).contiguous()
        w = topk_weights.to(torch.float32).contiguous()
        wu, wd = up_proj_weight.contiguous(), down_proj_weight.contiguous()
        ws = Workspace(T, H, I, E, K, x.device, shared_I=I_s)
        # with a caller histogram the id and histogram checks are waited for, so that a mismatch
        # raises here instead of leaving y unspecified
        flags = _abi.MM_FLAG_VALIDATE_IDS if tpe is not None else 0
        if not any(ctx.needs_input_grad):  # inference (no_grad or no input needs a gradient)
            flags |= _abi.MM_FLAG_FORWARD_ONLY
        y = forward(ws, x, ids, w, wu, wd, flags=flags, shared=shared, tokens_per_expert=tpe)
        ctx.dims = ws.dims
        ctx.wdtype = topk_weights.dtype
        ctx.has_shared = shared is not None
        # the workspace is saved like any other tensor: autograd frees it after the backward,
        # or keeps it for another one under retain_graph (a backward only reads what the
        # forward left in it)
        kept = (ws.buf,) if any(ctx.needs_input_grad) else ()
        ctx.save_for_backward(x, ids, w, wu, wd, *(shared or ()), *kept)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, ids, w, wu, wd, *rest = ctx.saved_tensors
        *shared, buf = rest
        ws = Workspace.wrap(ctx.dims, buf)
        out = backward(ws, dy.contiguous().to(torch.bfloat16), x, ids, w, wu, wd,
                       shared=tuple(shared) if ctx.has_shared else None)
        dx, d_topk, d_up, d_down = out[:4]
        ds_up, ds_down = out[4:] if ctx.has_shared else (None, None)
        return dx, None, d_topk.to(ctx.wdtype), d_up, d_down, ds_up, ds_down, None


def hyper_mega_moe(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, *,
                   shared_up_proj_weight=None, shared_down_proj_weight=None,
                   tokens_per_expert=None):
    """y[T,H] = sum_k topk_weights[t,k] * SwiGLU-FFN_{topk_ids[t,k]}(x[t])
    (+ SwiGLU-FFN_shared(x[t]) when the keyword-only shared-expert weights are given).

    tokens_per_expert (optional, [E] on x's device, int32 used as is, int64 or non-contiguous
    converted) is the caller's histogram of topk_ids; the layer checks it against its own (one
    host wait) and raises MMError(MM_ERR_TOKENS_PER_EXPERT) if they differ."""
    if (shared_up_proj_weight is None) != (shared_down_proj_weight is None):
        raise ValueError("give both shared-expert weights or neither")
    return HyperMegaMoEFunction.apply(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                                      shared_up_proj_weight, shared_down_proj_weight,
                                      tokens_per_expert)
