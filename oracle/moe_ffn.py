"""CPU oracle for the fused MoE-FFN forward and backward (HyperMegaMoE / HyperMegaMoEGrad).

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this module: only the test suite, the smoke check and the
benchmark's CPU-baseline leg use it. It shares no code with the CUDA path.

What it computes is the plain, unfused definition of the layer, written out
step by step in float64 from the (bf16-rounded) inputs, with no intermediate
rounding, no blocking and no fusion. Library primitives used as steps:
torch.bincount, torch.cumsum, a stable torch.argsort, torch.matmul, torch.sigmoid.

Sources (page titles and sections):
* "HyperParallel Multicore HyperMegaMoE fused forward/backward operator" RFC:
  - §2.1 forward chain Dispatch -> GMM1 (up_proj) -> SwiGLU -> GMM2 (down_proj) -> Combine;
  - §2.2 backward graph: dispatch dY, act_grad dHidden = dY_slot W2^T, SwiGLUGrad,
    input_grad GMM, W2Grad, W1Grad, Combine(dX); gradient list dx, d_up_proj_weight,
    d_down_proj_weight, d_topk_weights;
  - §3.1 tensor shapes x[T,H], topk_ids[T,K], topk_weights[T,K],
    up_proj_weight[E,H,2I], down_proj_weight[E,I,H];
  - §4.1 each token expands into K expert slots; combine is the topk_weights-weighted merge;
  - §4.2 the activation is SwiGLU.
* "MoE multicore parallel usage guide" (hyper_parallel/core/multicore), "inputs and
  weights": gate and up are concatenated on the last dim of up_proj_weight.

Readings where the pages leave a step open (each is also pinned by a test):
* gate = up_proj_weight[e][:, :I], up = up_proj_weight[e][:, I:];
* SwiGLU(g, u) = silu(g) * u with silu(z) = z * sigmoid(z), no bias, clamp or scale;
* the routing weight enters only at the combine: y[t] = sum_k w[t,k] * o[slot t*K+k];
* expert-sorted order is stable in the slot index s = t*K + k;
* d_topk_weights[t,k] = <dy[t], o[t*K+k]>.

Parity: every function here is pinned by the "not gpu" tests (closed forms,
a hand-derived scalar case, brute-force routing, a dense special case checked
against torch's own SwiGLU, and float64 finite differences).
"""
from __future__ import annotations

import torch

F64 = torch.float64


# ------------------------------------------------------------------ routing (RFC §3.3, §4.1)

def route(topk_ids: torch.Tensor, E: int):
    """Routing preprocessing.

    Slots are s = t*K + k. Returns
      counts[e]       number of slots routed to expert e           (int64 [E])
      offsets[e]      exclusive prefix sum of counts, offsets[E]=S  (int64 [E+1])
      row_of_slot[s]  position of slot s in the expert-sorted order (int64 [S])
      slot_of_row[r]  inverse permutation                           (int64 [S])
    The expert-sorted order groups slots by expert, ascending in s within an
    expert, so row_of_slot[s] = offsets[e] + #{s' < s : ids[s'] == e}.
    """
    flat = topk_ids.reshape(-1).to(torch.int64)
    S = flat.numel()
    if S and (int(flat.min()) < 0 or int(flat.max()) >= E):
        raise ValueError("expert id out of range")
    counts = torch.bincount(flat, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    slot_of_row = torch.argsort(flat, stable=True)
    row_of_slot = torch.empty(S, dtype=torch.int64)
    row_of_slot[slot_of_row] = torch.arange(S)
    return counts, offsets, row_of_slot, slot_of_row


def dispatch(rows_src: torch.Tensor, slot_of_row: torch.Tensor, K: int) -> torch.Tensor:
    """Dispatch (single device: a gather into expert order): row r takes token slot_of_row[r] // K."""
    return rows_src[slot_of_row // K]


def combine(rows: torch.Tensor, row_of_slot: torch.Tensor, weights, T: int, K: int) -> torch.Tensor:
    """Combine: out[t] = sum over k of weights[t,k] * rows[row_of_slot[t*K+k]].
    `weights=None` is the unweighted sum (the gradient combine)."""
    per_slot = rows[row_of_slot].reshape(T, K, -1)
    if weights is not None:
        per_slot = per_slot * weights.to(F64).reshape(T, K, 1)
    return per_slot.sum(1)


# ------------------------------------------------------------------ SwiGLU (RFC §4.2)

def silu(z: torch.Tensor) -> torch.Tensor:
    return z * torch.sigmoid(z)


def swiglu(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    return silu(gate) * up


def swiglu_grad(d_h: torch.Tensor, gate: torch.Tensor, up: torch.Tensor):
    """d/dgate and d/dup of silu(gate)*up given the upstream gradient d_h.
    silu'(z) = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    sg = torch.sigmoid(gate)
    d_gate = d_h * up * sg * (1.0 + gate * (1.0 - sg))
    d_up = d_h * (gate * sg)
    return d_gate, d_up


def _as64(t):
    return t.to(F64)


# ------------------------------------------------------------------ forward (RFC §2.1)

def expert_forward(X: torch.Tensor, w_up_e: torch.Tensor, w_down_e: torch.Tensor):
    """GMM1 -> SwiGLU -> GMM2 for the rows X of one expert. Returns (gate, up, h, o)."""
    I = w_up_e.shape[1] // 2
    W1 = _as64(w_up_e)
    gate = X @ W1[:, :I]
    up = X @ W1[:, I:]
    h = swiglu(gate, up)
    o = h @ _as64(w_down_e)
    return gate, up, h, o


def shared_expert_forward(x, shared_up, shared_down):
    """The shared expert of the RFC's optional shared-expert fusion (§6.1): one SwiGLU FFN
    applied to every token, whose output the combine adds with weight 1.
    shared_up [H, 2*I_s] (gate | up), shared_down [I_s, H]."""
    _, _, _, o = expert_forward(_as64(x), shared_up, shared_down)
    return o


def forward(x, topk_ids, topk_weights, w_up, w_down, return_saved=False, shared=None):
    """y[T,H] = combine(GMM2(SwiGLU(GMM1(dispatch(x))))) (+ the shared expert's output).

    `w_up` / `w_down` only need `[e]` indexing (a [E,...] tensor or a lazy
    per-expert source). Experts with no slots are never touched. `shared`, when given, is a
    (shared_up, shared_down) pair (RFC §6.1)."""
    T, H = x.shape
    K = topk_ids.shape[1]
    E = w_up.shape[0]
    counts, offsets, row_of_slot, slot_of_row = route(topk_ids, E)
    x_rows = dispatch(_as64(x), slot_of_row, K)
    o_rows = torch.zeros(T * K, H, dtype=F64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        _, _, _, o = expert_forward(x_rows[r0:r1], w_up[e], w_down[e])
        o_rows[r0:r1] = o
    y = combine(o_rows, row_of_slot, topk_weights, T, K)
    if shared is not None:
        y = y + shared_expert_forward(x, *shared)
    if return_saved:
        return y, dict(counts=counts, offsets=offsets, row_of_slot=row_of_slot,
                       slot_of_row=slot_of_row, o_rows=o_rows)
    return y


# ------------------------------------------------------------------ backward (RFC §2.2)

def expert_backward(X, dY, w, w_up_e, w_down_e):
    """Backward for the rows of one expert.

    X, dY: the dispatched token rows and upstream rows (unweighted); w: the
    routing weight of each row. The gradient reaching the expert output is
    dO = w * dY (combine's backward). Returns dict with the expert output o,
    d_topk per row <dY, o>, dX rows (before the combine), dW_up[e], dW_down[e].
    """
    I = w_up_e.shape[1] // 2
    W1 = _as64(w_up_e)
    W2 = _as64(w_down_e)
    gate, up, h, o = expert_forward(X, w_up_e, w_down_e)
    d_topk = (dY * o).sum(1)
    dO = w[:, None] * dY
    d_h = dO @ W2.T                      # act_grad
    d_gate, d_up = swiglu_grad(d_h, gate, up)
    d_gu = torch.cat([d_gate, d_up], 1)
    return dict(
        o=o,
        d_topk=d_topk,
        dx_rows=d_gu @ W1.T,             # input_grad
        dW_down=h.T @ dO,                # W2Grad
        dW_up=X.T @ d_gu,                # W1Grad
        I=I,
    )


def backward(x, topk_ids, topk_weights, w_up, w_down, dy, shared=None):
    """All gradients of sum(y * dy): dx[T,H], d_topk_weights[T,K], dW_up[E,H,2I], dW_down[E,I,H]
    (and, with a shared expert, dS_up[H,2I_s], dS_down[I_s,H]: its rows are all tokens with
    weight 1)."""
    T, H = x.shape
    K = topk_ids.shape[1]
    E = w_up.shape[0]
    I = w_up[0].shape[1] // 2
    counts, offsets, row_of_slot, slot_of_row = route(topk_ids, E)
    x_rows = dispatch(_as64(x), slot_of_row, K)
    dy_rows = dispatch(_as64(dy), slot_of_row, K)
    w_rows = _as64(topk_weights).reshape(-1)[slot_of_row]
    dx_rows = torch.zeros(T * K, H, dtype=F64)
    d_topk_rows = torch.zeros(T * K, dtype=F64)
    dW_up = torch.zeros(E, H, 2 * I, dtype=F64)
    dW_down = torch.zeros(E, I, H, dtype=F64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        g = expert_backward(x_rows[r0:r1], dy_rows[r0:r1], w_rows[r0:r1], w_up[e], w_down[e])
        dx_rows[r0:r1] = g["dx_rows"]
        d_topk_rows[r0:r1] = g["d_topk"]
        dW_up[e] = g["dW_up"]
        dW_down[e] = g["dW_down"]
    dx = combine(dx_rows, row_of_slot, None, T, K)
    d_topk = d_topk_rows[row_of_slot].reshape(T, K)
    out = dict(dx=dx, d_topk_weights=d_topk, dW_up=dW_up, dW_down=dW_down)
    if shared is not None:
        g = expert_backward(_as64(x), _as64(dy), torch.ones(T, dtype=F64), *shared)
        out["dx"] = dx + g["dx_rows"]
        out.update(dS_up=g["dW_up"], dS_down=g["dW_down"])
    return out


# ------------------------------------------------------------------ sampled evaluation

def token_outputs(tokens, x_tok, topk_ids_tok, topk_weights_tok, w_up, w_down, dy_tok=None):
    """y, and with dy also dx and d_topk_weights, for a subset of tokens only.

    x_tok/dy_tok [n,H], topk_ids_tok/topk_weights_tok [n,K] are those tokens'
    rows. Each slot goes through its own expert; the result equals the same
    rows of forward()/backward() (a token's outputs depend only on its own
    slots). Returns dict of float64 tensors."""
    n, H = x_tok.shape
    K = topk_ids_tok.shape[1]
    X = _as64(x_tok)
    y = torch.zeros(n, H, dtype=F64)
    dx = torch.zeros(n, H, dtype=F64)
    d_w = torch.zeros(n, K, dtype=F64)
    ids = topk_ids_tok.to(torch.int64)
    W = _as64(topk_weights_tok)
    for e in torch.unique(ids).tolist():
        ti, ki = (ids == e).nonzero(as_tuple=True)
        if dy_tok is None:
            _, _, _, o = expert_forward(X[ti], w_up[e], w_down[e])
        else:
            g = expert_backward(X[ti], _as64(dy_tok)[ti], W[ti, ki], w_up[e], w_down[e])
            o = g["o"]
            dx.index_add_(0, ti, g["dx_rows"])
            d_w[ti, ki] = g["d_topk"]
        y.index_add_(0, ti, W[ti, ki][:, None] * o)
    out = dict(y=y)
    if dy_tok is not None:
        out.update(dx=dx, d_topk_weights=d_w)
    return out


def expert_weight_grads(e, x, dy, topk_ids, topk_weights, w_up, w_down):
    """dW_up[e], dW_down[e] for one expert (all of its slots)."""
    K = topk_ids.shape[1]
    flat = topk_ids.reshape(-1).to(torch.int64)
    slots = (flat == e).nonzero().squeeze(1)
    H = x.shape[1]
    I = w_up[e].shape[1] // 2
    if slots.numel() == 0:
        return torch.zeros(H, 2 * I, dtype=F64), torch.zeros(I, H, dtype=F64)
    tok = slots // K
    g = expert_backward(_as64(x[tok]), _as64(dy[tok]),
                        _as64(topk_weights).reshape(-1)[slots], w_up[e], w_down[e])
    return g["dW_up"], g["dW_down"]
