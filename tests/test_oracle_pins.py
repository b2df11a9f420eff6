"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked fixtures, brute force, closed forms, a dense special case checked
against torch's own SwiGLU, algebraic invariants and float64 finite differences."""
import math
import os

import pytest
import torch
import torch.nn.functional as Fnn

import oracle
from workloads import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out[key] = rest
    return out


def _vals(text, L=None):
    env = {"L": L, "__builtins__": {}}
    rows = [r.split() for r in text.split(";")]
    return [[float(eval(tok, env)) for tok in r] for r in rows]


def _rand_case(T=6, H=8, I=4, E=5, K=3, seed=0, distinct=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g, dtype=F64)
    if distinct:
        ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)])
    else:
        ids = torch.randint(0, E, (T, K), generator=g)
    w = torch.softmax(torch.randn(T, K, generator=g, dtype=F64), 1)
    wu = torch.randn(E, H, 2 * I, generator=g, dtype=F64) / math.sqrt(H)
    wd = torch.randn(E, I, H, generator=g, dtype=F64) / math.sqrt(I)
    dy = torch.randn(T, H, generator=g, dtype=F64)
    return x, ids.to(torch.int32), w, wu, wd, dy


# ------------------------------------------------------------------ routing

def test_routing_golden_fixture():
    fx = _read_fixture("routing_t4_k2_e4.txt")
    T, K, E = int(fx["T"]), int(fx["K"]), int(fx["E"])
    ids = torch.tensor([int(v) for v in fx["ids"].split()], dtype=torch.int32).view(T, K)
    counts, offsets, row_of_slot, slot_of_row = oracle.route(ids, E)
    assert counts.tolist() == [int(v) for v in fx["counts"].split()]
    assert offsets.tolist() == [int(v) for v in fx["offsets"].split()]
    assert slot_of_row.tolist() == [int(v) for v in fx["slot_of_row"].split()]
    assert row_of_slot.tolist() == [int(v) for v in fx["row_of_slot"].split()]


@pytest.mark.parametrize("seed,T,K,E,distinct", [(0, 7, 3, 5, True), (1, 13, 2, 9, False),
                                                  (2, 1, 1, 1, True), (3, 9, 4, 4, True)])
def test_routing_brute_force(seed, T, K, E, distinct):
    _, ids, *_ = _rand_case(T=T, K=K, E=E, seed=seed, distinct=distinct)
    counts, offsets, row_of_slot, slot_of_row = oracle.route(ids, E)
    flat = ids.reshape(-1).tolist()
    S = T * K
    # brute force: walk experts in order, then slots in order, assigning rows
    bf_row = [None] * S
    r = 0
    bf_counts = []
    for e in range(E):
        c = 0
        for s in range(S):
            if flat[s] == e:
                bf_row[s] = r
                r += 1
                c += 1
        bf_counts.append(c)
    assert counts.tolist() == bf_counts
    assert int(counts.sum()) == S and int(offsets[-1]) == S and int(offsets[0]) == 0
    assert row_of_slot.tolist() == bf_row
    assert slot_of_row[row_of_slot].tolist() == list(range(S))


def test_routing_rejects_bad_ids():
    ids = torch.tensor([[0, 5]], dtype=torch.int32)
    with pytest.raises(ValueError):
        oracle.route(ids, 5)


# ------------------------------------------------------------------ hand-worked closed form

def test_scalar_two_expert_closed_form():
    L = math.log(3.0)
    fx = _read_fixture("scalar_two_experts.txt")
    x = torch.tensor([[float(fx["x"])]], dtype=F64)
    ids = torch.tensor([[int(v) for v in fx["topk_ids"].split()]], dtype=torch.int32)
    w = torch.tensor([_vals(fx["topk_weights"])[0]], dtype=F64)
    wu = torch.tensor(_vals(fx["w_up"], L), dtype=F64).view(2, 1, 2)
    wd = torch.tensor(_vals(fx["w_down"], L), dtype=F64).view(2, 1, 1)
    dy = torch.tensor([[float(fx["dy"])]], dtype=F64)
    y = oracle.forward(x, ids, w, wu, wd)
    assert y.item() == pytest.approx(_vals(fx["y"], L)[0][0], rel=1e-14)
    g = oracle.backward(x, ids, w, wu, wd, dy)
    assert g["d_topk_weights"].reshape(-1).tolist() == pytest.approx(
        [v[0] for v in _vals(fx["d_topk_weights"], L)], rel=1e-14, abs=1e-15)
    exp_up = torch.tensor(_vals(fx["dW_up"], L), dtype=F64).view(2, 1, 2)
    exp_down = torch.tensor(_vals(fx["dW_down"], L), dtype=F64).view(2, 1, 1)
    # fixture lists expert 0 first
    assert torch.allclose(g["dW_up"], exp_up, rtol=1e-14, atol=1e-15)
    assert torch.allclose(g["dW_down"], exp_down, rtol=1e-14, atol=1e-15)
    assert g["dx"].item() == pytest.approx(_vals(fx["dx"], L)[0][0], rel=1e-14)


# ------------------------------------------------------------------ dense special cases

def _dense_swiglu_ffn(x, wg, wu, wd):
    return (Fnn.silu(x @ wg) * (x @ wu)) @ wd


def test_single_expert_k1_is_dense_swiglu():
    g = torch.Generator().manual_seed(5)
    T, H, I = 9, 12, 6
    x = torch.randn(T, H, generator=g, dtype=F64)
    wg = torch.randn(H, I, generator=g, dtype=F64)
    wu = torch.randn(H, I, generator=g, dtype=F64)
    wd = torch.randn(I, H, generator=g, dtype=F64)
    ids = torch.zeros(T, 1, dtype=torch.int32)
    w = torch.ones(T, 1, dtype=F64)
    y = oracle.forward(x, ids, w, torch.cat([wg, wu], 1)[None], wd[None])
    assert torch.allclose(y, _dense_swiglu_ffn(x, wg, wu, wd), rtol=1e-12, atol=1e-12)


def test_identical_experts_reduce_to_dense():
    x, ids, w, wu, wd, _ = _rand_case(T=10, H=8, I=4, E=6, K=3, seed=3)
    wu = wu[:1].expand(6, -1, -1).contiguous()
    wd = wd[:1].expand(6, -1, -1).contiguous()
    y = oracle.forward(x, ids, w, wu, wd)   # softmax weights sum to 1 per token
    I = wu.shape[2] // 2
    assert torch.allclose(y, _dense_swiglu_ffn(x, wu[0][:, :I], wu[0][:, I:], wd[0]),
                          rtol=1e-12, atol=1e-12)


def test_dense_case_gradients_match_torch_autograd_of_dense_ffn():
    """E=1, K=1, w=1: the layer is a dense SwiGLU FFN; autograd of torch's own
    F.silu formulation gives dx, dWg|dWu, dWd."""
    g = torch.Generator().manual_seed(11)
    T, H, I = 7, 10, 4
    x = torch.randn(T, H, generator=g, dtype=F64, requires_grad=True)
    wg = torch.randn(H, I, generator=g, dtype=F64, requires_grad=True)
    wu = torch.randn(H, I, generator=g, dtype=F64, requires_grad=True)
    wd = torch.randn(I, H, generator=g, dtype=F64, requires_grad=True)
    dy = torch.randn(T, H, generator=g, dtype=F64)
    y = _dense_swiglu_ffn(x, wg, wu, wd)
    y.backward(dy)
    ids = torch.zeros(T, 1, dtype=torch.int32)
    w = torch.ones(T, 1, dtype=F64)
    got = oracle.backward(x.detach(), ids, w, torch.cat([wg, wu], 1).detach()[None],
                          wd.detach()[None], dy)
    assert torch.allclose(got["dx"], x.grad, rtol=1e-12, atol=1e-12)
    assert torch.allclose(got["dW_up"][0], torch.cat([wg.grad, wu.grad], 1), rtol=1e-12, atol=1e-12)
    assert torch.allclose(got["dW_down"][0], wd.grad, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ invariants

def test_permute_unpermute_round_trip():
    """dispatch then unweighted... weighted combine with weights summing to 1 and
    identity experts returns x exactly (one-hot weights) or to rounding (softmax)."""
    x, ids, w, *_ = _rand_case(T=11, H=5, E=7, K=3, seed=9)
    counts, offsets, row_of_slot, slot_of_row = oracle.route(ids, 7)
    rows = oracle.dispatch(x, slot_of_row, 3)
    assert torch.allclose(oracle.combine(rows, row_of_slot, w, 11, 3), x, rtol=1e-13, atol=1e-13)
    onehot = torch.zeros(11, 3, dtype=F64)
    onehot[:, 1] = 1
    assert torch.equal(oracle.combine(rows, row_of_slot, onehot, 11, 3), x)
    # each dispatched row is the token of its slot
    for r in range(33):
        assert torch.equal(rows[r], x[int(slot_of_row[r]) // 3])


def test_linearity_in_topk_weights():
    x, ids, w, wu, wd, _ = _rand_case(seed=4)
    y1 = oracle.forward(x, ids, w, wu, wd)
    y2 = oracle.forward(x, ids, 2.5 * w, wu, wd)
    assert torch.allclose(y2, 2.5 * y1, rtol=1e-13, atol=1e-13)


def test_token_permutation_equivariance():
    x, ids, w, wu, wd, dy = _rand_case(T=9, seed=6)
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(1))
    y = oracle.forward(x, ids, w, wu, wd)
    yp = oracle.forward(x[perm], ids[perm], w[perm], wu, wd)
    assert torch.allclose(yp, y[perm], rtol=1e-13, atol=1e-13)
    g = oracle.backward(x, ids, w, wu, wd, dy)
    gp = oracle.backward(x[perm], ids[perm], w[perm], wu, wd, dy[perm])
    assert torch.allclose(gp["dx"], g["dx"][perm], rtol=1e-12, atol=1e-12)
    assert torch.allclose(gp["dW_up"], g["dW_up"], rtol=1e-12, atol=1e-12)


def test_empty_expert_has_exactly_zero_weight_grads():
    x, ids, w, wu, wd, dy = _rand_case(T=8, E=5, K=2, seed=2)
    ids = torch.where(ids == 4, torch.full_like(ids, 0), ids)
    ids[:, 1] = torch.where(ids[:, 0] == ids[:, 1], (ids[:, 0] + 1) % 4, ids[:, 1])
    assert not (ids == 4).any()
    g = oracle.backward(x, ids, w, wu, wd, dy)
    assert torch.count_nonzero(g["dW_up"][4]) == 0
    assert torch.count_nonzero(g["dW_down"][4]) == 0


def test_duplicate_expert_in_one_token():
    """Two slots of one token on the same expert: both contribute."""
    x, ids, w, wu, wd, dy = _rand_case(T=3, E=4, K=2, seed=8)
    ids = torch.tensor([[1, 1], [0, 2], [3, 3]], dtype=torch.int32)
    y = oracle.forward(x, ids, w, wu, wd)
    ids1 = torch.tensor([[1], [0], [3]], dtype=torch.int32)
    wsum = torch.stack([w[0].sum(), w[1, 0], w[2].sum()])[:, None]
    y1 = oracle.forward(x, ids1, wsum, wu, wd)
    # token 1 loses its second slot in the single-slot version: add it separately
    y1[1] += oracle.forward(x[1:2], torch.tensor([[2]], dtype=torch.int32), w[1:2, 1:2], wu, wd)[0]
    assert torch.allclose(y, y1, rtol=1e-13, atol=1e-13)


def test_d_topk_equals_hidden_side_dot():
    """<dy[t], o[s]> = <dy[t] W_down^T, h[s]> (the identity the GPU uses)."""
    x, ids, w, wu, wd, dy = _rand_case(seed=12)
    g = oracle.backward(x, ids, w, wu, wd, dy)
    I = wu.shape[2] // 2
    for t in range(x.shape[0]):
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            h = oracle.swiglu(x[t] @ wu[e][:, :I], x[t] @ wu[e][:, I:])
            alt = (dy[t] @ wd[e].T) @ h
            assert abs(alt - g["d_topk_weights"][t, k]) <= 1e-10 * max(1.0, abs(alt))


# ------------------------------------------------------------------ finite differences

def _loss(x, ids, w, wu, wd, dy):
    return float((oracle.forward(x, ids, w, wu, wd) * dy).sum())


def _fd_failures():
    """Central float64 finite differences of sum(y * dy) against the oracle's backward on a tiny
    case; returns {gradient name: first mismatch} (empty when every sampled element agrees)."""
    T, H, I, E, K = 8, 16, 8, 4, 2
    x, ids, w, wu, wd, dy = _rand_case(T=T, H=H, I=I, E=E, K=K, seed=21)
    g = oracle.backward(x, ids, w, wu, wd, dy)
    eps = 1e-6
    gen = torch.Generator().manual_seed(0)
    bad = {}

    def check(name, tensor, grad, n=25):
        flat = tensor.view(-1)
        idx = torch.randperm(flat.numel(), generator=gen)[:n]
        for i in idx.tolist():
            old = flat[i].item()
            flat[i] = old + eps
            lp = _loss(x, ids, w, wu, wd, dy)
            flat[i] = old - eps
            lm = _loss(x, ids, w, wu, wd, dy)
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = grad.reshape(-1)[i].item()
            if abs(fd - an) > 1e-6 * max(1.0, abs(an)):
                bad[name] = (i, fd, an)
                return

    check("x", x, g["dx"])
    check("w", w, g["d_topk_weights"], n=T * K)
    check("w_up", wu, g["dW_up"], n=60)
    check("w_down", wd, g["dW_down"], n=40)
    return bad


def test_finite_difference_gradients():
    assert _fd_failures() == {}


# ------------------------------------------------------------------ sampled evaluation

def test_token_and_expert_subsets_match_full():
    x, ids, w, wu, wd, dy = _rand_case(T=12, H=8, I=4, E=5, K=3, seed=31)
    y = oracle.forward(x, ids, w, wu, wd)
    g = oracle.backward(x, ids, w, wu, wd, dy)
    toks = torch.tensor([0, 5, 11])
    sub = oracle.token_outputs(toks, x[toks], ids[toks], w[toks], wu, wd, dy[toks])
    assert torch.allclose(sub["y"], y[toks], rtol=1e-13, atol=1e-13)
    assert torch.allclose(sub["dx"], g["dx"][toks], rtol=1e-12, atol=1e-12)
    assert torch.allclose(sub["d_topk_weights"], g["d_topk_weights"][toks], rtol=1e-12, atol=1e-12)
    for e in range(5):
        du, dd = oracle.expert_weight_grads(e, x, dy, ids, w, wu, wd)
        assert torch.allclose(du, g["dW_up"][e], rtol=1e-12, atol=1e-12)
        assert torch.allclose(dd, g["dW_down"][e], rtol=1e-12, atol=1e-12)


def test_lazy_expert_weights_match_full_tensor():
    wl = synth.small("t", 4, 16, 8, 3, 2)
    full_up, full_down = synth.w_up(wl), synth.w_down(wl)
    lu, ld = synth.LazyExperts(wl, "up"), synth.LazyExperts(wl, "down")
    for e in range(3):
        assert torch.equal(lu[e], full_up[e]) and torch.equal(ld[e], full_down[e])


# ------------------------------------------------------------------ a planted mistake is caught

def test_planted_gate_up_swap_is_caught(monkeypatch):
    """Swapping gate and up inside the oracle must break the dense pin."""
    g = torch.Generator().manual_seed(5)
    T, H, I = 5, 6, 3
    x = torch.randn(T, H, generator=g, dtype=F64)
    wg = torch.randn(H, I, generator=g, dtype=F64)
    wu = torch.randn(H, I, generator=g, dtype=F64)
    wd = torch.randn(I, H, generator=g, dtype=F64)
    ref = _dense_swiglu_ffn(x, wg, wu, wd)
    from oracle import moe_ffn
    monkeypatch.setattr(moe_ffn, "swiglu", lambda a, b: moe_ffn.silu(b) * a)
    y = oracle.forward(x, torch.zeros(T, 1, dtype=torch.int32), torch.ones(T, 1, dtype=F64),
                       torch.cat([wg, wu], 1)[None], wd[None])
    assert not torch.allclose(y, ref, rtol=1e-6, atol=1e-6)


def _plant_silu_slope(moe_ffn):
    # d_gate without the (1 + gate (1 - sigmoid)) factor of silu's derivative
    def wrong(d_h, gate, up):
        sg = torch.sigmoid(gate)
        return d_h * up * sg, d_h * gate * sg
    return "swiglu_grad", wrong


def _plant_d_up_factor(moe_ffn):
    # d_up = d_h * sigmoid(gate) instead of d_h * silu(gate)
    def wrong(d_h, gate, up):
        sg = torch.sigmoid(gate)
        return d_h * up * sg * (1.0 + gate * (1.0 - sg)), d_h * sg
    return "swiglu_grad", wrong


def _plant_unweighted_w2grad(moe_ffn):
    # W2Grad from the unweighted dY rows (the routing weight dropped)
    orig = moe_ffn.expert_backward

    def wrong(X, dY, w, w_up_e, w_down_e):
        g = orig(X, dY, w, w_up_e, w_down_e)
        h = moe_ffn.expert_forward(X, w_up_e, w_down_e)[2]
        g["dW_down"] = h.T @ dY
        return g
    return "expert_backward", wrong


def _plant_weighted_d_topk(moe_ffn):
    # d_topk_weights scaled by the routing weight, as if dO were used instead of dY
    orig = moe_ffn.expert_backward

    def wrong(X, dY, w, w_up_e, w_down_e):
        g = orig(X, dY, w, w_up_e, w_down_e)
        g["d_topk"] = g["d_topk"] * w
        return g
    return "expert_backward", wrong


@pytest.mark.parametrize("plant,caught_by", [(_plant_silu_slope, {"x", "w_up"}),
                                             (_plant_d_up_factor, {"x", "w_up"}),
                                             (_plant_unweighted_w2grad, {"w_down"}),
                                             (_plant_weighted_d_topk, {"w"})])
def test_planted_backward_mistakes_are_caught(monkeypatch, plant, caught_by):
    """Each plausible slip in the backward's arithmetic, planted in the oracle, must fail the
    finite-difference pin on the gradients it touches."""
    from oracle import moe_ffn
    name, wrong = plant(moe_ffn)
    monkeypatch.setattr(moe_ffn, name, wrong)
    bad = _fd_failures()
    assert caught_by <= set(bad), (plant.__name__, sorted(bad))


# ------------------------------------------------------------------ shared expert (RFC §6.1)

def _shared_case(seed, T=9, H=8, I=4, E=5, K=2, Is=6):
    x, ids, w, wu, wd, dy = _rand_case(T=T, H=H, I=I, E=E, K=K, seed=seed)
    g = torch.Generator().manual_seed(seed + 100)
    su = torch.randn(H, 2 * Is, generator=g, dtype=F64) / math.sqrt(H)
    sd = torch.randn(Is, H, generator=g, dtype=F64) / math.sqrt(Is)
    return x, ids, w, wu, wd, dy, (su, sd)


def test_shared_expert_alone_is_the_dense_swiglu_ffn():
    """Routed experts with zero down-projections: y is torch's own SwiGLU FFN of the shared
    expert, and its weight gradients are torch autograd's."""
    x, ids, w, wu, wd, dy, (su, sd) = _shared_case(1)
    Is = sd.shape[0]
    y = oracle.forward(x, ids, w, wu, torch.zeros_like(wd), shared=(su, sd))
    assert torch.allclose(y, _dense_swiglu_ffn(x, su[:, :Is], su[:, Is:], sd), rtol=1e-12, atol=1e-12)
    su_t, sd_t = su.clone().requires_grad_(True), sd.clone().requires_grad_(True)
    (_dense_swiglu_ffn(x, su_t[:, :Is], su_t[:, Is:], sd_t) * dy).sum().backward()
    g = oracle.backward(x, ids, w, wu, torch.zeros_like(wd), dy, shared=(su, sd))
    assert torch.allclose(g["dS_up"], su_t.grad, rtol=1e-12, atol=1e-12)
    assert torch.allclose(g["dS_down"], sd_t.grad, rtol=1e-12, atol=1e-12)


def test_shared_expert_equals_an_extra_always_on_slot():
    """A shared expert with I_s = I is the same as an extra expert routed from every token with
    weight 1 (one more slot per token)."""
    x, ids, w, wu, wd, dy, (su, sd) = _shared_case(2, Is=4)
    T, K = ids.shape
    E = wu.shape[0]
    ids1 = torch.cat([ids, torch.full((T, 1), E, dtype=torch.int32)], 1)
    w1 = torch.cat([w, torch.ones(T, 1, dtype=F64)], 1)
    wu1, wd1 = torch.cat([wu, su[None]]), torch.cat([wd, sd[None]])
    assert torch.allclose(oracle.forward(x, ids, w, wu, wd, shared=(su, sd)),
                          oracle.forward(x, ids1, w1, wu1, wd1), rtol=1e-12, atol=1e-12)
    g = oracle.backward(x, ids, w, wu, wd, dy, shared=(su, sd))
    g1 = oracle.backward(x, ids1, w1, wu1, wd1, dy)
    assert torch.allclose(g["dx"], g1["dx"], rtol=1e-12, atol=1e-12)
    assert torch.allclose(g["dS_up"], g1["dW_up"][E], rtol=1e-12, atol=1e-12)
    assert torch.allclose(g["dS_down"], g1["dW_down"][E], rtol=1e-12, atol=1e-12)
    assert torch.allclose(g["d_topk_weights"], g1["d_topk_weights"][:, :K], rtol=1e-12, atol=1e-12)


def test_shared_expert_finite_differences():
    x, ids, w, wu, wd, dy, (su, sd) = _shared_case(3, Is=6)
    g = oracle.backward(x, ids, w, wu, wd, dy, shared=(su, sd))
    eps = 1e-6

    def loss():
        return float((oracle.forward(x, ids, w, wu, wd, shared=(su, sd)) * dy).sum())

    gen = torch.Generator().manual_seed(4)
    for name, t, grad in (("x", x, g["dx"]), ("su", su, g["dS_up"]), ("sd", sd, g["dS_down"])):
        flat = t.view(-1)
        for i in torch.randperm(flat.numel(), generator=gen)[:20].tolist():
            old = flat[i].item()
            flat[i] = old + eps
            lp = loss()
            flat[i] = old - eps
            lm = loss()
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = grad.reshape(-1)[i].item()
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, i, fd, an)
