"""Parity of the CUDA path (through the C ABI) with the float64 CPU oracle.

Routing is compared bit for bit; y, dx and the weight gradients within
|gpu - oracle| <= 1e-2 + 1e-2 |oracle|; d_topk_weights within 2e-2 * max(|oracle|, rms).
The tiny, skew, tail and qwen workloads are compared in full, every token and every expert,
qwen (the benchmark's workload, in its launch configuration) also with the counter-fused forward
forms; large_hidden on all of its hot experts, eight seeded cold experts and 256 seeded tokens,
which the oracle computes one by one."""
import functools

import pytest
import torch

import oracle
from layer_harness import (assert_close, assert_dtopk, export_routing, make_inputs,
                           run_layer)
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu


def _host(inp):
    return {k: v.cpu() for k, v in inp.items()}


def _check_routing(out, ids, E):
    counts, offsets, row_of_slot, _ = oracle.route(ids.cpu(), E)
    g_counts, g_offsets, g_rows = export_routing(out, E, ids.numel())
    assert torch.equal(g_counts.long(), counts)
    assert torch.equal(g_offsets.long(), offsets)
    assert torch.equal(g_rows.long(), row_of_slot)


def _oracle_full(inp):
    h = _host(inp)
    y = oracle.forward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"])
    g = oracle.backward(h["x"], h["topk_ids"], h["topk_weights"], h["w_up"], h["w_down"], h["dy"])
    return y, g


def _compare_full(out, y, g, tag=""):
    """Every element; the weight gradients one expert at a time (bounded host memory)."""
    assert_close("y" + tag, out["y"], y)
    assert_close("dx" + tag, out["dx"], g["dx"])
    assert_dtopk(out["d_topk_weights"], g["d_topk_weights"])
    for e in range(g["dW_up"].shape[0]):
        assert_close(f"dW_down[{e}]" + tag, out["dW_down"][e], g["dW_down"][e])
        assert_close(f"dW_up[{e}]" + tag, out["dW_up"][e], g["dW_up"][e])


def _check_full(inp, out):
    y, g = _oracle_full(inp)
    _compare_full(out, y, g)


def _check_sampled(inp, out, n_tokens, experts, seed=0):
    T = inp["x"].shape[0]
    gen = torch.Generator().manual_seed(seed)
    toks = torch.randperm(T, generator=gen)[:n_tokens].sort().values
    toks = torch.cat([toks, torch.tensor([0, T - 1])]).unique()
    ids = inp["topk_ids"].cpu()
    needed = sorted(set(ids[toks].reshape(-1).tolist()) | set(experts))
    wu = {e: inp["w_up"][e].cpu() for e in needed}
    wd = {e: inp["w_down"][e].cpu() for e in needed}

    class _Sel:
        shape = (inp["w_up"].shape[0],)

        def __init__(self, d):
            self.d = d

        def __getitem__(self, e):
            return self.d[int(e)]

    x_t = inp["x"][toks.to(inp["x"].device)].cpu()
    dy_t = inp["dy"][toks.to(inp["x"].device)].cpu()
    ref = oracle.token_outputs(toks, x_t, ids[toks], inp["topk_weights"].cpu()[toks], _Sel(wu), _Sel(wd), dy_t)
    dev_t = toks.to(inp["x"].device)
    assert_close("y[sample]", out["y"][dev_t], ref["y"])
    assert_close("dx[sample]", out["dx"][dev_t], ref["dx"])
    assert_dtopk(out["d_topk_weights"][dev_t], ref["d_topk_weights"])
    x_all, dy_all = inp["x"].cpu(), inp["dy"].cpu()
    for e in experts:
        du, dd = oracle.expert_weight_grads(e, x_all, dy_all, ids, inp["topk_weights"].cpu(),
                                            _Sel(wu), _Sel(wd))
        assert_close(f"dW_up[{e}]", out["dW_up"][e], du)
        assert_close(f"dW_down[{e}]", out["dW_down"][e], dd)


@pytest.mark.parametrize("name", ["tiny", "skew", "tail"])
def test_workload_full_parity(name):
    w = synth.BY_NAME[name]
    inp = make_inputs(w)
    out = run_layer(inp)
    assert out["status"] == _abi.MM_OK
    _check_routing(out, inp["topk_ids"], w.E)
    _check_full(inp, out)
    if name == "skew":  # experts 14 and 15 receive nothing: exactly zero gradients
        assert torch.count_nonzero(out["dW_up"][14:]) == 0
        assert torch.count_nonzero(out["dW_down"][14:]) == 0


@functools.lru_cache(maxsize=1)
def _qwen_reference():
    """The oracle's outputs over the whole qwen workload (its inputs drawn on the device, which
    gives the host generator's values bit for bit, and copied to the host)."""
    w = synth.BY_NAME["qwen"]
    y, g = _oracle_full(make_inputs(w))
    torch.cuda.empty_cache()
    return w, y, g


@pytest.mark.parametrize("fwd_flags", [0, _abi.MM_FLAG_FUSED_FORWARD_GEMMS | _abi.MM_FLAG_FUSED_COMBINE],
                         ids=["default", "counter_fused_forward"])
def test_qwen_full_parity(fwd_flags):
    """The benchmark's workload (T=16384, H=2048, I=768, E=128, K=8) in the benchmark's launch
    configuration, and with GEMM2 released by the ready counters and the combine fused into its
    epilogue: routing bit for bit, and y, dx, d_topk_weights and both weight gradients of all
    128 experts against the float64 oracle, element by element."""
    w, y, g = _qwen_reference()
    inp = make_inputs(w)
    out = run_layer(inp, flags=fwd_flags)
    assert out["status"] == _abi.MM_OK
    _check_routing(out, inp["topk_ids"], w.E)
    _compare_full(out, y, g, tag=f" (forward flags 0x{fwd_flags:x})")
    del out, inp
    torch.cuda.empty_cache()


def test_large_hidden_sampled_parity():
    """T=8192, H=7168, I=2048, E=256, K=8 (22.5 GB of expert weights), 25 % of the slots on the
    hot experts 0..7: routing bit for bit; the weight gradients of all eight hot experts and of
    eight seeded cold ones, and y, dx, d_topk_weights of 256 seeded tokens (plus the first and
    the last), against the oracle."""
    w = synth.BY_NAME["large_hidden"]
    inp = make_inputs(w)
    out = run_layer(inp)
    assert out["status"] == _abi.MM_OK
    _check_routing(out, inp["topk_ids"], w.E)
    gen = torch.Generator().manual_seed(4)
    cold = (8 + torch.randperm(w.E - 8, generator=gen)[:8]).sort().values.tolist()
    _check_sampled(inp, out, 256, list(range(8)) + cold, seed=4)
    del out, inp
    torch.cuda.empty_cache()


def test_two_million_slots_sampled_parity():
    """The largest layer in the tests: 2^21 slots (T=262144, K=8), a 13 GB workspace, row and
    element offsets far past 2^31 bytes. Routing is checked bit for bit, y/dx/d_topk on sampled
    tokens and the weight gradients of two experts (32k rows each) against the oracle."""
    w = synth.small("huge", 262144, 512, 128, 64, 8, seed=11)
    inp = make_inputs(w)
    out = run_layer(inp)
    assert out["status"] == _abi.MM_OK
    _check_routing(out, inp["topk_ids"], w.E)
    _check_sampled(inp, out, 24, [0, 63])
    del out, inp
    torch.cuda.empty_cache()


def test_device_generator_matches_host():
    w = synth.small("g", 3, 64, 16, 5, 2)
    assert torch.equal(synth.w_up(w, device="cuda").cpu(), synth.w_up(w))
    assert torch.equal(synth.x(w, device="cuda").cpu(), synth.x(w))
    key = synth.stream_key(9, 3)
    big = synth.normal_bf16(key, (1 << 20,), 0.5, device="cuda", start=(1 << 32) - 7)
    assert torch.equal(big.cpu(), synth.normal_bf16(key, (1 << 20,), 0.5, start=(1 << 32) - 7))


# ------------------------------------------------------------------ edge cases

def _custom(T, H, I, E, K, ids=None, seed=3):
    w = synth.small("edge", T, H, I, E, K, seed=seed)
    return w, make_inputs(w, ids=ids)


@pytest.mark.parametrize("T,H,I,E,K", [
    (1, 64, 64, 1, 1),        # one token, one expert (dense SwiGLU FFN)
    (3, 128, 64, 7, 2),       # fewer slots than experts: most experts empty
    (200, 136, 72, 5, 3),     # H, I not multiples of 64: masked columns and zero-filled K tails
    (130, 256, 128, 2, 1),    # one expert gets 129+ rows: tail tile
    (64, 512, 256, 64, 16),   # K = 16
    (40, 64, 32, 1024, 4),    # E = 1024
    (1, 8, 8, 16, 16),        # the smallest H and I (one 16-byte row), one token in 16 experts
    (5, 24, 16, 3, 3),        # H and I below one 64-wide block: every tile is mostly padding
])
def test_edge_shapes(T, H, I, E, K):
    w, inp = _custom(T, H, I, E, K)
    out = run_layer(inp)
    assert out["status"] == _abi.MM_OK
    _check_routing(out, inp["topk_ids"], E)
    _check_full(inp, out)


def test_duplicate_experts_in_a_token():
    ids = torch.tensor([[1, 1], [0, 2], [3, 3], [2, 0]] * 8, dtype=torch.int32)
    w, inp = _custom(32, 128, 64, 4, 2, ids=ids)
    out = run_layer(inp)
    _check_routing(out, inp["topk_ids"], 4)
    _check_full(inp, out)


def test_all_slots_on_one_expert_and_hot_tail():
    T, E, K = 300, 8, 2
    ids = torch.stack([torch.zeros(T, dtype=torch.int32), 1 + (torch.arange(T) % 7).int()], 1)
    w, inp = _custom(T, 128, 128, E, K, ids=ids)
    out = run_layer(inp)
    _check_routing(out, inp["topk_ids"], E)
    _check_full(inp, out)


# ------------------------------------------------------------------ stability

def test_deterministic_and_poisoned_workspace():
    """Three calls on one workspace, poisoned with NaN bytes in between, give bitwise
    identical results (no stale counters or tables from an earlier call)."""
    w = synth.BY_NAME["tail"]
    inp = make_inputs(w)
    first = run_layer(inp)
    keys = ["y", "dx", "d_topk_weights", "dW_up", "dW_down"]
    ref = {k: first[k].clone() for k in keys}
    ws = first["ws"]
    for _ in range(2):
        ws.fill_(0xFF)
        again = run_layer(inp, ws=ws)
        assert again["status"] == _abi.MM_OK
        for k in keys:
            assert torch.equal(again[k], ref[k]), k


def test_two_forwards_then_two_backwards():
    wa = synth.small("a", 96, 256, 128, 6, 2, seed=11)
    wb = synth.small("b", 96, 256, 128, 6, 2, seed=12)
    ia, ib = make_inputs(wa), make_inputs(wb)
    ref_a, ref_b = run_layer(ia), run_layer(ib)
    fa = run_layer(ia, backward=False)
    fb = run_layer(ib, backward=False)
    # backward of a on its own workspace after b's forward
    for inp, f, ref in ((ia, fa, ref_a), (ib, fb, ref_b)):
        x, wu, wd = inp["x"], inp["w_up"], inp["w_down"]
        dx = torch.empty_like(x)
        dt = torch.empty(inp["topk_ids"].shape, dtype=torch.float32, device="cuda")
        du, dd = torch.empty_like(wu), torch.empty_like(wd)
        _abi.check(_abi.mm_backward(f["dims"], inp["dy"].data_ptr(), x.data_ptr(),
                                    inp["topk_ids"].data_ptr(), inp["topk_weights"].data_ptr(),
                                    wu.data_ptr(), wd.data_ptr(), f["ws"].data_ptr(),
                                    f["ws"].numel(), dx.data_ptr(), dt.data_ptr(), du.data_ptr(),
                                    dd.data_ptr(), torch.cuda.current_stream().cuda_stream, 0),
                   "mm_backward")
        assert torch.equal(dx, ref["dx"]) and torch.equal(du, ref["dW_up"])
        assert torch.equal(dd, ref["dW_down"]) and torch.equal(dt, ref["d_topk_weights"])


def test_bad_expert_id_is_reported_and_recovers():
    w = synth.small("bad", 64, 128, 64, 4, 2)
    inp = make_inputs(w)
    good = run_layer(inp)
    bad_ids = inp["topk_ids"].clone()
    bad_ids[5, 1] = 4          # == E: out of range
    bad = dict(inp, topk_ids=bad_ids)
    out = run_layer(bad)
    assert out["status"] == _abi.MM_ERR_BAD_EXPERT_ID
    # with the host-side pre-check, mm_forward itself refuses
    d = out["dims"]
    y = torch.empty_like(inp["x"])
    st = _abi.mm_forward(d, inp["x"].data_ptr(), bad_ids.data_ptr(), inp["topk_weights"].data_ptr(),
                         inp["w_up"].data_ptr(), inp["w_down"].data_ptr(), y.data_ptr(),
                         out["ws"].data_ptr(), out["ws"].numel(),
                         torch.cuda.current_stream().cuda_stream, _abi.MM_FLAG_VALIDATE_IDS)
    assert st == _abi.MM_ERR_BAD_EXPERT_ID
    neg = inp["topk_ids"].clone()
    neg[0, 0] = -1
    assert run_layer(dict(inp, topk_ids=neg))["status"] == _abi.MM_ERR_BAD_EXPERT_ID
    # the same workspace then serves a correct call
    again = run_layer(inp, ws=out["ws"])
    assert again["status"] == _abi.MM_OK
    assert torch.equal(again["y"], good["y"]) and torch.equal(again["dW_up"], good["dW_up"])


def test_host_side_argument_errors():
    w = synth.small("args", 16, 64, 32, 4, 2)
    inp = make_inputs(w)
    d = _abi.dims(16, 64, 32, 4, 2)
    n = _abi.mm_workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(inp["x"])
    st = torch.cuda.current_stream().cuda_stream
    args = [inp["x"].data_ptr(), inp["topk_ids"].data_ptr(), inp["topk_weights"].data_ptr(),
            inp["w_up"].data_ptr(), inp["w_down"].data_ptr(), y.data_ptr()]
    assert _abi.mm_forward(d, *args, ws.data_ptr(), n - 1, st, 0) == _abi.MM_ERR_WORKSPACE
    assert _abi.mm_forward(d, *args, ws.data_ptr() + 16, n, st, 0) == _abi.MM_ERR_WORKSPACE
    bad = list(args)
    bad[0] += 2
    assert _abi.mm_forward(d, *bad, ws.data_ptr(), n, st, 0) == _abi.MM_ERR_INVALID_ARG
    bad = list(args)
    bad[3] = 0
    assert _abi.mm_forward(d, *bad, ws.data_ptr(), n, st, 0) == _abi.MM_ERR_INVALID_ARG
    assert _abi.mm_forward(_abi.dims(16, 60, 32, 4, 2), *args, ws.data_ptr(), n, st, 0) == _abi.MM_ERR_UNSUPPORTED
    assert _abi.mm_forward(d, *args, ws.data_ptr(), n, st, 0) == _abi.MM_OK
    assert _abi.mm_get_status(ws.data_ptr(), st) == _abi.MM_OK


def test_torch_autograd_entry_point():
    from moe_ffn_expert_gb300.torch_api import hyper_mega_moe
    w = synth.small("ag", 48, 128, 64, 5, 2, seed=4)
    inp = make_inputs(w)
    ref = run_layer(inp)
    x = inp["x"].clone().requires_grad_(True)
    tw = inp["topk_weights"].clone().requires_grad_(True)
    wu = inp["w_up"].clone().requires_grad_(True)
    wd = inp["w_down"].clone().requires_grad_(True)
    y = hyper_mega_moe(x, inp["topk_ids"].long(), tw, wu, wd)
    y.backward(inp["dy"])
    assert torch.equal(y.detach(), ref["y"])
    assert torch.equal(x.grad, ref["dx"]) and torch.equal(tw.grad, ref["d_topk_weights"])
    assert torch.equal(wu.grad, ref["dW_up"]) and torch.equal(wd.grad, ref["dW_down"])


def test_bounded_wait_times_out_and_the_next_call_is_clean():
    """A withheld accumulator hand-off (test hook) must end in MM_ERR_TIMEOUT reported through
    the status word, not in a hang or a fault; the same workspace then gives correct results."""
    w = synth.small("stall", 700, 256, 128, 6, 2, seed=6)
    inp = make_inputs(w)
    ref = run_layer(inp)
    out = run_layer(inp, flags=_abi.MM_FLAG_TEST_STALL, ws=ref["ws"], backward=False)
    assert out["status"] == _abi.MM_ERR_TIMEOUT
    again = run_layer(inp, ws=ref["ws"])
    assert again["status"] == _abi.MM_OK
    for k in ("y", "dx", "d_topk_weights", "dW_up", "dW_down"):
        assert torch.equal(again[k], ref[k]), k


def test_accumulate_weight_grads_adds_into_the_outputs():
    """MM_FLAG_ACCUMULATE_WEIGHT_GRADS: dW += the step's gradient (bf16 adds), experts without
    slots keep their previous contents bit for bit; dx and d_topk are still overwritten."""
    T, E, K = 300, 8, 2
    ids = torch.stack([torch.arange(T) % 7, (torch.arange(T) + 3) % 7], 1).int()  # expert 7 empty
    w, inp = _custom(T, 256, 128, E, K, ids=ids, seed=13)
    ref = run_layer(inp)
    g = torch.Generator(device="cuda").manual_seed(5)
    base_up = torch.randn(inp["w_up"].shape, generator=g, device="cuda").to(torch.bfloat16)
    base_down = torch.randn(inp["w_down"].shape, generator=g, device="cuda").to(torch.bfloat16)
    out = run_layer(inp, bwd_flags=_abi.MM_FLAG_ACCUMULATE_WEIGHT_GRADS, d_up=base_up.clone(),
                    d_down=base_down.clone())
    assert out["status"] == _abi.MM_OK
    for name, base in (("dW_up", base_up), ("dW_down", base_down)):
        exp = base.double() + ref[name].double()
        got = out[name].double()
        assert ((got - exp).abs() <= 2.0 ** -8 * exp.abs() + 1e-6).all(), name
        assert torch.equal(out[name][7], base[7]), name  # the empty expert is untouched
    assert torch.equal(out["dx"], ref["dx"]) and torch.equal(out["d_topk_weights"], ref["d_topk_weights"])
