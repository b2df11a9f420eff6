"""mm_route_noalloc: routing tables for callers that cannot allocate device memory (for example
code running where a framework owns the device heap and forbids allocation mid-step). It keeps
its scratch in a static device array instead of a caller workspace. Checked here, through the
C ABI, against the workspace-based entry point (mm_forward + mm_routing_export): the tables are
integers, so they must match bit for bit, on consecutive calls that share the static scratch.

This file is collected last so that a failure here cannot hide the rest of the suite."""
import ctypes

import pytest
import torch

from moe_ffn_expert_gb300 import _abi
from moe_ffn_expert_gb300 import build as mm_build
from workloads import synth

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    mm_build.build()
    lib = ctypes.CDLL(_abi.LIB_PATH)
    fn = lib.mm_route_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_abi.mm_dims] + [ctypes.c_void_p] * 5
    return fn


def _reference(w, ids):
    """Routing tables from the workspace-based forward (small H and I keep it cheap)."""
    T, E, K = w.T, w.E, w.K
    H = I = 64
    d = _abi.dims(T, H, I, E, K)
    n = _abi.mm_workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    tw = torch.full((T, K), 1.0 / K, dtype=torch.float32, device="cuda")
    wu = torch.zeros(E, H, 2 * I, dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros(E, I, H, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    st = torch.cuda.current_stream().cuda_stream
    _abi.check(_abi.mm_forward(d, x.data_ptr(), ids.data_ptr(), tw.data_ptr(), wu.data_ptr(),
                               wd.data_ptr(), y.data_ptr(), ws.data_ptr(), n, st, 0), "mm_forward")
    counts = torch.empty(E, dtype=torch.int32)
    offsets = torch.empty(E + 1, dtype=torch.int32)
    rows = torch.empty(T * K, dtype=torch.int32)
    _abi.check(_abi.mm_routing_export(d, ws.data_ptr(), counts.data_ptr(), offsets.data_ptr(),
                                      rows.data_ptr(), st), "mm_routing_export")
    return counts, offsets, rows


def _noalloc(fn, w, ids):
    T, E, K = w.T, w.E, w.K
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    rows = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    st = fn(_abi.dims(T, 64, 64, E, K), ids.data_ptr(), counts.data_ptr(), offsets.data_ptr(),
            rows.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == _abi.MM_OK, _abi.mm_status_string(st)
    torch.cuda.synchronize()
    return counts.cpu(), offsets.cpu(), rows.cpu()


def test_noalloc_routing_matches_workspace_routing_on_consecutive_calls():
    fn = _noalloc_fn()
    cases = [synth.BY_NAME["qwen"], synth.BY_NAME["tail"], synth.BY_NAME["skew"]]
    for w in cases:  # consecutive calls, each with different sizes, on the shared scratch
        ids = synth.routing(w).cuda()
        ref = _reference(w, ids)
        got = _noalloc(fn, w, ids)
        for name, a, b in zip(("counts", "offsets", "row_of_slot"), got, ref):
            assert torch.equal(a, b), (w.name, name)
    # and the first case again after the others overwrote the scratch
    w = cases[0]
    ids = synth.routing(w).cuda()
    assert all(torch.equal(a, b) for a, b in zip(_noalloc(fn, w, ids), _reference(w, ids)))


def test_noalloc_rejects_sizes_beyond_its_scratch_and_bad_ids():
    fn = _noalloc_fn()
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    p = buf.data_ptr()
    assert fn(_abi.dims((1 << 20) // 8 + 1, 64, 64, 4, 8), p, p, p, p, st) == _abi.MM_ERR_UNSUPPORTED
    assert fn(_abi.dims(16, 64, 64, 1025, 2), p, p, p, p, st) == _abi.MM_ERR_UNSUPPORTED
    assert fn(_abi.dims(16, 64, 64, 4, 2), 0, p, p, p, st) == _abi.MM_ERR_INVALID_ARG
    w = synth.small("bad", 300, 64, 64, 8, 2)
    ids = synth.routing(w).cuda()
    ids[17, 1] = 8
    counts, offsets, rows = _noalloc(fn, w, ids)
    assert (counts == -1).all() and (offsets == -1).all() and (rows == -1).all()
    # a good call right after restores correct tables
    ids[17, 1] = 3 if int(ids[17, 0]) != 3 else 4
    assert all(torch.equal(a, b) for a, b in zip(_noalloc(fn, w, ids), _reference(w, ids)))
