"""A layer step run by a C program through include/mm.h and libmm.so (no Python or PyTorch in
that process) equals the same step through the Python binding bit for bit."""
import subprocess

import pytest
import torch

from c_abi_util import build_layer_step
from layer_harness import make_inputs, run_layer
from workloads import synth

pytestmark = pytest.mark.gpu


def _raw(t):
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().tobytes()


@pytest.mark.parametrize("T,H,I,E,K", [(1536, 256, 128, 4, 2), (333, 136, 72, 9, 3)])
def test_c_program_step_equals_python_binding(tmp_path, T, H, I, E, K):
    exe = build_layer_step(str(tmp_path))
    w = synth.small("c_abi", T, H, I, E, K, seed=77)
    inp = make_inputs(w)
    for name, key in (("x", "x"), ("ids", "topk_ids"), ("tw", "topk_weights"), ("wu", "w_up"),
                      ("wd", "w_down"), ("dy", "dy")):
        t = inp[key].to(torch.int32) if key == "topk_ids" else inp[key]
        (tmp_path / f"{name}.bin").write_bytes(_raw(t))
    r = subprocess.run([exe, str(tmp_path), str(T), str(H), str(I), str(E), str(K)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    ref = run_layer(inp)
    for name, key in (("y", "y"), ("dx", "dx"), ("dtk", "d_topk_weights"), ("du", "dW_up"),
                      ("dd", "dW_down")):
        got = (tmp_path / f"{name}.bin").read_bytes()
        assert got == _raw(ref[key]), name
