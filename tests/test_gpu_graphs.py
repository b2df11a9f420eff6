"""A forward + backward step captured into a CUDA graph and replayed.

mm_forward and mm_backward only enqueue work on the caller's stream (the backward forks one
library stream for Combine(dX) and joins it back with events), so a training step can be
captured once and replayed with new inputs copied into the captured buffers. The replays must
equal eager calls bit for bit."""
import pytest
import torch

from moe_ffn_expert_gb300 import _abi
from layer_harness import make_inputs, run_layer
from workloads import synth

pytestmark = pytest.mark.gpu

NAMES = ("x", "topk_ids", "topk_weights", "w_up", "w_down", "dy")


def _step(inp, bufs, st):
    d, ws, nbytes = bufs["dims"], bufs["ws"], bufs["nbytes"]
    x, ids, tw, wu, wd, dy = (inp[k] for k in NAMES)
    _abi.check(_abi.mm_forward(d, x.data_ptr(), ids.data_ptr(), tw.data_ptr(), wu.data_ptr(),
                               wd.data_ptr(), bufs["y"].data_ptr(), ws.data_ptr(), nbytes, st, 0),
               "mm_forward")
    _abi.check(_abi.mm_backward(d, dy.data_ptr(), x.data_ptr(), ids.data_ptr(), tw.data_ptr(),
                                wu.data_ptr(), wd.data_ptr(), ws.data_ptr(), nbytes,
                                bufs["dx"].data_ptr(), bufs["d_topk"].data_ptr(),
                                bufs["d_up"].data_ptr(), bufs["d_down"].data_ptr(), st, 0),
               "mm_backward")


@pytest.mark.parametrize("T,H,I,E,K", [(2000, 256, 128, 6, 2),     # pair-MMA weight gradients
                                       (700, 136, 72, 20, 3)])     # one-CTA weight gradients
def test_forward_backward_step_replays_from_a_cuda_graph(T, H, I, E, K):
    inputs = [make_inputs(synth.small(f"graph{i}", T, H, I, E, K, seed=41 + i)) for i in range(2)]
    d = _abi.dims(T, H, I, E, K)
    nbytes = _abi.mm_workspace_size(d)
    dev = inputs[0]["x"].device
    bufs = dict(dims=d, nbytes=nbytes, ws=torch.empty(nbytes, dtype=torch.uint8, device=dev),
                y=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                dx=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                d_topk=torch.empty(T, K, dtype=torch.float32, device=dev),
                d_up=torch.empty(E, H, 2 * I, dtype=torch.bfloat16, device=dev),
                d_down=torch.empty(E, I, H, dtype=torch.bfloat16, device=dev))
    static = {k: inputs[0][k].clone() for k in NAMES}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager step first: the library's one-time set-up
        _step(static, bufs, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(static, bufs, s.cuda_stream)
    for src in (inputs[1], inputs[0], inputs[1]):
        for k in NAMES:
            static[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        st = torch.cuda.current_stream().cuda_stream
        assert _abi.mm_get_status(bufs["ws"].data_ptr(), st) == _abi.MM_OK
        ref = run_layer(src)
        for name, got in (("y", bufs["y"]), ("dx", bufs["dx"]), ("d_topk_weights", bufs["d_topk"]),
                          ("dW_up", bufs["d_up"]), ("dW_down", bufs["d_down"])):
            assert torch.equal(got, ref[name]), name
