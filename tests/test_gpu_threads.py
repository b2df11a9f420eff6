"""Two host threads, each running forward + backward steps on its own stream and workspace at the
same time, get the same bits as one thread running them in turn (each thread forks and joins its
own library side stream)."""
import threading

import pytest
import torch

from layer_harness import make_inputs, run_layer
from moe_ffn_expert_gb300 import _abi
from workloads import synth

pytestmark = pytest.mark.gpu


def test_concurrent_calls_from_two_threads():
    cases = [make_inputs(synth.small(f"thr{i}", 2000, 256, 128, 6, 2, seed=300 + i)) for i in range(2)]
    refs = [run_layer(inp) for inp in cases]
    torch.cuda.synchronize()
    results = [[], []]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(6):
                    out = run_layer(cases[i], stream=s)
                    results[i].append({k: out[k].clone() for k in
                                       ("y", "dx", "d_topk_weights", "dW_up", "dW_down")} |
                                      {"status": out["status"]})
            s.synchronize()
        except Exception as exc:  # reported below, on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert len(results[i]) == 6
        for out in results[i]:
            assert out["status"] == _abi.MM_OK
            for k in ("y", "dx", "d_topk_weights", "dW_up", "dW_down"):
                assert torch.equal(out[k], refs[i][k]), (i, k)
