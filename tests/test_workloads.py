"""The seeded input generator: determinism, slice consistency and routing structure."""
import torch

from workloads import synth


def test_slices_equal_full_draw():
    w = synth.small("t", 5, 24, 8, 3, 2)
    full = synth.x(w)
    assert torch.equal(synth.x(w, rows=[3, 0]), full[[3, 0]])
    assert torch.equal(synth.normal_bf16(synth.stream_key(1, 2), (6, 7), 1.0, chunk=5),
                       synth.normal_bf16(synth.stream_key(1, 2), (6, 7), 1.0))


def test_moments_and_determinism():
    w = synth.BY_NAME["tiny"]
    a, b = synth.x(w), synth.x(w)
    assert torch.equal(a, b)
    f = a.float()
    assert abs(f.mean().item()) < 0.01 and abs(f.std().item() - 1.0) < 0.01
    wu = synth.w_up(w).float()
    assert abs(wu.std().item() - (1 / 512) ** 0.5) < 1e-3


def _distinct(ids):
    s = ids.sort(1).values
    return not (s[:, 1:] == s[:, :-1]).any()


def test_routing_structures():
    for w in synth.WORKLOADS:
        ids = synth.routing(w)
        assert ids.shape == (w.T, w.K) and ids.dtype == torch.int32
        assert int(ids.min()) >= 0 and int(ids.max()) < w.E
        assert _distinct(ids)
        c = torch.bincount(ids.flatten().long(), minlength=w.E)
        if w.routing == "skew":
            assert int(c[0]) == w.T and int(c[14]) == 0 and int(c[15]) == 0
        if w.routing == "hot8":
            assert int(c[:8].sum()) == 2 * w.T   # exactly 25 % of slots
        tw = synth.topk_weights(w)
        assert torch.allclose(tw.sum(1), torch.ones(w.T), atol=1e-5)
    # tail workload: counts not multiples of 128 for most experts
    c = torch.bincount(synth.routing(synth.BY_NAME["tail"]).flatten().long(), minlength=32)
    assert int((c % 128 != 0).sum()) > 16
