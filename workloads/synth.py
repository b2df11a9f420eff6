"""Seeded synthetic inputs for the fused MoE-FFN layer.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It only draws inputs; it holds none of the layer's arithmetic.

Values are produced by a counter-based generator written with exact integer
tensor arithmetic, so the same (stream, element index) gives the same value
on the CPU and on a GPU. That lets the large weight tensors be generated
directly in device memory while the oracle regenerates just the slices it
needs (one expert's weights, a few tokens) on the host, bit for bit.

* Normal-like values: the sum of four 16-bit uniforms (Irwin-Hall with n=4),
  centred and scaled to the requested standard deviation, computed as an
  integer and converted to float32 with one correctly rounded multiply, then
  rounded to bf16 (round-to-nearest-even). Its tails stop at about 3.46 sigma.
* Routing (expert ids) and the routing weights are always drawn on the host:
  they are small ([T, K]) and the Zipf routing uses floating-point logs.

The five workloads are the layer shapes used throughout the tests and the
benchmark (tokens T, hidden H, intermediate I, experts E, top-k K).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

M32 = 0xFFFFFFFF


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    routing: str  # "uniform" | "skew" | "zipf" | "hot8"
    seed: int

    @property
    def S(self) -> int:
        return self.T * self.K

    def flops(self) -> dict:
        """Routed-work FLOPs: fwd 6HI, bwd 12HI per slot (no padding counted)."""
        per = self.H * self.I
        return {"fwd": 6 * per * self.S, "bwd": 12 * per * self.S, "total": 18 * per * self.S}


WORKLOADS = [
    Workload("tiny", 1024, 512, 128, 4, 2, "uniform", 1000),
    Workload("skew", 4096, 1024, 512, 16, 4, "skew", 1001),
    Workload("tail", 1000, 2048, 768, 32, 6, "zipf", 1002),
    Workload("qwen", 16384, 2048, 768, 128, 8, "uniform", 1003),
    Workload("large_hidden", 8192, 7168, 2048, 256, 8, "hot8", 1004),
]
BY_NAME = {w.name: w for w in WORKLOADS}

# Stream identifiers (combined with the workload seed into a per-stream key).
STREAM_X, STREAM_WUP, STREAM_WDOWN, STREAM_DY, STREAM_ROUTE, STREAM_TOPKW, STREAM_POS = range(1, 8)
STREAM_SHARED_UP, STREAM_SHARED_DOWN = 8, 9


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer finaliser (xorshift-multiply rounds) on int64 tensors
    holding values in [0, 2^32). Multipliers are below 2^31 so no product
    overflows int64."""
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & M32
    x = x ^ (x >> 15)
    x = (x * 0x2C1B3C6D) & M32
    x = x ^ (x >> 16)
    return x


def _mix32_int(v: int) -> int:
    v &= M32
    v ^= v >> 16
    v = (v * 0x7FEB352D) & M32
    v ^= v >> 15
    v = (v * 0x2C1B3C6D) & M32
    v ^= v >> 16
    return v


def stream_key(seed: int, stream: int) -> int:
    return _mix32_int(_mix32_int(seed * 0x10001 + 0x3C6EF372) ^ (stream * 0x45D9F3B))


def raw_bits(key: int, start: int, count: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Two 32-bit words (as int64 tensors) per element index in [start, start+count)."""
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    lo = i & M32
    hi = i >> 32
    k = _mix32((hi * 0x632BE5AB + key) & M32)
    a = _mix32(lo ^ k)
    b = _mix32(a ^ 0x5BD1E995)
    return a, b


_IH_CENTER = 131070  # 4 * 32767.5
_IH_SD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)


def normal_f32(key: int, start: int, count: int, sigma: float, device="cpu") -> torch.Tensor:
    a, b = raw_bits(key, start, count, device)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _IH_CENTER
    scale = torch.tensor(sigma / _IH_SD, dtype=torch.float32, device=device)
    return s.to(torch.float32) * scale


def normal_bf16(key: int, shape, sigma: float, device="cpu", start: int = 0,
                chunk: int = 1 << 26) -> torch.Tensor:
    """bf16 tensor of `shape` whose flat element j is stream element start+j."""
    n = 1
    for d in shape:
        n *= d
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for c0 in range(0, n, chunk):
        c = min(chunk, n - c0)
        out[c0:c0 + c] = normal_f32(key, start + c0, c, sigma, device).to(torch.bfloat16)
    return out.view(*shape)


# ----------------------------------------------------------------------------- routing

def _uniform_keys(key: int, rows: int, cols: int) -> torch.Tensor:
    a, _ = raw_bits(key, 0, rows * cols)
    return a.view(rows, cols)


def _top_by_key(keys: torch.Tensor, k: int) -> torch.Tensor:
    """Columns of the k largest keys per row (ties: lower column first)."""
    order = torch.sort(keys, dim=1, descending=True, stable=True).indices
    return order[:, :k]


def _shuffle_rows(key: int, ids: torch.Tensor) -> torch.Tensor:
    T, K = ids.shape
    perm = torch.sort(_uniform_keys(key, T, K), dim=1, stable=True).indices
    return torch.gather(ids, 1, perm)


def routing(w: Workload) -> torch.Tensor:
    """topk_ids int32 [T, K]: K distinct experts per token."""
    T, E, K = w.T, w.E, w.K
    key = stream_key(w.seed, STREAM_ROUTE)
    if w.routing == "uniform":
        ids = _top_by_key(_uniform_keys(key, T, E), K)
    elif w.routing == "skew":
        # expert 0 in every token (the feasible maximum share, 1/K of slots),
        # K-1 others uniform over experts 1..E-3; the last two experts stay empty
        rest = _top_by_key(_uniform_keys(key, T, E - 3), K - 1) + 1
        ids = torch.cat([torch.zeros(T, 1, dtype=torch.int64), rest], 1)
        ids = _shuffle_rows(stream_key(w.seed, STREAM_POS), ids)
    elif w.routing == "hot8":
        # exactly two slots per token from hot experts 0..7, the rest uniform
        # over experts 8..E-1: the hot share is exactly 2/K of slots
        hot = _top_by_key(_uniform_keys(key, T, 8), 2)
        cold = _top_by_key(_uniform_keys(key ^ 0x55555555, T, E - 8), K - 2) + 8
        ids = _shuffle_rows(stream_key(w.seed, STREAM_POS), torch.cat([hot, cold], 1))
    elif w.routing == "zipf":
        # Gumbel-top-K sampling without replacement, popularity p_e ~ (e+1)^-1.2
        a = _uniform_keys(key, T, E).to(torch.float64)
        u = (a + 0.5) / 4294967296.0
        logp = -1.2 * torch.log(torch.arange(1, E + 1, dtype=torch.float64))
        ids = _top_by_key(logp[None, :] - torch.log(-torch.log(u)), K)
    else:
        raise ValueError(w.routing)
    return ids.to(torch.int32).contiguous()


def topk_weights(w: Workload) -> torch.Tensor:
    """fp32 [T, K]: softmax over K of normal draws."""
    z = normal_f32(stream_key(w.seed, STREAM_TOPKW), 0, w.T * w.K, 1.0).view(w.T, w.K)
    return torch.softmax(z, dim=1).contiguous()


# ----------------------------------------------------------------------------- tensors

def _token_rows(key, w: Workload, device, rows):
    if rows is None:
        return normal_bf16(key, (w.T, w.H), 1.0, device)
    if isinstance(rows, range) and rows.step == 1:
        return normal_bf16(key, (len(rows), w.H), 1.0, device, start=rows.start * w.H)
    return torch.stack([normal_bf16(key, (w.H,), 1.0, device, start=int(t) * w.H) for t in rows])


def x(w: Workload, device="cpu", rows=None) -> torch.Tensor:
    """bf16 [T, H] ~ N(0,1); `rows` (token indices) draws only those rows."""
    return _token_rows(stream_key(w.seed, STREAM_X), w, device, rows)


def dy(w: Workload, device="cpu", rows=None) -> torch.Tensor:
    """bf16 [T, H] ~ N(0,1): the upstream gradient of y."""
    return _token_rows(stream_key(w.seed, STREAM_DY), w, device, rows)


def w_up(w: Workload, device="cpu", expert=None) -> torch.Tensor:
    """bf16 [E, H, 2I] ~ N(0, 1/H), gate in the first I columns; or one expert's [H, 2I]."""
    key = stream_key(w.seed, STREAM_WUP)
    n = w.H * 2 * w.I
    if expert is None:
        return normal_bf16(key, (w.E, w.H, 2 * w.I), 1.0 / math.sqrt(w.H), device)
    return normal_bf16(key, (w.H, 2 * w.I), 1.0 / math.sqrt(w.H), device, start=int(expert) * n)


def w_down(w: Workload, device="cpu", expert=None) -> torch.Tensor:
    """bf16 [E, I, H] ~ N(0, 1/I); or one expert's [I, H]."""
    key = stream_key(w.seed, STREAM_WDOWN)
    n = w.I * w.H
    if expert is None:
        return normal_bf16(key, (w.E, w.I, w.H), 1.0 / math.sqrt(w.I), device)
    return normal_bf16(key, (w.I, w.H), 1.0 / math.sqrt(w.I), device, start=int(expert) * n)


def shared_up(w: Workload, I_s: int, device="cpu") -> torch.Tensor:
    """Shared expert's bf16 [H, 2*I_s] ~ N(0, 1/H), gate in the first I_s columns."""
    return normal_bf16(stream_key(w.seed, STREAM_SHARED_UP), (w.H, 2 * I_s), 1.0 / math.sqrt(w.H), device)


def shared_down(w: Workload, I_s: int, device="cpu") -> torch.Tensor:
    """Shared expert's bf16 [I_s, H] ~ N(0, 1/I_s)."""
    return normal_bf16(stream_key(w.seed, STREAM_SHARED_DOWN), (I_s, w.H), 1.0 / math.sqrt(I_s), device)


class LazyExperts:
    """Indexable stand-in for a [E, ...] weight tensor that draws one expert on demand
    (host memory holds only the experts actually touched)."""

    def __init__(self, w: Workload, which: str):
        self.w, self.which = w, which
        self.cache = {}
        self.shape = (w.E, w.H, 2 * w.I) if which == "up" else (w.E, w.I, w.H)

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            fn = w_up if self.which == "up" else w_down
            self.cache[e] = fn(self.w, expert=e)
        return self.cache[e]


def small(name: str, T: int, H: int, I: int, E: int, K: int, routing_kind="uniform", seed=7) -> Workload:
    """An ad-hoc workload (edge-case tests)."""
    return Workload(name, T, H, I, E, K, routing_kind, seed)
