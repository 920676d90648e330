"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and names the workloads; it holds none
of the attention arithmetic.  It is the one piece shared by the tests, the
benchmark and the CPU oracle's callers, so that the CUDA path and the oracle
read byte-identical bf16 tensors.

Recipe: fp32 draws from a CPU ``torch.Generator`` seeded per tensor, rounded
to bf16 (round-to-nearest-even, ``Tensor.to``), then copied to the device by
the caller.  Seeds are ``base + {0: Q, 1: K, 2: V, 3: outlier-row choice}``.
The long-sequence workload scales a seeded random choice of round(0.01*N) key
rows per (b, h) by 8, which is exact in bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # causal flags this workload is run with
    dist: str  # "normal" (N(0,1)) or "uniform" (U(-1,1))
    seed: int
    k_outlier_frac: float = 0.0  # fraction of K rows per (b,h) scaled by 8
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self, causal: bool) -> float:
        """Algorithmic FLOPs: 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if causal else f

    def min_hbm_bytes(self) -> int:
        """Read Q, K, V once, write O once (bf16) and LSE once (fp32)."""
        return 4 * self.B * self.H * self.N * self.d * 2 + 4 * self.B * self.H * self.N

    def describe(self, causal: bool) -> str:
        c = "causal" if causal else "non-causal"
        s = f"{self.name}: B={self.B} H={self.H} N={self.N} d={self.d} {c} bf16 {self.dist}"
        if self.k_outlier_frac:
            s += f", {self.k_outlier_frac:.0%} of K rows x8"
        return s


# The five workload families (the d-sweep contributes three entries).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 64, (False, True), "normal", 1000),
    "gpt2": Workload("gpt2", 8, 12, 1024, 64, (True,), "normal", 2000),
    "mid": Workload("mid", 4, 16, 4096, 128, (False, True), "normal", 3000),
    "long": Workload("long", 1, 32, 16384, 128, (True,), "normal", 4000,
                     k_outlier_frac=0.01),
    "dsweep64": Workload("dsweep64", 4, 16, 8192, 64, (False, True), "uniform", 5000),
    "dsweep128": Workload("dsweep128", 4, 16, 8192, 128, (False, True), "uniform", 5100),
    "dsweep256": Workload("dsweep256", 4, 16, 8192, 256, (False, True), "uniform", 5200),
    # not one of the five workload families: a narrow launch (B*H*N/256 = 128
    # query blocks < the SM count) where split-KV is meant to help
    "narrow": Workload("narrow", 1, 4, 8192, 128, (False, True), "normal", 6000),
}


def _draw(shape, dist: str, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.bfloat16)


def make_inputs(B: int, H: int, N: int, d: int, dist: str = "normal", seed: int = 0,
                k_outlier_frac: float = 0.0):
    """Return bf16 CPU tensors (q, k, v), contiguous [B, H, N, d]."""
    shape = (B, H, N, d)
    q = _draw(shape, dist, seed + 0)
    k = _draw(shape, dist, seed + 1)
    v = _draw(shape, dist, seed + 2)
    if k_outlier_frac > 0.0:
        n_out = int(round(k_outlier_frac * N))
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed + 3))
        kv = k.view(B * H, N, d)
        for bh in range(B * H):
            idx = torch.randperm(N, generator=g)[:n_out]
            kv[bh, idx] = kv[bh, idx] * 8  # power of two: exact in bf16
    return q, k, v


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.N, w.d, w.dist, w.seed, w.k_outlier_frac)


def sample_rows(B: int, H: int, N: int, count: int, seed: int = 0, tile: int = 128):
    """Flat row ids ((b*H+h)*N + i) to check at full size.

    Always includes the first and last rows of every head that is sampled,
    rows on both sides of each 128-row tile boundary near the start, middle
    and end, plus seeded random rows.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 77)
    rows = set()
    BH = B * H
    heads = sorted(set([0, BH - 1] + torch.randint(0, BH, (4,), generator=g).tolist()))
    special = {0, 1, N - 1, N - 2}
    for t in (tile, N // 2 - (N // 2) % tile, N - (N % tile or tile)):
        for delta in (-1, 0, 1, tile - 1):
            special.add(t + delta)
    special = {i for i in special if 0 <= i < N}
    for bh in heads:
        for i in special:
            rows.add(bh * N + i)
    count = min(count, BH * N)
    while len(rows) < count:
        rows.add(int(torch.randint(0, BH * N, (1,), generator=g).item()))
    return sorted(rows)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 codes of a CPU tensor: ``(codes uint8, descale)`` with
    descale the power of two 2^ceil(log2(amax / 448)), so that every
    |x| / descale fits the format's largest finite value (448) and
    ``descale * decode(codes)`` is the value the attention sees.  Rounding is
    torch's round-to-nearest-even conversion to ``float8_e4m3fn``."""
    amax = float(x.abs().max())
    descale = 2.0 ** math.ceil(math.log2(amax / 448.0)) if amax > 0 else 1.0
    codes = (x.float() / descale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), descale


def make_inputs_e4m3(B: int, H: int, N: int, d: int, dist: str, seed: int,
                     k_outlier_frac: float = 0.0):
    """``make_inputs`` drawn the same way, then each tensor quantised to e4m3
    with its own power-of-two scale: returns ``(q8, k8, v8, (sq, sk, sv))``
    as uint8 CPU tensors and floats."""
    q, k, v = make_inputs(B, H, N, d, dist, seed, k_outlier_frac)
    (q8, sq), (k8, sk), (v8, sv) = (quantize_e4m3(t.float()) for t in (q, k, v))
    return q8, k8, v8, (sq, sk, sv)
