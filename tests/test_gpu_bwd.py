"""Backward pass (attn_bwd through the C ABI) against the fp64 backward
oracle on the same bf16 inputs.

Tolerance (no figure on the pages or in the forward's bar): per gradient
tensor, ||dX_gpu - dX_ref||_2 / ||dX_ref||_2 <= 2e-2 and
max|dX_gpu - dX_ref| <= 5e-2 * max|dX_ref|.  The kernel rounds P and dS to
bf16 (relative 2^-9 each) before the tensor-core products, computes D from
the forward's bf16 O, and rounds the outputs to bf16 (2^-9); dS = P(dP - D)
loses relative precision where dP ~ D, so the bound keeps about an order of
magnitude above those unit roundings.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_51_gb300 as ea
import oracle
from exact_attention_51_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

REL_RMS = 2e-2
REL_MAX = 5e-2
_ORC = None


def orc():
    global _ORC
    if _ORC is None:
        _ORC = oracle.Oracle()
    return _ORC


def grads(B, H, N, d, causal, seed, scale=None):
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=seed)
    g = wl.make_inputs(B, H, N, d, "normal", seed=seed + 50)[0]
    scale = 1 / math.sqrt(d) if scale is None else scale
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, o, lse, gd, causal=causal, scale=scale)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    ref = orc().attn_bwd_bf16(q, k, v, g, causal, scale)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)], ref


def check(got, ref, label):
    msgs = []
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        rel = np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30)
        mx = np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)
        if not (np.all(np.isfinite(a)) and rel <= REL_RMS and mx <= REL_MAX):
            msgs.append(f"{label} {name}: relRMS {rel:.2e} (<= {REL_RMS}) max {mx:.2e} (<= {REL_MAX})")
    return msgs


# d = 256 runs its own kernels (64-row streamed tiles): ragged against both
# 64 and 128, a single tile, several 128-row blocks
SHAPES = [(1, 2, 128, 64), (2, 1, 300, 128), (1, 2, 513, 64), (1, 1, 1000, 128), (1, 1, 2, 64),
          (1, 2, 300, 256), (2, 1, 64, 256), (1, 1, 1000, 256), (1, 1, 3, 256)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", SHAPES, ids=[f"B{b}H{h}N{n}d{d}" for b, h, n, d in SHAPES])
def test_backward_matches_oracle(B, H, N, d, causal):
    got, ref = grads(B, H, N, d, causal, seed=N + d)
    msgs = check(got, ref, f"{(B, H, N, d)} causal={causal}")
    assert not msgs, "\n".join(msgs)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_single_key(d, causal):
    """N = 1: P = [1], so dV = dO and dQ = dK = 0 exactly (dS = 1*(dP - D)
    with D = dP).  The kernel forms dP on the tensor cores and D from the
    bf16 O = V in fp32, so dP - D is a rounding residual of two d-term fp32
    sums.  Taken as 2^-23 per addition on each side (the tensor cores' adder
    is not documented as round-to-nearest), doubled for slack:
    |dS| <= 2 d 2^-22 sum_c |dO_c V_c|, and dQ_c = scale * dS * K_c,
    dK_c = scale * dS * Q_c."""
    B, H, N = 2, 3, 1
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=7)
    g = wl.make_inputs(B, H, N, d, "normal", seed=8)[0]
    scale = 1 / math.sqrt(d)
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, o, lse, gd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(dv.cpu(), g), "dV must equal dO when one key is visible"
    ds_bound = 2 * d * 2.0**-22 * (g.double() * v.double()).abs().sum(-1, keepdim=True)
    for got, other in ((dq, k), (dk, q)):
        bound = 1.01 * scale * ds_bound * other.double().abs()
        assert bool((got.double().cpu().abs() <= bound).all())


def test_backward_sums():
    """sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 per head (non-causal and
    causal), up to the bf16 output rounding."""
    B, H, N, d = 1, 2, 700, 128
    q, k, v, g = (t.cuda() for t in wl.make_inputs(B, H, N, d, "normal", seed=1) + (
        wl.make_inputs(B, H, N, d, "normal", seed=99)[0],))
    for causal in (False, True):
        o, lse = ea.attn_fwd(q, k, v, causal=causal)
        dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, g, causal=causal)
        torch.cuda.synchronize()
        sv = dv.double().sum(2)
        sg = g.double().sum(2)
        assert (sv - sg).abs().max().item() <= 0.05 * sg.abs().max().item() + 0.05
        assert dk.double().sum(2).abs().max().item() <= 0.05 * dk.double().abs().sum(2).max().item()


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_backward_full_size_sampled_heads(causal):
    """The mid workload (B=4 H=16 N=4096 d=128) in one call; two heads
    compared whole against the fp64 oracle run on those heads alone."""
    w = wl.WORKLOADS["mid"]
    q, k, v = wl.workload_inputs(w)
    g = wl.make_inputs(w.B, w.H, w.N, w.d, w.dist, w.seed + 500)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, o, lse, gd, causal=causal)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
        ref = orc().attn_bwd_bf16(sl(q), sl(k), sl(v), sl(g), causal, w.scale)
        got = [sl(t).float().cpu().numpy() for t in (dq, dk, dv)]
        msgs = check(got, ref, f"mid head ({b},{h}) causal={causal}")
        assert not msgs, "\n".join(msgs)


def test_backward_long_column_sums():
    """The long workload (B=1 H=32 N=16384, 1% of K rows x8), causal, in one
    call; properties that hold at any size: per head, sum_j dV_j = sum_i dO_i
    and sum_j dK_j = 0 (softmax rows sum to one), up to bf16 rounding."""
    w = wl.WORKLOADS["long"]
    q, k, v = (t.cuda() for t in wl.workload_inputs(w))
    g = wl.make_inputs(w.B, w.H, w.N, w.d, w.dist, w.seed + 500)[0].cuda()
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, g, causal=True)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    assert bool(torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all())
    sv, sg = dv.double().sum(2), g.double().sum(2)
    assert (sv - sg).abs().max().item() <= 0.02 * sg.abs().max().item() + 0.5
    sk = dk.double().sum(2)
    assert sk.abs().max().item() <= 0.02 * dk.double().abs().sum(2).max().item()
