"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every case draws seeded bf16 inputs on the CPU, runs ``attn_fwd`` on the GPU
and compares with the oracle on the same bf16 bytes, using the tolerances in
``parity.py``.  Small shapes are compared element by element (several tiles
plus ragged tails); the full-size workloads are compared on sampled rows that
the oracle computes one by one.  Every case also checks that no device-side
wait timed out.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_51_gb300 as ea
import oracle
from exact_attention_51_gb300 import workloads as wl
from parity import describe, metrics, record, within

pytestmark = pytest.mark.gpu

_ORC = None


def orc():
    global _ORC
    if _ORC is None:
        _ORC = oracle.Oracle()
    return _ORC


def run_gpu(q, k, v, causal, scale=None):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_full(q, k, v, causal, scale=None, label=""):
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = orc().attn_bf16(q, k, v, causal, scale)
    m = metrics(o, o_ref, lse, lse_ref)
    record(f"{label} {tuple(q.shape)} causal={causal} scale={scale:.4g}", m)
    assert within(m), f"{label} {tuple(q.shape)} causal={causal}: {describe(m)}"
    return m


# ----------------------------------------------------------- small, full tensor

SMALL_SHAPES = [(1, 2, 128), (1, 1, 1), (2, 1, 7), (1, 1, 127), (1, 2, 129), (1, 1, 255),
                (2, 2, 256), (1, 1, 300), (1, 1, 513), (1, 3, 1000)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N", SMALL_SHAPES, ids=[f"B{b}H{h}N{n}" for b, h, n in SMALL_SHAPES])
def test_small_shapes(B, H, N, d, causal):
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=10 * N + d + (1 if causal else 0))
    check_full(q, k, v, causal, label="small")


# head dim 64 runs two CTAs per SM with one query tile each up to 1024 keys
# and two query tiles per CTA beyond: both shapes, with ragged tails, on
# either side of the switch
D64_SHAPES = [(1, 2, 1023), (1, 1, 1024), (1, 2, 1025), (2, 1, 1300), (1, 1, 2049)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N", D64_SHAPES, ids=[f"B{b}H{h}N{n}" for b, h, n in D64_SHAPES])
def test_d64_both_shapes(B, H, N, causal):
    q, k, v = wl.make_inputs(B, H, N, 64, "normal", seed=3 * N + (1 if causal else 0))
    check_full(q, k, v, causal, label="d64 shape switch")


# d = 64 and 128 run one query tile per CTA when two per CTA would not fill
# the GPU once (the small shapes above); with enough heads the launch takes
# the default two-tile shape: ragged tails there too
WIDE_SHAPES = [(1, 160, 300, 128), (2, 80, 129, 128), (1, 80, 1100, 64)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", WIDE_SHAPES, ids=[f"B{b}H{h}N{n}d{d}" for b, h, n, d in WIDE_SHAPES])
def test_default_shape_many_heads(B, H, N, d, causal):
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=5 * N + d + (1 if causal else 0))
    check_full(q, k, v, causal, label="default shape")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_tiny_workload_full_tensor(causal):
    w = wl.WORKLOADS["tiny"]
    q, k, v = wl.workload_inputs(w)
    check_full(q, k, v, causal, label="tiny")


# ------------------------------------------------------- invariants on the GPU

@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_zero_keys_give_uniform_weights(d, causal):
    """K = 0 makes every visible score 0: O_i = mean of the visible V rows and
    LSE_i = ln(#visible).  Exercises the P.V product independently of Q.K^T."""
    B, H, N = 1, 2, 300
    q, _, v = wl.make_inputs(B, H, N, d, "normal", seed=77 + d)
    k = torch.zeros_like(q)
    o, lse = run_gpu(q, k, v, causal)
    vf = v.double().numpy()
    if causal:
        ref = np.cumsum(vf, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        lref = np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape)
    else:
        ref = np.broadcast_to(vf.mean(axis=2, keepdims=True), o.shape)
        lref = np.full(lse.shape, math.log(N))
    m = metrics(o, ref, lse, lref)
    assert within(m), describe(m)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_identity_values_expose_probabilities(d, causal):
    """V = I (N = d) makes O the probability matrix P: rows sum to 1 and match
    the oracle's P.  Exercises Q.K^T and the softmax independently of V."""
    N = d
    q, k, _ = wl.make_inputs(1, 1, N, d, "normal", seed=91 + d)
    v = torch.eye(N, dtype=torch.bfloat16).reshape(1, 1, N, d)
    o, lse = run_gpu(q, k, v, causal)
    o_ref, lse_ref = orc().attn_bf16(q, k, v, causal, 1.0 / math.sqrt(d))
    assert np.abs(o.sum(-1) - 1.0).max() < 2e-2
    m = metrics(o, o_ref, lse, lse_ref)
    assert within(m), describe(m)
    if causal:
        assert np.all(np.triu(o[0, 0], 1) == 0), "weight on a future key"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_constant_values(d):
    q, k, _ = wl.make_inputs(1, 2, 700, d, "normal", seed=5 + d)
    v = torch.full_like(q, -1.75)
    for causal in (False, True):
        o, _ = run_gpu(q, k, v, causal)
        assert np.abs(o + 1.75).max() <= 2e-2


@pytest.mark.parametrize("d", [64, 128, 256])
def test_single_key(d):
    """N = 1: O = V and LSE = scale * q.k."""
    q, k, v = wl.make_inputs(3, 2, 1, d, "normal", seed=3 + d)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal)
        assert np.array_equal(o, v.float().numpy())
        ref = (q.double() * k.double()).sum(-1).numpy() / math.sqrt(d)
        assert np.abs(lse - ref).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 128, 256])
def test_permutation_invariance(d):
    q, k, v = wl.make_inputs(1, 2, 333, d, "normal", seed=17 + d)
    perm = torch.randperm(333, generator=torch.Generator().manual_seed(1))
    o1, l1 = run_gpu(q, k, v, False)
    o2, l2 = run_gpu(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False)
    m = metrics(o2, o1, l2, l1)
    assert within(m), describe(m)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_causal_ignores_future_keys(d):
    N, t = 600, 250
    q, k, v = wl.make_inputs(1, 1, N, d, "normal", seed=29 + d)
    o1, l1 = run_gpu(q, k, v, True)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, t + 1:] = 30.0
    v2[:, :, t + 1:] = 1000.0
    o2, l2 = run_gpu(q, k2, v2, True)
    assert np.array_equal(o1[:, :, :t + 1], o2[:, :, :t + 1])
    assert np.array_equal(l1[:, :, :t + 1], l2[:, :, :t + 1])


@pytest.mark.parametrize("scale", [0.0, 1.0, 0.02])
def test_scale_values(scale):
    q, k, v = wl.make_inputs(1, 2, 400, 128, "normal", seed=int(scale * 100) + 1)
    for causal in (False, True):
        check_full(q, k, v, causal, scale=scale, label=f"scale={scale}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_peaked_rows_many_tiles(d, scale):
    """Large scores over several key tiles: row maxima grow tile after tile
    while the exponent offset stays stale (up to the rescale threshold), so
    dominant weights are not exactly 1 when rounded into P."""
    q, k, v = wl.make_inputs(1, 2, 1000, d, "normal", seed=int(scale * 10) + d)
    for causal in (False, True):
        check_full(q, k, v, causal, scale=scale, label=f"peaked scale={scale}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("step", [2.8, 4.2], ids=["no-rescale", "one-rescale"])
def test_row_max_growing_tile_by_tile(d, step):
    """Scores that grow by `step` (natural units) per 128-key tile along a
    fixed direction: over 8 tiles a row's maximum rises by about 28 or 42
    (log2 units), so the exponent offset stays stale for many tiles (P up to
    about 2^28) or moves once past the rescale threshold.  Whole tensor
    against the oracle, at scale 1."""
    B, H, N = 1, 2, 1024
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=int(step * 10) + d)
    q = (q.float() * 0.1).to(torch.bfloat16)
    k = (k.float() * 0.1).to(torch.bfloat16)
    q[..., 0] = 1.0
    k[..., 0] = (step * (torch.arange(N) // 128).float()).to(torch.bfloat16).view(1, 1, N)
    for causal in (False, True):
        check_full(q, k, v, causal, scale=1.0, label=f"growing max step={step}")


def test_outlier_keys_small():
    q, k, v = wl.make_inputs(1, 4, 1500, 128, "normal", seed=4321, k_outlier_frac=0.01)
    for causal in (False, True):
        check_full(q, k, v, causal, label="outliers")


def test_deterministic():
    q, k, v = wl.make_inputs(2, 3, 1111, 128, "uniform", seed=8)
    for causal in (False, True):
        a = run_gpu(q, k, v, causal)
        b = run_gpu(q, k, v, causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_out_parameters_and_stream():
    q, k, v = (t.cuda() for t in wl.make_inputs(1, 2, 256, 64, "normal", seed=9))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((1, 2, 256), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = ea.attn_fwd(q, k, v, causal=True, out=out, lse=lse)
    s.synchronize()
    assert o2.data_ptr() == out.data_ptr() and l2.data_ptr() == lse.data_ptr()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    ref_o, ref_l = ea.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(ref_o, out) and torch.equal(ref_l, lse)


def test_cuda_graph_replay():
    """attn_fwd enqueues one kernel and allocates nothing, so a captured CUDA
    graph replays it: new inputs copied into the captured buffers give the
    same bytes as an eager call (the way to amortise launch cost for short
    sequences)."""
    q, k, v = (t.cuda() for t in wl.make_inputs(2, 3, 300, 128, "normal", seed=21))
    out = torch.empty_like(q)
    lse = torch.empty((2, 3, 300), device="cuda")
    ea.attn_fwd(q, k, v, causal=True, out=out, lse=lse)  # first call: per-device set-up
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ea.attn_fwd(q, k, v, causal=True, out=out, lse=lse)
    for seed in (22, 23):
        q2, k2, v2 = (t.cuda() for t in wl.make_inputs(2, 3, 300, 128, "normal", seed=seed))
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = ea.attn_fwd(q2, k2, v2, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(ref_o, out) and torch.equal(ref_l, lse)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"


# ------------------------------------------------ full-size workloads, sampled

WL_CASES = [(name, c) for name, w in wl.WORKLOADS.items() if name != "tiny" for c in w.causal]


@pytest.mark.parametrize("name,causal", WL_CASES,
                         ids=[f"{n}-{'causal' if c else 'full'}" for n, c in WL_CASES])
def test_workload_sampled_rows(name, causal):
    w = wl.WORKLOADS[name]
    q, k, v = wl.workload_inputs(w)
    o, lse = run_gpu(q, k, v, causal)
    rows = wl.sample_rows(w.B, w.H, w.N, 384, seed=w.seed)
    o_ref, lse_ref = orc().attn_bf16_rows(q, k, v, causal, w.scale, rows)
    o_s = o.reshape(-1, w.d)[rows]
    l_s = lse.reshape(-1)[rows]
    m = metrics(o_s, o_ref, l_s, lse_ref)
    record(f"workload {w.describe(causal)} ({len(rows)} sampled rows)", m)
    assert within(m), f"{w.describe(causal)}: {describe(m)}"
    # properties that hold at any size, checked on every row
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    vmax = float(v.abs().max())
    assert np.abs(o).max() <= vmax * (1 + 2 ** -7)  # a convex combination of value rows


def test_long_sequence_single_head():
    """N = 2^18 keys (a long row: 2048 key tiles), sampled rows."""
    B, H, N, d = 1, 1, 1 << 18, 64
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=2718)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal)
        rows = [0, 1, 127, 128, 255, 256, N // 2, N - 257, N - 2, N - 1]
        o_ref, lse_ref = orc().attn_bf16_rows(q, k, v, causal, 1 / 8, rows)
        m = metrics(o.reshape(-1, d)[rows], o_ref, lse.reshape(-1)[rows], lse_ref)
        assert within(m), describe(m)


def test_many_heads():
    """B*H = 8192 heads of N = 130 (ragged 2-tile heads): the grid's head axis."""
    B, H, N, d = 64, 128, 130, 64
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=31)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal)
        rows = wl.sample_rows(B, H, N, 512, seed=5)
        o_ref, lse_ref = orc().attn_bf16_rows(q, k, v, causal, 1 / 8, rows)
        m = metrics(o.reshape(-1, d)[rows], o_ref, lse.reshape(-1)[rows], lse_ref)
        assert within(m), describe(m)
