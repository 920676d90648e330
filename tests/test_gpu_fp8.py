"""e4m3 forward (attn_fwd_fp8 through the C ABI) against the fp64 oracle on
the dequantised inputs.

Inputs: the seeded bf16 draws of the other parity tests, quantised per
tensor to e4m3 with a power-of-two scale (``workloads.quantize_e4m3``); the
oracle decodes the same codes by the format's definition and multiplies by
the same scales, so the only differences left are the kernel's own roundings.

Tolerance (derived; neither the pages nor the bf16 bar covers 8-bit P): the
kernel rounds each softmax weight to e4m3 before P V.  A normal e4m3 number
has 3 mantissa bits, so round-to-nearest moves a weight by at most 2^-4 of
itself and, for weights spread log-uniformly over a binade, by about
0.0265 of itself in RMS (2^-4 * sqrt(0.18)).  O is a weighted mean of V, so

    |O_gpu - O_ref| <= 2^-4 * max|V| (+ 2^-8 |O| for the bf16 output),

and with independent rounding errors the RMS of O's error relative to the
RMS of O is about 0.0265 whatever the attention's shape.  Bars: relRMS <=
0.04 (1.5x that), max|dO| <= 0.07 * max|V|, LSE (row max and row sum stay
fp32, scores are exact products of 4-bit mantissas) <= 1e-3 as for bf16.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_51_gb300 as ea
import oracle
from exact_attention_51_gb300 import workloads as wl
from parity import record

pytestmark = pytest.mark.gpu

F8_REL_RMS = 0.04
F8_MAX_OF_VMAX = 0.07
LSE_MAX_ABS = 1e-3
_ORC = None


def orc():
    global _ORC
    if _ORC is None:
        _ORC = oracle.Oracle()
    return _ORC


def run_fp8(q8, k8, v8, sc, causal, scale):
    qd, kd, vd = (t.cuda() for t in (q8, k8, v8))
    o, lse = ea.attn_fwd_fp8(qd, kd, vd, *sc, causal=causal, scale=scale)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def compare(o, o_ref, lse, lse_ref, vmax, label):
    err = np.abs(o - o_ref)
    den = np.linalg.norm(o_ref.ravel())
    rel = float(np.linalg.norm((o - o_ref).ravel()) / den) if den > 0 else float(err.max())
    m = {"o_max_abs": float(err.max()), "o_rel_rms": rel,
         "lse_max_abs": float(np.abs(lse - lse_ref).max()),
         "finite": bool(np.isfinite(o).all() and np.isfinite(lse).all())}
    record(f"e4m3 {label}", m)
    ok = (m["finite"] and rel <= F8_REL_RMS and m["o_max_abs"] <= F8_MAX_OF_VMAX * vmax
          and m["lse_max_abs"] <= LSE_MAX_ABS)
    assert ok, (f"{label}: relRMS {rel:.3e} (<= {F8_REL_RMS}) max {m['o_max_abs']:.3e} "
                f"(<= {F8_MAX_OF_VMAX * vmax:.3e}) lse {m['lse_max_abs']:.3e} finite {m['finite']}")
    return m


SHAPES = [(1, 2, 128), (1, 1, 1), (2, 1, 7), (1, 1, 129), (1, 2, 300), (2, 2, 256), (1, 3, 1000),
          (1, 1, 2049)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N", SHAPES, ids=[f"B{b}H{h}N{n}" for b, h, n in SHAPES])
def test_fp8_small_shapes(B, H, N, causal, d):
    q8, k8, v8, sc = wl.make_inputs_e4m3(B, H, N, d, "normal", seed=7 * N + d + (1 if causal else 0))
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(q8, k8, v8, sc, causal, scale)
    o_ref, lse_ref = orc().attn_e4m3(q8, k8, v8, *sc, causal, scale)
    vmax = float(v8.view(torch.float8_e4m3fn).double().abs().max()) * sc[2]
    compare(o, o_ref, lse, lse_ref, vmax, f"{(B, H, N, d)} causal={causal}")


# small grids run one query tile per CTA (the shapes above); enough heads for
# the default two-tile shape, with ragged tails
FP8_WIDE = [(1, 160, 300, 128), (1, 80, 1100, 64)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", FP8_WIDE, ids=[f"B{b}H{h}N{n}d{d}" for b, h, n, d in FP8_WIDE])
def test_fp8_default_shape_many_heads(B, H, N, d, causal):
    q8, k8, v8, sc = wl.make_inputs_e4m3(B, H, N, d, "normal", seed=11 * N + d + (1 if causal else 0))
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(q8, k8, v8, sc, causal, scale)
    o_ref, lse_ref = orc().attn_e4m3(q8, k8, v8, *sc, causal, scale)
    vmax = float(v8.view(torch.float8_e4m3fn).double().abs().max()) * sc[2]
    compare(o, o_ref, lse, lse_ref, vmax, f"default shape {(B, H, N, d)} causal={causal}")


@pytest.mark.parametrize("name,causal", [("mid", True), ("mid", False), ("long", True),
                                         ("dsweep256", True), ("dsweep64", True)])
def test_fp8_full_size_sampled_rows(name, causal):
    w = wl.WORKLOADS[name]
    q8, k8, v8, sc = wl.make_inputs_e4m3(w.B, w.H, w.N, w.d, w.dist, w.seed, w.k_outlier_frac)
    o, lse = run_fp8(q8, k8, v8, sc, causal, w.scale)
    rows = wl.sample_rows(w.B, w.H, w.N, 384, seed=w.seed)
    o_ref, lse_ref = orc().attn_e4m3(q8, k8, v8, *sc, causal, w.scale, rows=rows)
    o_s = o.reshape(-1, w.d)[rows]
    lse_s = lse.reshape(-1)[rows]
    vmax = float(v8.view(torch.float8_e4m3fn).double().abs().max()) * sc[2]
    compare(o_s, o_ref, lse_s, lse_ref, vmax, f"{name} causal={causal} rows={len(rows)}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_fp8_zero_keys_exact_weights(causal, d):
    """K = 0: every visible score is 0, so every e4m3 weight is exactly 2^4
    (no rounding): O_i = mean of the visible V rows, LSE_i = ln(#visible), to
    the bf16 bar."""
    B, H, N = 1, 2, 300
    q8, _, v8, sc = wl.make_inputs_e4m3(B, H, N, d, "normal", seed=3)
    k8 = torch.zeros_like(q8)
    o, lse = run_fp8(q8, k8, v8, (sc[0], 1.0, sc[2]), causal, 1 / math.sqrt(d))
    vd = v8.view(torch.float8_e4m3fn).double().numpy() * sc[2]
    if causal:
        ref = np.cumsum(vd, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        lref = np.log(np.arange(1, N + 1, dtype=np.float64))[None, None, :].repeat(H, 1)
    else:
        ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
        lref = np.full((B, H, N), math.log(N))
    assert np.abs(o - ref).max() <= 2e-2
    assert np.linalg.norm((o - ref).ravel()) / np.linalg.norm(ref.ravel()) <= 5e-3
    assert np.abs(lse - lref).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_single_key_returns_v(d):
    """N = 1: the one weight is exactly 2^4, so O = descale_v * V8 (exact in
    bf16: 4 significant bits times a power of two) and LSE = scale * s."""
    B, H, N = 2, 3, 1
    q8, k8, v8, sc = wl.make_inputs_e4m3(B, H, N, d, "normal", seed=11)
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(q8, k8, v8, sc, False, scale)
    vd = v8.view(torch.float8_e4m3fn).double().numpy() * sc[2]
    assert np.array_equal(o, vd)
    s = (q8.view(torch.float8_e4m3fn).double() * k8.view(torch.float8_e4m3fn).double()).sum(-1)
    assert np.abs(lse - (s.numpy() * sc[0] * sc[1] * scale)).max() <= 1e-3


KV_SHAPES = [(1, 2, 1, 1000, 128), (1, 2, 7, 4096, 128), (2, 1, 128, 129, 256),
             (1, 2, 300, 300, 128), (1, 1, 513, 2000, 256), (2, 2, 16, 16384, 128),
             (1, 3, 200, 777, 64), (2, 2, 5, 3000, 64)]


@pytest.mark.parametrize("splits", [1, None], ids=["whole", "auto-split"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", KV_SHAPES,
                         ids=[f"B{b}H{h}q{nq}k{nk}d{d}" for b, h, nq, nk, d in KV_SHAPES])
def test_fp8_kvcache(B, H, Nq, Nk, d, causal, splits):
    """Queries as the last Nq positions of Nk (bottom-right causal diagonal),
    whole and split-KV, against the oracle on the dequantised codes."""
    q = wl.make_inputs(B, H, Nq, d, "normal", seed=Nq + d)[0]
    _, k, v = wl.make_inputs(B, H, Nk, d, "normal", seed=Nk + d + 1)
    (q8, sq), (k8, sk), (v8, sv) = (wl.quantize_e4m3(t.float()) for t in (q, k, v))
    scale = 1 / math.sqrt(d)
    o, lse = ea.attn_fwd_fp8_kvcache(q8.cuda(), k8.cuda(), v8.cuda(), sq, sk, sv, causal=causal,
                                     scale=scale, num_splits=splits)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    o_ref, lse_ref = orc().attn_e4m3_qk(q8, k8, v8, sq, sk, sv, causal, scale)
    vmax = float(v8.view(torch.float8_e4m3fn).double().abs().max()) * sv
    compare(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, vmax,
            f"kvcache {(B, H, Nq, Nk, d)} causal={causal} splits={splits}")
