"""Whole-tensor parity at full size: every element of O and LSE of every
benchmark workload against the fp64 oracle.

Each case runs the workload in one call through the C ABI, in the launch
configuration the benchmark times (``attn_fwd``: one fused kernel over all
heads), and compares all B*H*N rows with ``oracle.dense`` -- the plain
definition in fp64 matrix products, pinned against the row-by-row C oracle in
``test_oracle_dense.py``.  Sampled-row checks elsewhere are the quick tier;
these are the ones that would catch a single query tile written wrong.

The e4m3 forward is checked the same way on its quantised inputs (tolerance
derived in ``test_gpu_fp8.py``), and the backward on a whole head group of
the mid workload (the heads one causal launch interleaves) and on the whole
gpt2-shaped problem and on the first heads of the d = 256 workload (tolerance
in ``test_gpu_bwd.py``).
"""
import numpy as np
import pytest
import torch

import exact_attention_51_gb300 as ea
from exact_attention_51_gb300 import workloads as wl
from oracle import dense
from parity import describe, metrics, record, within

pytestmark = pytest.mark.gpu


def _status_ok():
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"


BF16_CASES = [(name, c) for name, w in wl.WORKLOADS.items() for c in w.causal]


@pytest.mark.parametrize("name,causal", BF16_CASES,
                         ids=[f"{n}-{'causal' if c else 'full'}" for n, c in BF16_CASES])
def test_whole_tensor_bf16(name, causal):
    w = wl.WORKLOADS[name]
    q, k, v = wl.workload_inputs(w)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    _status_ok()
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    o_ref, lse_ref = dense.attn_bf16(q, k, v, causal, w.scale)
    m = metrics(o, o_ref, lse, lse_ref)
    record(f"whole tensor {w.describe(causal)}", m)
    assert within(m), f"{w.describe(causal)}: {describe(m)}"


F8_CASES = [(name, c) for name, w in wl.WORKLOADS.items() if w.d in ea.FP8_HEAD_DIMS
            and w.N >= 1024 for c in w.causal]


@pytest.mark.parametrize("name,causal", F8_CASES,
                         ids=[f"{n}-{'causal' if c else 'full'}" for n, c in F8_CASES])
def test_whole_tensor_e4m3(name, causal):
    from test_gpu_fp8 import compare
    w = wl.WORKLOADS[name]
    q8, k8, v8, sc = wl.make_inputs_e4m3(w.B, w.H, w.N, w.d, w.dist, w.seed, w.k_outlier_frac)
    o, lse = ea.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), *sc, causal=causal, scale=w.scale)
    _status_ok()
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    o_ref, lse_ref = dense.attn_e4m3(q8, k8, v8, *sc, causal, w.scale)
    vmax = float(dense.decode_e4m3(v8, sc[2]).abs().max())
    compare(o, o_ref, lse, lse_ref, vmax, f"whole tensor {w.describe(causal)}")


def _bwd_whole(w, causal, heads):
    """attn_bwd over the whole workload in one call; the flat heads `heads`
    (a slice of B*H) compared whole with the dense backward oracle."""
    from test_gpu_bwd import check
    q, k, v = wl.workload_inputs(w)
    g = wl.make_inputs(w.B, w.H, w.N, w.d, w.dist, w.seed + 500)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = ea.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, o, lse, gd, causal=causal)
    _status_ok()
    flat = lambda t: t.reshape(w.B * w.H, 1, w.N, w.d)[heads].reshape(1, -1, w.N, w.d).contiguous()
    ref = dense.attn_bwd_bf16(flat(q), flat(k), flat(v), flat(g), causal, w.scale)
    got = [flat(t.cpu()).float().numpy() for t in (dq, dk, dv)]
    msgs = check(got, ref, f"{w.describe(causal)} heads {heads.start}..{heads.stop - 1}")
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        rel = float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))
        record(f"backward whole heads {w.describe(causal)} {name}",
               {"rel_rms": rel, "max_rel": float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)),
                "heads": [heads.start, heads.stop]})
    assert not msgs, "\n".join(msgs)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_whole_head_group_backward_mid(causal):
    """The mid workload (B=4 H=16 N=4096 d=128): the first 32 heads, the
    group whose K and V one launch keeps in L2 together."""
    _bwd_whole(wl.WORKLOADS["mid"], causal, slice(0, 32))


def test_whole_tensor_backward_gpt2():
    """The gpt2-shaped workload (B=8 H=12 N=1024 d=64, causal), every head."""
    w = wl.WORKLOADS["gpt2"]
    _bwd_whole(w, True, slice(0, w.B * w.H))


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_whole_head_group_backward_dsweep256(causal):
    """The d = 256 workload (B=4 H=16 N=8192): its three backward kernels in
    one call, the first four heads (one causal head group) compared whole."""
    _bwd_whole(wl.WORKLOADS["dsweep256"], causal, slice(0, 4))


KV_CASES = [("long", 16), ("long", 1), ("mid", 16)]


@pytest.mark.parametrize("name,nq", KV_CASES, ids=[f"{n}-q{q}" for n, q in KV_CASES])
def test_whole_tensor_kvcache(name, nq):
    """The KV-cache benchmark's shapes (nq new queries against the
    workload's K/V as the cache, bottom-right causal, the split count
    attn_fwd_kvcache picks): every element of O and LSE."""
    from oracle import Oracle
    w = wl.WORKLOADS[name]
    _, k, v = wl.workload_inputs(w)
    q = wl.make_inputs(w.B, w.H, nq, w.d, w.dist, w.seed + 700)[0]
    o, lse = ea.attn_fwd_kvcache(q.cuda(), k.cuda(), v.cuda(), causal=True)
    _status_ok()
    o_ref, lse_ref = Oracle().attn_bf16_qk(q, k, v, True, w.scale)
    m = metrics(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)
    record(f"whole tensor kvcache {w.describe(True)} nq={nq}", m)
    assert within(m), f"kvcache {name} nq={nq}: {describe(m)}"
