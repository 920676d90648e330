"""Split-KV forward against the fp64 oracle and against the single-pass
kernel, through the C ABI (attn_fwd_splitkv + its merge kernel)."""
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


def split_run(q, k, v, causal, splits, scale=None):
    o, lse = ea.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                                 num_splits=splits)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    return o.float().cpu().numpy(), lse.cpu().numpy()


CASES = [(1, 2, 1000, 64, 2), (1, 1, 4096, 128, 4), (2, 1, 777, 256, 3), (1, 3, 300, 128, 8),
         (1, 1, 129, 64, 5), (1, 1, 1, 128, 2), (1, 2, 2048, 128, 64)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,S", CASES, ids=[f"B{b}H{h}N{n}d{d}S{s}" for b, h, n, d, s in CASES])
def test_splitkv_matches_oracle(B, H, N, d, S, causal):
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=N + d + S)
    o, lse = split_run(q, k, v, causal, S)
    o_ref, lse_ref = orc().attn_bf16(q, k, v, causal, 1 / math.sqrt(d))
    m = metrics(o, o_ref, lse, lse_ref)
    record(f"splitkv {(B, H, N, d)} S={S} causal={causal}", m)
    assert within(m), describe(m)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_splitkv_agrees_with_single_pass(causal):
    q, k, v = (t.cuda() for t in wl.make_inputs(1, 4, 3000, 128, "uniform", seed=12))
    o1, l1 = ea.attn_fwd(q, k, v, causal=causal)
    for S in (1, 2, 7):
        o2, l2 = ea.attn_fwd_splitkv(q, k, v, causal=causal, num_splits=S)
        torch.cuda.synchronize()
        d = (o1.float() - o2.float()).abs().max().item()
        assert d <= 2 * 2 ** -8, (S, d)  # two bf16 roundings of the same value
        assert (l1 - l2).abs().max().item() <= 1e-4
        if S == 1:
            assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_splitkv_outliers_sampled_rows():
    w = wl.WORKLOADS["long"]
    q, k, v = wl.make_inputs(1, 4, w.N, w.d, w.dist, w.seed, w.k_outlier_frac)
    o, lse = split_run(q, k, v, True, 6)
    rows = wl.sample_rows(1, 4, w.N, 256, seed=3)
    o_ref, lse_ref = orc().attn_bf16_rows(q, k, v, True, w.scale, rows)
    m = metrics(o.reshape(-1, w.d)[rows], o_ref, lse.reshape(-1)[rows], lse_ref)
    record("splitkv long-shaped 4 heads S=6 causal (sampled rows)", m)
    assert within(m), describe(m)


def test_splitkv_default_split_count():
    q, k, v = (t.cuda() for t in wl.make_inputs(1, 1, 8192, 128, "normal", seed=4))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = ea.attn_fwd_splitkv_num_splits(1, 1, 8192, 128, False, sms)
    assert s > 1
    o, lse = ea.attn_fwd_splitkv(q, k, v)
    o1, l1 = ea.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= 2 * 2 ** -8
