"""Attention with separate query and key lengths (KV-cache shapes) against
the fp64 oracle; causal is aligned to the bottom-right corner."""
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


def inputs(B, H, Nq, Nk, d, seed):
    q = wl.make_inputs(B, H, Nq, d, "normal", seed=seed)[0]
    _, k, v = wl.make_inputs(B, H, Nk, d, "normal", seed=seed + 7)
    return q, k, v


SHAPES = [(1, 2, 1, 1000, 128), (1, 2, 7, 4096, 64), (2, 1, 128, 129, 256), (1, 2, 300, 300, 128),
          (1, 3, 200, 1000, 64), (1, 1, 513, 2000, 128), (2, 2, 16, 16384, 128)]


@pytest.mark.parametrize("splits", [1, None], ids=["whole", "auto-split"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES, ids=[f"B{b}H{h}q{nq}k{nk}d{d}" for b, h, nq, nk, d in SHAPES])
def test_kvcache_matches_oracle(B, H, Nq, Nk, d, causal, splits):
    q, k, v = inputs(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    o, lse = ea.attn_fwd_kvcache(q.cuda(), k.cuda(), v.cuda(), causal=causal, num_splits=splits)
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    o_ref, lse_ref = orc().attn_bf16_qk(q, k, v, causal, 1 / math.sqrt(d))
    m = metrics(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)
    record(f"kvcache {(B, H, Nq, Nk, d)} causal={causal} splits={splits}", m)
    assert within(m), describe(m)


def test_more_queries_than_keys_non_causal():
    q, k, v = inputs(1, 2, 1000, 70, 128, seed=3)
    o, lse = ea.attn_fwd_kvcache(q.cuda(), k.cuda(), v.cuda(), causal=False, num_splits=1)
    o_ref, lse_ref = orc().attn_bf16_qk(q, k, v, False, 1 / math.sqrt(128))
    m = metrics(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)
    assert within(m), describe(m)


def test_square_kvcache_is_attn_fwd():
    q, k, v = (t.cuda() for t in wl.make_inputs(1, 2, 777, 128, "normal", seed=5))
    for causal in (False, True):
        o1, l1 = ea.attn_fwd(q, k, v, causal=causal)
        o2, l2 = ea.attn_fwd_kvcache(q, k, v, causal=causal, num_splits=1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_step_is_last_row_of_prefill():
    """One new query against the cache = the last row of the causal attention
    over the whole sequence."""
    B, H, N, d = 1, 4, 5000, 128
    q, k, v = (t.cuda() for t in wl.make_inputs(B, H, N, d, "normal", seed=9))
    o_full, l_full = ea.attn_fwd(q, k, v, causal=True)
    o_dec, l_dec = ea.attn_fwd_kvcache(q[:, :, -1:].contiguous(), k, v, causal=True)
    torch.cuda.synchronize()
    assert (o_dec.float() - o_full[:, :, -1:].float()).abs().max().item() <= 2 * 2 ** -8
    assert (l_dec - l_full[:, :, -1:]).abs().max().item() <= 1e-4
