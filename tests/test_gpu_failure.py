"""Failure detection on the GPU without a fault: the bounded-wait self-test
kernel waits on a barrier nothing arrives on, gives up after a short limit and
reports through the device status word; the context stays usable and the
next attention call is correct."""
import math
import time

import numpy as np
import pytest
import torch

import exact_attention_51_gb300 as ea
import oracle
from exact_attention_51_gb300 import workloads as wl
from parity import describe, metrics, within

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    st, _ = ea.attn_fwd_device_status()  # start from a clean status word
    assert st in (ea.ATTN_OK, ea.ATTN_ERR_TIMEOUT)
    t0 = time.perf_counter()
    assert ea.attn_selftest_wait_timeout(200) == ea.ATTN_OK
    st, detail = ea.attn_fwd_device_status()
    elapsed = time.perf_counter() - t0
    assert st == ea.ATTN_ERR_TIMEOUT and detail == 0x1F1, (st, hex(detail))
    assert 0.15 <= elapsed < 5.0, elapsed
    assert ea.attn_fwd_device_status() == (ea.ATTN_OK, 0)  # read-and-clear

    # the context is still usable and the kernels still correct
    q, k, v = wl.make_inputs(1, 2, 300, 128, "normal", seed=11)
    o, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert ea.attn_fwd_device_status() == (ea.ATTN_OK, 0)
    o_ref, lse_ref = oracle.Oracle().attn_bf16(q, k, v, True, 1 / math.sqrt(128))
    m = metrics(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)
    assert within(m), describe(m)


def test_selftest_rejects_out_of_range_limits():
    assert ea.attn_selftest_wait_timeout(0) == ea.ATTN_ERR_INVALID_ARG
    assert ea.attn_selftest_wait_timeout(10001) == ea.ATTN_ERR_INVALID_ARG
