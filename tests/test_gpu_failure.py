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


# codes a wait of the fused kernel records: producer (empty slot), MMA warp
# (Q, K/V, P), softmax (S, O, final O)
KERNEL_WAIT_CODES = {0x101, 0x111, 0x112, 0x113, 0x121, 0x122, 0x123}


@pytest.mark.parametrize("d,causal,drop", [(128, True, 3), (64, False, 1), (256, True, 3)],
                         ids=["d128-causal-V1", "d64-full-V0", "d256-causal-V1"])
def test_forward_abort_path(d, causal, drop):
    """The fused kernel's own abort path, without a fault: in every block the
    producer leaves out the copy of one K/V ring position, so the MMA warp's
    bounded wait for it runs out (one role's wait records its code first);
    every role leaves its waits, lets its own copies and MMAs finish, tensor
    memory is freed and the kernel returns.  The status word reports it, the
    context stays usable and the next attn_fwd is correct."""
    B, H, N = 1, 2, 640
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=70 + d)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), device="cuda")
    ea.attn_fwd_device_status()  # start from a clean status word
    t0 = time.perf_counter()
    assert ea.attn_selftest_fwd_dropped_load(qd, kd, vd, o, lse, causal, drop,
                                             timeout_ms=50) == ea.ATTN_OK
    st, detail = ea.attn_fwd_device_status()
    elapsed = time.perf_counter() - t0
    assert st == ea.ATTN_ERR_TIMEOUT and detail in KERNEL_WAIT_CODES, (st, hex(detail))
    assert 0.04 <= elapsed < 5.0, elapsed
    assert ea.attn_fwd_device_status() == (ea.ATTN_OK, 0)

    o2, lse2 = ea.attn_fwd(qd, kd, vd, causal=causal)
    assert ea.attn_fwd_device_status() == (ea.ATTN_OK, 0)
    o_ref, lse_ref = oracle.Oracle().attn_bf16(q, k, v, causal, 1 / math.sqrt(d))
    m = metrics(o2.float().cpu().numpy(), o_ref, lse2.cpu().numpy(), lse_ref)
    assert within(m), describe(m)


def test_forward_abort_selftest_rejects_bad_arguments():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), device="cuda")
    assert ea.attn_selftest_fwd_dropped_load(q, q, q, o, lse, False, -1) == ea.ATTN_ERR_INVALID_ARG
    assert ea.attn_selftest_fwd_dropped_load(q, q, q, o, lse, False, 0,
                                             timeout_ms=0) == ea.ATTN_ERR_INVALID_ARG
