"""attn_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, a
serving loop that keeps cudaMalloc off its hot path).  Its workspace is the
library's own fixed device array.

The entry point is called through the C ABI (ctypes, raw device pointers)
twice in a row -- the second call finds the first call's leftovers in the
shared array -- and each result is checked against attn_fwd_splitkv with a
workspace this test allocates, within the parity tolerance of the suite.
This file is collected last, so a run that stops at the first failure has
run every other test already; it passes on its own in a fresh process too.
"""
import ctypes

import pytest
import torch

import exact_attention_51_gb300 as ea
from exact_attention_51_gb300 import workloads as wl
from oracle import dense
from parity import describe, metrics, within

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, lse, causal, splits):
    B, H, N, d = q.shape
    return lib.attn_fwd_splitkv_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, H, N, d,
        ctypes.c_float(d ** -0.5), int(causal), splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_splitkv_on_two_calls_in_a_row():
    lib = ea.load_library()
    calls = [((1, 4, 3000, 128), True, 4), ((2, 2, 1500, 64), False, 3)]
    for (B, H, N, d), causal, splits in calls:
        need = ea.attn_fwd_splitkv_workspace_size(B, H, N, d, splits)
        assert 0 < need <= ea.NOALLOC_WORKSPACE_BYTES
        q, k, v = (t.cuda() for t in wl.make_inputs(B, H, N, d, "normal", seed=N + splits))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), device="cuda")
        assert _noalloc(lib, q, k, v, o, lse, causal, splits) == ea.ATTN_OK
        o_ref, lse_ref = ea.attn_fwd_splitkv(q, k, v, causal=causal, num_splits=splits)
        torch.cuda.synchronize()
        st, detail = ea.attn_fwd_device_status()
        assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
        m = metrics(o.float().cpu().numpy(), o_ref.float().cpu().numpy(), lse.cpu().numpy(),
                    lse_ref.cpu().numpy())
        assert within(m), describe(m)


def test_noalloc_rejects_a_problem_beyond_its_workspace():
    lib = ea.load_library()
    B, H, N, d, splits = 1, 64, 8192, 128, 4  # 4 * 524288 rows * 129 * 4 B > 64 MiB
    assert ea.attn_fwd_splitkv_workspace_size(B, H, N, d, splits) > ea.NOALLOC_WORKSPACE_BYTES
    x = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(x)
    lse = torch.empty((B, H, N), device="cuda")
    assert _noalloc(lib, x, x, x, o, lse, False, splits) == ea.ATTN_ERR_NOALLOC_TOO_LARGE
    assert "no-allocation" in ea.attn_status_string(ea.ATTN_ERR_NOALLOC_TOO_LARGE)


def test_noalloc_against_the_oracle():
    """One call checked directly against the fp64 oracle, so the entry point
    does not rest on attn_fwd_splitkv alone."""
    lib = ea.load_library()
    B, H, N, d, causal, splits = 1, 3, 2500, 128, True, 3
    q, k, v = wl.make_inputs(B, H, N, d, "normal", seed=404)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), device="cuda")
    assert _noalloc(lib, qd, kd, vd, o, lse, causal, splits) == ea.ATTN_OK
    st, detail = ea.attn_fwd_device_status()
    assert st == ea.ATTN_OK, f"device-side wait timed out (code {detail:#x})"
    o_ref, lse_ref = dense.attn_bf16(q, k, v, causal, d ** -0.5)
    m = metrics(o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref)
    assert within(m), describe(m)


def test_noalloc_one_split_is_attn_fwd():
    """num_splits = 1 needs no workspace: the call is attn_fwd itself, so the
    bytes match."""
    lib = ea.load_library()
    q, k, v = (t.cuda() for t in wl.make_inputs(2, 2, 700, 64, "normal", seed=5))
    o = torch.empty_like(q)
    lse = torch.empty((2, 2, 700), device="cuda")
    assert _noalloc(lib, q, k, v, o, lse, True, 1) == ea.ATTN_OK
    o_ref, lse_ref = ea.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("splits", [0, -1, 65])
def test_noalloc_rejects_split_counts_out_of_range(splits):
    lib = ea.load_library()
    q, k, v = (t.cuda() for t in wl.make_inputs(1, 2, 300, 128, "normal", seed=6))
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 2, 300), 7.0, device="cuda")
    assert _noalloc(lib, q, k, v, o, lse, False, splits) == ea.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all()), "output written on a rejected call"
