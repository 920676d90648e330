"""Host-side pieces of bench.py that need no GPU: the per-row FLOP count the
CPU baseline is scaled by, and the two oracle timings it reports (a bounded
row sample, and the whole tiny workload on one thread)."""
import math

import bench
from exact_attention_51_gb300 import workloads as wl


def test_row_flops_closed_forms():
    w = wl.WORKLOADS["tiny"]
    rows = list(range(w.B * w.H * w.N))
    # non-causal: every row sees N keys, 4*d FLOPs per key = the workload's count
    assert bench.row_flops(w, False, rows) == w.flops(False)
    # causal: row i of a head sees i + 1 keys, sum = N(N+1)/2 per head, so the
    # rows' count exceeds the halved convention by the diagonal's N keys
    per_head = 4.0 * w.d * w.N * (w.N + 1) / 2
    assert bench.row_flops(w, True, rows) == w.B * w.H * per_head
    assert bench.row_flops(w, True, rows) - w.flops(True) == 2.0 * w.d * w.N * w.B * w.H


def test_oracle_row_sample_timing():
    w = wl.WORKLOADS["tiny"]
    q, k, v = wl.workload_inputs(w)
    tf, secs, nrows, threads = bench.time_oracle(w, True, q, k, v, 0.05, 7)
    assert 0 < nrows <= w.B * w.H * w.N
    assert secs > 0 and threads >= 1
    assert math.isfinite(tf) and tf > 0


def test_oracle_tiny_one_thread_timing():
    us, tf = bench.time_oracle_tiny_one_thread(reps=3)
    assert math.isfinite(us) and us > 0
    # the value is the workload's non-causal FLOPs over the median time
    w = wl.WORKLOADS["tiny"]
    assert abs(tf - w.flops(False) / (us * 1e-6) / 1e12) <= 1e-9 * tf
