"""The fp64 backward oracle (oracle/attn_bwd_ref.c) against things other than
itself: central finite differences of the forward oracle, torch autograd
through scaled_dot_product_attention in fp64, and closed-form column sums.
Planted mistakes in copies of its source are each caught."""
import math
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle

ORC = None


def orc():
    global ORC
    if ORC is None:
        ORC = oracle.Oracle()
    return ORC


def _rand(shape, seed, mag=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * mag


def finite_difference_grads(o, q, k, v, g, causal, scale, h=1e-6):
    """dL/dq, dL/dk, dL/dv of L = sum(O * g) by central differences of the
    forward oracle (fp64)."""
    out = []
    for which in range(3):
        x = [q.copy(), k.copy(), v.copy()]
        grad = np.zeros_like(x[which])
        for idx in np.ndindex(*x[which].shape):
            plus = [a.copy() for a in x]
            minus = [a.copy() for a in x]
            plus[which][idx] += h
            minus[which][idx] -= h
            lp = (o.attn_f64(*plus, causal, scale)[0] * g).sum()
            lm = (o.attn_f64(*minus, causal, scale)[0] * g).sum()
            grad[idx] = (lp - lm) / (2 * h)
        out.append(grad)
    return out


def check_bwd(o, tol_fd=1e-6):
    """Pins for an oracle build; returns a list of failures."""
    fails = []
    for causal in (False, True):
        shp = (1, 2, 5, 3)
        q, k, v, g = (_rand(shp, s) for s in (1, 2, 3, 4))
        dq, dk, dv = o.attn_bwd_f64(q, k, v, g, causal, 0.7)
        fd = finite_difference_grads(o, q, k, v, g, causal, 0.7)
        for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), fd):
            err = np.abs(a - b).max()
            if not err <= tol_fd:
                fails.append(f"finite differences {name} causal={causal}: {err:.2e}")
        # torch autograd through SDPA (fp64)
        shp = (2, 1, 17, 8)
        q, k, v, g = (_rand(shp, s) for s in (5, 6, 7, 8))
        tq, tk, tv = (torch.from_numpy(a).requires_grad_() for a in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                               scale=0.3)
        out.backward(torch.from_numpy(g))
        dq, dk, dv = o.attn_bwd_f64(q, k, v, g, causal, 0.3)
        for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), (tq.grad, tk.grad, tv.grad)):
            err = np.abs(a - b.numpy()).max()
            if not err <= 1e-10:
                fails.append(f"sdpa autograd {name} causal={causal}: {err:.2e}")
        # closed forms: rows of P sum to 1 -> sum_j dV_j = sum_i dO_i (non-causal
        # and causal alike); rows of dS sum to 0 -> sum_j dK_j = 0
        if not np.allclose(dv.sum(2), g.sum(2), atol=1e-12):
            fails.append(f"sum of dV rows != sum of dO rows causal={causal}")
        if not np.allclose(dk.sum(2), 0.0, atol=1e-12):
            fails.append(f"sum of dK rows != 0 causal={causal}")
    # identical keys: uniform P, dS rows sum to 0 -> dQ = scale * dS K = 0
    q, v, g = (_rand((1, 1, 9, 4), s) for s in (9, 10, 11))
    k = np.broadcast_to(_rand((1, 1, 1, 4), 12), (1, 1, 9, 4)).copy()
    dq, _, _ = o.attn_bwd_f64(q, k, v, g, False, 1.0)
    if not np.abs(dq).max() <= 1e-12:
        fails.append("identical keys give dQ != 0")
    return fails


def test_backward_oracle_pins():
    fails = check_bwd(orc())
    assert not fails, "\n".join(fails)


def test_bf16_entry_point_matches_f64():
    g = torch.Generator().manual_seed(3)
    q, k, v, d = (torch.randn((1, 2, 33, 16), generator=g).to(torch.bfloat16) for _ in range(4))
    for causal in (False, True):
        a = orc().attn_bwd_bf16(q, k, v, d, causal, 0.25)
        b = orc().attn_bwd_f64(*(t.double().numpy() for t in (q, k, v, d)), causal, 0.25)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


BWD_MUTANTS = [
    ("D term dropped", "for (int64_t j = 0; j <= last; ++j) ds[j] = p[j] * (ds[j] - Di);",
     "for (int64_t j = 0; j <= last; ++j) ds[j] = p[j] * ds[j];"),
    ("dK without scale", "dK[j * d + c] = scale * ak;", "dK[j * d + c] = ak;"),
    ("dQ from V instead of K", "acc += dS[i * N + j] * K[j * d + c];",
     "acc += dS[i * N + j] * V[j * d + c];"),
    ("dK uses dS instead of its transpose", "ak += dS[i * N + j] * Q[i * d + c];",
     "ak += dS[j * N + i] * Q[i * d + c];"),
    ("dV uses dS instead of P", "av += P[i * N + j] * dO[i * d + c];",
     "av += dS[i * N + j] * dO[i * d + c];"),
    ("causal mask off in backward", "const int64_t last = causal ? i : N - 1;",
     "const int64_t last = N - 1;"),
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("desc,old,new", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_backward_pins_catch_mutant(desc, old, new):
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "attn_bwd_ref.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    with tempfile.TemporaryDirectory() as td:
        msrc = os.path.join(td, "mutant_bwd.c")
        open(msrc, "w").write(src.replace(old, new))
        lib = oracle.build(force=True, src=os.path.join(here, "attn_ref.c"),
                           out=os.path.join(td, "libmutant.so"), src_bwd=msrc)
        fails = check_bwd(oracle.Oracle(oracle.load(lib)))
    assert fails, f"no pin caught the planted mistake: {desc}"
