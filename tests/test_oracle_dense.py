"""Pins of the dense whole-tensor oracle (``oracle/dense.py``), CPU only.

The dense oracle writes the plain definition with library matrix products so
that full-size workloads can be checked element by element.  It is pinned
three ways:

* against the C oracle (``oracle/attn_ref.c``), an independent implementation
  of the same definition (per-row loops in C), on ragged shapes, Nq != Nk,
  both causal flags and row blocks smaller than the problem;
* by the C oracle's own pins (closed forms, invariants, torch SDPA, the
  blocked online softmax, hand-derived golden files), run through an adapter
  with the C oracle's method names;
* by planted mistakes in copies of its source, each of which must fail a pin.
"""
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle
import oracle_pins
from oracle import dense
from oracle_pins import ALL_PINS, pin_e4m3_decode
from test_oracle_bwd import check_bwd

# the e4m3 decoder pin compares a decoder with torch's conversion, which is
# what the dense oracle uses, so it says nothing about this implementation
DENSE_PINS = [p for p in ALL_PINS if p is not pin_e4m3_decode]


@pytest.fixture(autouse=True)
def _regroup_tolerance(monkeypatch):
    # matrix products of different shapes may round the last bits differently
    monkeypatch.setattr(oracle_pins, "SHAPE_REGROUP_ATOL", 1e-13)


class DenseAdapter:
    """The dense oracle behind the method names the pins call."""

    def __init__(self, mod=dense):
        self.m = mod

    def attn_f64(self, q, k, v, causal, scale, nthreads=0):
        return self.m.attn_f64(q, k, v, causal, scale)

    def attn_f64_qk(self, q, k, v, causal, scale, nthreads=0):
        return self.m.attn_f64_qk(q, k, v, causal, scale)

    def attn_bf16(self, q, k, v, causal, scale, nthreads=0):
        return self.m.attn_bf16(q, k, v, causal, scale)

    attn_bf16_qk = attn_bf16

    def attn_bf16_rows(self, q, k, v, causal, scale, rows, nthreads=0):
        o, lse = self.m.attn_bf16(q, k, v, causal, scale)
        return o.reshape(-1, o.shape[-1])[rows], lse.reshape(-1)[rows]

    attn_bf16_qk_rows = attn_bf16_rows

    def attn_e4m3(self, q, k, v, sq, sk, sv, causal, scale, rows=None, nthreads=0):
        o, lse = self.m.attn_e4m3(q, k, v, sq, sk, sv, causal, scale)
        if rows is None:
            return o, lse
        return o.reshape(-1, o.shape[-1])[rows], lse.reshape(-1)[rows]

    attn_e4m3_qk = attn_e4m3

    def attn_bwd_f64(self, q, k, v, dout, causal, scale, nthreads=0):
        return self.m.attn_bwd_f64(q, k, v, dout, causal, scale)


_C = None


def c_oracle():
    global _C
    if _C is None:
        _C = oracle.Oracle()
    return _C


@pytest.mark.parametrize("pin", DENSE_PINS, ids=lambda p: p.__name__)
def test_dense_pin(pin):
    fails = pin(DenseAdapter())
    assert not fails, "\n".join(fails[:10])


CASES = [(1, 2, 37, 37, 16), (2, 1, 5, 61, 8), (1, 3, 130, 130, 32), (1, 1, 1, 1, 4),
         (2, 2, 64, 200, 24)]


@pytest.mark.parametrize("block", [1024, 7])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,Nq,Nk,d", CASES, ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}d{c[4]}" for c in CASES])
def test_dense_matches_c_oracle(B, H, Nq, Nk, d, causal, block):
    g = torch.Generator().manual_seed(Nq * 31 + Nk + d)
    q = torch.randn((B, H, Nq, d), generator=g).mul(1.5).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g).mul(1.5).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = dense.attn_f64_qk(q, k, v, causal, scale, rows_per_block=block)
    o_c, lse_c = c_oracle().attn_bf16_qk(q, k, v, causal, scale)
    assert np.abs(o - o_c).max() <= 1e-12
    assert np.abs(lse - lse_c).max() <= 1e-12


@pytest.mark.parametrize("block", [1024, 5])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_dense_backward_matches_c_oracle(causal, block):
    g = torch.Generator().manual_seed(11)
    q, k, v, dout = (torch.randn((2, 2, 67, 16), generator=g).to(torch.bfloat16) for _ in range(4))
    got = dense.attn_bwd_f64(q, k, v, dout, causal, 0.3, rows_per_block=block)
    ref = c_oracle().attn_bwd_bf16(q, k, v, dout, causal, 0.3)
    for a, b in zip(got, ref):
        assert np.abs(a - b).max() <= 1e-12


def test_dense_backward_pins():
    fails = check_bwd(DenseAdapter())
    assert not fails, "\n".join(fails)


def test_dense_e4m3_matches_c_oracle():
    g = torch.Generator().manual_seed(3)
    shp = (1, 2, 70, 32)
    codes = []
    for _ in range(3):
        c = torch.randint(0, 256, shp, generator=g, dtype=torch.int64).to(torch.uint8)
        c[(c & 0x7F) == 0x7F] = 0x3A  # no NaN codes
        codes.append(c)
    sc = (0.5, 0.25, 2.0)
    for causal in (False, True):
        o, lse = dense.attn_e4m3(*codes, *sc, causal, 0.05)
        o_c, lse_c = c_oracle().attn_e4m3(*codes, *sc, causal, 0.05)
        assert np.abs(o - o_c).max() <= 1e-12
        assert np.abs(lse - lse_c).max() <= 1e-12


def test_dense_rejects_bad_shapes():
    z = torch.zeros((1, 1, 4, 2), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dense.attn_f64_qk(z, z[:, :, :2], z[:, :, :2], True, 1.0)  # causal needs Nk >= Nq
    with pytest.raises(ValueError):
        dense.attn_f64_qk(z, z, z[:, :, :3], False, 1.0)


# ------------------------------------------------------------ mutation tests
# (description, exact text in dense.py, replacement)
MUTANTS = [
    ("causal mask excludes the diagonal", "s.masked_fill_(j > i + off,", "s.masked_fill_(j >= i + off,"),
    ("causal diagonal top-left aligned", "s.masked_fill_(j > i + off,", "s.masked_fill_(j > i,"),
    ("scale dropped", "s = scale * (q[b, h, r0:r1] @ kk.T)", "s = (q[b, h, r0:r1] @ kk.T)"),
    ("lse without the max", "(m + torch.log(l)).squeeze(1)", "torch.log(l).squeeze(1)"),
    ("missing normalisation", "o[b, h, r0:r1] = (p @ vv) / l", "o[b, h, r0:r1] = (p @ vv)"),
    ("last visible key dropped", "kk, vv = k[b, h, :last + 1], v[b, h, :last + 1]",
     "kk, vv = k[b, h, :last], v[b, h, :last]"),
    ("exp sign flipped", "p = torch.exp(s - m)", "p = torch.exp(m - s)"),
    ("keys read from V", "kk, vv = k[b, h, :last + 1], v[b, h, :last + 1]",
     "kk, vv = v[b, h, :last + 1], v[b, h, :last + 1]"),
    ("e4m3 descale dropped", "return codes.to(torch.float64) * float(descale)",
     "return codes.to(torch.float64)"),
]

BWD_MUTANTS = [
    ("D term dropped", "ds = p * (dp - D)", "ds = p * dp"),
    ("dK without scale", "dk[b, h, :nvis] += scale * (ds.T @ qb)",
     "dk[b, h, :nvis] += (ds.T @ qb)"),
    ("dQ from V instead of K", "dq[b, h, r0:r1] = scale * (ds @ kk)",
     "dq[b, h, r0:r1] = scale * (ds @ vv)"),
    ("dV uses dS instead of P", "dv[b, h, :nvis] += p.T @ gb", "dv[b, h, :nvis] += ds.T @ gb"),
    ("last visible key dropped in backward", "nvis = r1 if causal else N", "nvis = r1 - 1 if causal else N - 1"),
    ("causal mask off in backward", "s.masked_fill_(j > i, -math.inf)", "pass"),
    ("dP from K instead of V", "dp = gb @ vv.T", "dp = gb @ kk.T"),
]


def _mutant_module(old, new):
    src = open(dense.__file__).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mod = types.ModuleType("dense_mutant")
    exec(compile(src.replace(old, new), os.path.join("mutant", "dense.py"), "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("desc,old,new", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_dense_backward_pins_catch_mutant(desc, old, new):
    fails = check_bwd(DenseAdapter(_mutant_module(old, new)))
    assert fails, f"no pin caught the planted mistake: {desc}"


@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_dense_pins_catch_mutant(desc, old, new):
    adapter = DenseAdapter(_mutant_module(old, new))
    res = {}
    for pin in DENSE_PINS:
        try:
            res[pin.__name__] = pin(adapter)
        except Exception as e:  # a broken oracle may raise
            res[pin.__name__] = [f"raised {type(e).__name__}: {e}"]
    assert any(res.values()), f"no pin caught the planted mistake: {desc}"
