"""The fp64 oracle against its pins, and the pins against planted mistakes.

The oracle is test infrastructure (see oracle/__init__.py).  These tests run on
the CPU only.  The second half compiles deliberately broken copies of
oracle/attn_ref.c (one plausible mistake each) and requires that every copy
fails at least one pin, so the pins are known to catch that class of error.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle_pins import ALL_PINS, run_all

ORC = None


def _orc():
    global ORC
    if ORC is None:
        ORC = oracle.Oracle()
    return ORC


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    fails = pin(_orc())
    assert not fails, "\n".join(fails[:10])


def test_threads_reported():
    assert _orc().max_threads() >= 1


def test_rejects_bad_sizes():
    orc = _orc()
    z = np.zeros((1, 1, 1, 1))
    with pytest.raises(ValueError):
        orc.attn_f64(np.zeros((1, 1, 2)), z, z, False, 1.0)
    rc = orc.lib.attn_ref_f64(z.ctypes.data, z.ctypes.data, z.ctypes.data, z.ctypes.data,
                              z.ctypes.data, 1, 1, 0, 1, 1.0, 0, 0)
    assert rc != 0
    q = torch.zeros((1, 1, 4, 2), dtype=torch.bfloat16)
    with pytest.raises(RuntimeError):
        orc.attn_bf16_rows(q, q, q, False, 1.0, [4])  # row id out of range


# ------------------------------------------------------------ mutation tests
# (description, exact text in attn_ref.c, replacement)
MUTANTS = [
    ("causal mask excludes the diagonal",
     "int64_t last = causal ? i + off : Nk - 1;",
     "int64_t last = causal ? (i + off > 0 ? i + off - 1 : 0) : Nk - 1;"),
    ("causal mask off (always full row)",
     "int64_t last = causal ? i + off : Nk - 1;",
     "int64_t last = Nk - 1;"),
    ("causal diagonal top-left aligned when Nk > Nq",
     "int64_t last = causal ? i + off : Nk - 1;",
     "int64_t last = causal ? i : Nk - 1;"),
    ("key rows indexed with the query length",
     "decode_head(k + bh * (int64_t)kv_elems, Kh, (int64_t)kv_elems);\n        decode_head(v + bh * (int64_t)kv_elems, Vh, (int64_t)kv_elems);\n        rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, NULL, Nq,",
     "decode_head(k + bh * (int64_t)q_elems, Kh, (int64_t)kv_elems);\n        decode_head(v + bh * (int64_t)q_elems, Vh, (int64_t)kv_elems);\n        rc = head_rows(Qh, Kh, Vh, Nq, Nk, d, scale, causal, NULL, Nq,"),
    ("scale dropped", "s[j] = scale * acc;", "s[j] = acc;"),
    ("scale applied twice", "s[j] = scale * acc;", "s[j] = scale * scale * acc;"),
    ("lse without the max", "*lse_i = m + log(l);", "*lse_i = log(l);"),
    ("lse in base 2", "*lse_i = m + log(l);", "*lse_i = m + log2(l);"),
    ("keys read from V", "const double *k_j = K + j * d;", "const double *k_j = V + j * d;"),
    ("missing normalisation", "const double p = s[j] / l;", "const double p = s[j];"),
    ("values in reverse order", "const double *v_j = V + j * d;",
     "const double *v_j = V + (last - j) * d;"),
    ("exp sign flipped", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("max replaced by first score", "if (s[j] > m) m = s[j];", "if (j == 0) m = s[j];"),
    ("bf16 decode shift wrong", "((uint32_t)h) << 16;", "((uint32_t)h) << 15;"),
    ("e4m3 exponent bias 8", "x = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "x = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3 subnormals scaled like normals", "x = ldexp((double)m / 8.0, -6);",
     "x = ldexp((double)m / 8.0, -7);"),
    ("e4m3 descale dropped", "dst[t] = descale * e4m3_to_f64(src[t]);",
     "dst[t] = e4m3_to_f64(src[t]);"),
    ("e4m3 sign ignored", "return (c & 0x80) ? -x : x;", "return x;"),
    ("dot product drops last feature", "for (int64_t c = 0; c < d; ++c) acc += q_i[c] * k_j[c];",
     "for (int64_t c = 0; c + 1 < d; ++c) acc += q_i[c] * k_j[c];"),
    ("q row of the wrong query", "attend_row(Qh + i * d,", "attend_row(Qh + (i > 0 ? i - 1 : 0) * d,"),
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("desc,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(desc, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    with tempfile.TemporaryDirectory() as td:
        msrc = os.path.join(td, "mutant.c")
        open(msrc, "w").write(src.replace(old, new))
        lib = oracle.build(force=True, src=msrc, out=os.path.join(td, "libmutant.so"),
                           src_bwd=None)
        res = run_all(oracle.Oracle(oracle.load(lib)))
    failed = [k for k, v in res.items() if v]
    assert failed, f"no pin caught the planted mistake: {desc}"
