"""fp64 CPU oracle for exact softmax attention (forward).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference``) may import this
package.  The product path (``exact_attention_51_gb300``) never imports it and
shares no code with it; the two meet only through the seeded input generator
in ``exact_attention_51_gb300.workloads``, which holds none of the method's
arithmetic.

The arithmetic lives in ``attn_ref.c`` (plain three-pass definition, fp64,
OpenMP over rows).  This module builds it with gcc on first use and marshals
numpy / torch-CPU arrays through ctypes.

Sources: "Tri Dao: prediction" (podcast transcript: exact attention, the
softmax row dependency, the online-softmax trick reaching the same answer);
HN item 40939030, FlashAttention-3 thread (softmax of the triangular matrix).

Parity status: pinned -- see ``tests/test_oracle.py`` for the pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_SRC_BWD = os.path.join(_HERE, "attn_bwd_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH,
          src_bwd: str | None = _SRC_BWD) -> str:
    """Compile the forward source ``src`` (and the backward source
    ``src_bwd`` unless None) with gcc -O2 -fopenmp into ``out``.

    Plain portable C: no -march flags, so the same source builds on x86_64 and
    aarch64 hosts.  Returns the path of the library.
    """
    srcs = [src] + ([src_bwd] if src_bwd else [])
    if (not force and os.path.exists(out)
            and all(os.path.getmtime(out) >= os.path.getmtime(f) for f in srcs)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, *srcs, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.attn_ref_f64.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                 _dbl, ctypes.c_int, ctypes.c_int]
    lib.attn_ref_f64.restype = ctypes.c_int
    lib.attn_ref_bf16.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                  _dbl, ctypes.c_int, ctypes.c_int]
    lib.attn_ref_bf16.restype = ctypes.c_int
    lib.attn_ref_bf16_rows.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _dbl,
                                       ctypes.c_int, _vp, _i64, _vp, _vp, ctypes.c_int]
    lib.attn_ref_bf16_rows.restype = ctypes.c_int
    lib.attn_ref_f64_qk.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                    _dbl, ctypes.c_int, ctypes.c_int]
    lib.attn_ref_f64_qk.restype = ctypes.c_int
    lib.attn_ref_bf16_qk.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                     _dbl, ctypes.c_int, ctypes.c_int]
    lib.attn_ref_bf16_qk.restype = ctypes.c_int
    lib.attn_ref_bf16_qk_rows.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _dbl,
                                          ctypes.c_int, _vp, _i64, _vp, _vp, ctypes.c_int]
    lib.attn_ref_bf16_qk_rows.restype = ctypes.c_int
    if hasattr(lib, "attn_bwd_ref_f64"):
        lib.attn_bwd_ref_f64.argtypes = [_vp] * 7 + [_i64] * 4 + [_dbl, ctypes.c_int, ctypes.c_int]
        lib.attn_bwd_ref_f64.restype = ctypes.c_int
        lib.attn_bwd_ref_bf16.argtypes = [_vp] * 7 + [_i64] * 4 + [_dbl, ctypes.c_int, ctypes.c_int]
        lib.attn_bwd_ref_bf16.restype = ctypes.c_int
    lib.attn_ref_e4m3.argtypes = [_vp, _vp, _vp, _dbl, _dbl, _dbl, _i64, _i64, _i64, _i64,
                                  _dbl, ctypes.c_int, _vp, _i64, _vp, _vp, ctypes.c_int]
    lib.attn_ref_e4m3.restype = ctypes.c_int
    lib.attn_ref_e4m3_qk.argtypes = [_vp, _vp, _vp, _dbl, _dbl, _dbl, _i64, _i64, _i64, _i64,
                                     _i64, _dbl, ctypes.c_int, _vp, _i64, _vp, _vp, ctypes.c_int]
    lib.attn_ref_e4m3_qk.restype = ctypes.c_int
    lib.attn_ref_e4m3_decode.argtypes = [ctypes.c_int]
    lib.attn_ref_e4m3_decode.restype = _dbl
    lib.attn_ref_max_threads.argtypes = []
    lib.attn_ref_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another
    build of an oracle source (the mutation tests use this)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _as_bf16_bits(t) -> np.ndarray:
    """torch bf16 CPU tensor -> contiguous uint16 numpy view of its bits."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
        raise TypeError("expected a torch.bfloat16 CPU tensor")
    if t.device.type != "cpu":
        raise TypeError("oracle inputs live on the CPU")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _shape4(a):
    if a.ndim != 4:
        raise ValueError("expected [B,H,N,d]")
    return a.shape


class Oracle:
    """Callable wrapper around one build of the oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def max_threads(self) -> int:
        return int(self.lib.attn_ref_max_threads())

    def attn_f64(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        """fp64 inputs [B,H,N,d] (numpy) -> (o fp64 [B,H,N,d], lse fp64 [B,H,N])."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        B, H, N, d = _shape4(q)
        if k.shape != q.shape or v.shape != q.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        o = np.empty((B, H, N, d), np.float64)
        lse = np.empty((B, H, N), np.float64)
        rc = self.lib.attn_ref_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                   o.ctypes.data, lse.ctypes.data, B, H, N, d,
                                   float(scale), int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_f64 failed: {rc}")
        return o, lse

    def attn_bf16(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        """torch bf16 CPU [B,H,N,d] -> (o fp64, lse fp64), whole tensors."""
        qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        B, H, N, d = _shape4(qb)
        if kb.shape != qb.shape or vb.shape != qb.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        o = np.empty((B, H, N, d), np.float64)
        lse = np.empty((B, H, N), np.float64)
        rc = self.lib.attn_ref_bf16(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                    o.ctypes.data, lse.ctypes.data, B, H, N, d,
                                    float(scale), int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_bf16 failed: {rc}")
        return o, lse

    def attn_bf16_rows(self, q, k, v, causal: bool, scale: float, rows,
                       nthreads: int = 0):
        """Selected flat rows ((b*H+h)*N + i) -> (o fp64 [R,d], lse fp64 [R])."""
        qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        B, H, N, d = _shape4(qb)
        if kb.shape != qb.shape or vb.shape != qb.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
        o = np.empty((max(R, 1), d), np.float64)
        lse = np.empty((max(R, 1),), np.float64)
        rc = self.lib.attn_ref_bf16_rows(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                         B, H, N, d, float(scale), int(bool(causal)),
                                         rows.ctypes.data, R, o.ctypes.data,
                                         lse.ctypes.data, int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_bf16_rows failed: {rc}")
        return o[:R], lse[:R]


    # -- gradients (attn_bwd_ref.c): dQ, dK, dV for upstream gradient dO

    def attn_bwd_f64(self, q, k, v, dout, causal: bool, scale: float, nthreads: int = 0):
        """fp64 [B,H,N,d] inputs -> (dq, dk, dv) fp64 [B,H,N,d]."""
        q, k, v, dout = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, dout))
        B, H, N, d = _shape4(q)
        if k.shape != q.shape or v.shape != q.shape or dout.shape != q.shape:
            raise ValueError("q, k, v, dout must share one [B,H,N,d] shape")
        dq, dk, dv = (np.empty((B, H, N, d), np.float64) for _ in range(3))
        rc = self.lib.attn_bwd_ref_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                       dout.ctypes.data, dq.ctypes.data, dk.ctypes.data,
                                       dv.ctypes.data, B, H, N, d, float(scale),
                                       int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_bwd_ref_f64 failed: {rc}")
        return dq, dk, dv

    def attn_bwd_bf16(self, q, k, v, dout, causal: bool, scale: float, nthreads: int = 0):
        """torch bf16 CPU [B,H,N,d] inputs -> (dq, dk, dv) fp64."""
        qb, kb, vb, gb = (_as_bf16_bits(t) for t in (q, k, v, dout))
        B, H, N, d = _shape4(qb)
        if kb.shape != qb.shape or vb.shape != qb.shape or gb.shape != qb.shape:
            raise ValueError("q, k, v, dout must share one [B,H,N,d] shape")
        dq, dk, dv = (np.empty((B, H, N, d), np.float64) for _ in range(3))
        rc = self.lib.attn_bwd_ref_bf16(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                        gb.ctypes.data, dq.ctypes.data, dk.ctypes.data,
                                        dv.ctypes.data, B, H, N, d, float(scale),
                                        int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_bwd_ref_bf16 failed: {rc}")
        return dq, dk, dv

    # -- a key length of its own: q [B,H,Nq,d], k / v [B,H,Nk,d]; causal
    # -- means key j visible to query i iff j <= i + Nk - Nq (needs Nk >= Nq)

    def attn_f64_qk(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
        B, H, Nq, Nk, d = _qk_shapes(q, k, v)
        o = np.empty((B, H, Nq, d), np.float64)
        lse = np.empty((B, H, Nq), np.float64)
        rc = self.lib.attn_ref_f64_qk(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                                      lse.ctypes.data, B, H, Nq, Nk, d, float(scale),
                                      int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_f64_qk failed: {rc}")
        return o, lse

    def attn_bf16_qk(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        B, H, Nq, Nk, d = _qk_shapes(qb, kb, vb)
        o = np.empty((B, H, Nq, d), np.float64)
        lse = np.empty((B, H, Nq), np.float64)
        rc = self.lib.attn_ref_bf16_qk(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                       o.ctypes.data, lse.ctypes.data, B, H, Nq, Nk, d,
                                       float(scale), int(bool(causal)), int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_bf16_qk failed: {rc}")
        return o, lse

    def attn_bf16_qk_rows(self, q, k, v, causal: bool, scale: float, rows, nthreads: int = 0):
        qb, kb, vb = _as_bf16_bits(q), _as_bf16_bits(k), _as_bf16_bits(v)
        B, H, Nq, Nk, d = _qk_shapes(qb, kb, vb)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
        o = np.empty((max(R, 1), d), np.float64)
        lse = np.empty((max(R, 1),), np.float64)
        rc = self.lib.attn_ref_bf16_qk_rows(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, H,
                                            Nq, Nk, d, float(scale), int(bool(causal)),
                                            rows.ctypes.data, R, o.ctypes.data, lse.ctypes.data,
                                            int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_bf16_qk_rows failed: {rc}")
        return o[:R], lse[:R]


    # -- e4m3 inputs with per-tensor dequantisation scales (attn_ref_e4m3)

    def e4m3_decode(self, code: int) -> float:
        """Value of one OCP e4m3 code (0..255) by the format's definition."""
        return float(self.lib.attn_ref_e4m3_decode(int(code)))

    def attn_e4m3(self, q, k, v, descale_q: float, descale_k: float, descale_v: float,
                  causal: bool, scale: float, rows=None, nthreads: int = 0):
        """e4m3 codes (uint8 numpy or torch uint8 / float8_e4m3fn CPU) [B,H,N,d]
        -> (o fp64, lse fp64): whole tensors, or the listed flat rows
        ((b*H+h)*N + i) as (o [R,d], lse [R])."""
        qc, kc, vc = (_as_u8(t) for t in (q, k, v))
        B, H, N, d = _shape4(qc)
        if kc.shape != qc.shape or vc.shape != qc.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        if rows is None:
            o = np.empty((B, H, N, d), np.float64)
            lse = np.empty((B, H, N), np.float64)
            rp, R = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            R = rows.shape[0]
            o = np.empty((max(R, 1), d), np.float64)
            lse = np.empty((max(R, 1),), np.float64)
            rp = rows.ctypes.data
        rc = self.lib.attn_ref_e4m3(qc.ctypes.data, kc.ctypes.data, vc.ctypes.data,
                                    float(descale_q), float(descale_k), float(descale_v),
                                    B, H, N, d, float(scale), int(bool(causal)), rp, R,
                                    o.ctypes.data, lse.ctypes.data, int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_e4m3 failed: {rc}")
        return (o, lse) if rows is None else (o[:R], lse[:R])


    def attn_e4m3_qk(self, q, k, v, descale_q: float, descale_k: float, descale_v: float,
                     causal: bool, scale: float, rows=None, nthreads: int = 0):
        """e4m3 codes, q [B,H,Nq,d] and k, v [B,H,Nk,d] -> (o fp64, lse fp64),
        whole tensors or the listed flat rows ((b*H+h)*Nq + i)."""
        qc, kc, vc = (_as_u8(t) for t in (q, k, v))
        B, H, Nq, Nk, d = _qk_shapes(qc, kc, vc)
        if rows is None:
            o = np.empty((B, H, Nq, d), np.float64)
            lse = np.empty((B, H, Nq), np.float64)
            rp, R = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            R = rows.shape[0]
            o = np.empty((max(R, 1), d), np.float64)
            lse = np.empty((max(R, 1),), np.float64)
            rp = rows.ctypes.data
        rc = self.lib.attn_ref_e4m3_qk(qc.ctypes.data, kc.ctypes.data, vc.ctypes.data,
                                       float(descale_q), float(descale_k), float(descale_v),
                                       B, H, Nq, Nk, d, float(scale), int(bool(causal)), rp, R,
                                       o.ctypes.data, lse.ctypes.data, int(nthreads))
        if rc:
            raise RuntimeError(f"oracle attn_ref_e4m3_qk failed: {rc}")
        return (o, lse) if rows is None else (o[:R], lse[:R])


def _as_u8(t) -> np.ndarray:
    """e4m3 codes as a contiguous uint8 numpy array (torch CPU tensors of
    dtype uint8 or float8_e4m3fn are viewed, not converted)."""
    if isinstance(t, np.ndarray):
        if t.dtype != np.uint8:
            raise TypeError("expected uint8 e4m3 codes")
        return np.ascontiguousarray(t)
    import torch
    if t.device.type != "cpu":
        raise TypeError("oracle inputs live on the CPU")
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("expected uint8 or float8_e4m3fn codes")
    return t.contiguous().view(torch.uint8).numpy()


def _qk_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected [B,H,Nq,d] queries and [B,H,Nk,d] keys / values")
    B, H, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k, v must be [B,H,Nk,d] with q's B, H and d")
    return B, H, Nq, k.shape[2], d


def default() -> Oracle:
    return Oracle()
