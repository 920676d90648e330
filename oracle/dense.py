"""Exact softmax attention, forward, as dense fp64 tensor algebra: the
whole-tensor ORACLE for problems too large for the row-by-row C oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` may import this module; the product
path (``exact_attention_51_gb300``) never does, and the two share no code.

What it computes is the plain definition, the same one ``attn_ref.c`` loops
over, written with library primitives (torch CPU fp64 matrix products,
``exp``, ``log``, row max and row sum).  For one head, and query rows i taken
a block at a time:

    S_ij  = scale * q_i . k_j              (fp64 matrix product Q_rows K^T)
    S_ij  = -inf  for j > i + Nk - Nq      (causal: the "triangular matrix",
                                            bottom-right aligned when Nk > Nq)
    m_i   = max_j S_ij
    P_ij  = exp(S_ij - m_i),   l_i = sum_j P_ij
    o_i   = (sum_j P_ij v_j) / l_i         (fp64 matrix product P V)
    lse_i = m_i + ln l_i

Query rows are grouped only to bound memory: each row still sees all of its
visible keys in one pass, so nothing here is tiled over keys and no online
rescaling takes place -- the result is the three-pass definition that the
fused kernel's rescaling must reproduce ("Tri Dao: prediction": exact
attention, the softmax's sum across the whole row, "still get the right
answer"; HN item 40939030, FlashAttention-3 thread: the softmax of the
triangular matrix).  Keys past the last key any row of a block can see are
left out of that block's product; they would only add exp(-inf) = 0 terms.

Inputs are decoded by torch's own exact conversions: bf16 -> fp64, and e4m3
(``float8_e4m3fn``) -> fp64 times the tensor's dequantisation scale, the
conversion the C oracle's e4m3 decoder is pinned against code by code.

The gradients (``attn_bwd_f64``) are the textbook derivative of the same
definition, as ``attn_bwd_ref.c`` states them: with P the row-stochastic
attention matrix and dO the upstream gradient,

    dV = P^T dO,  dP = dO V^T,  D_i = dO_i . o_i,  dS = P o (dP - D),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Parity status: pinned -- ``tests/test_oracle_dense.py`` checks it against the
C oracles (an independent implementation: per-row loops in C against blocked
library matrix products) and runs the C oracles' pins (closed forms,
invariants, torch SDPA and its autograd, finite differences, the tiled online
softmax, hand-derived golden files) on it.
"""
from __future__ import annotations

import math

import numpy as np
import torch

ROWS_PER_BLOCK = 1024


def _f64(x) -> torch.Tensor:
    if isinstance(x, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    if x.device.type != "cpu":
        raise TypeError("oracle inputs live on the CPU")
    return x.to(torch.float64).contiguous()


def attn_f64_qk(q, k, v, causal: bool, scale: float, rows_per_block: int = ROWS_PER_BLOCK):
    """q [B,H,Nq,d], k and v [B,H,Nk,d] (fp64-convertible CPU arrays) ->
    (o fp64 [B,H,Nq,d], lse fp64 [B,H,Nq]) as numpy arrays.  Causal: key j is
    visible to query i iff j <= i + Nk - Nq (needs Nk >= Nq)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B,H,Nq,d] queries and [B,H,Nk,d] keys / values")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k, v must be [B,H,Nk,d] with q's B, H and d")
    if Nq < 1 or Nk < 1 or (causal and Nk < Nq):
        raise ValueError("need Nq, Nk >= 1 and, when causal, Nk >= Nq")
    off = Nk - Nq
    o = torch.empty((B, H, Nq, d), dtype=torch.float64)
    lse = torch.empty((B, H, Nq), dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, Nq, rows_per_block):
                r1 = min(Nq, r0 + rows_per_block)
                last = (r1 - 1 + off) if causal else Nk - 1  # last key any row here sees
                kk, vv = k[b, h, :last + 1], v[b, h, :last + 1]
                s = scale * (q[b, h, r0:r1] @ kk.T)
                if causal:
                    i = torch.arange(r0, r1).unsqueeze(1)
                    j = torch.arange(last + 1).unsqueeze(0)
                    s.masked_fill_(j > i + off, -math.inf)
                m = s.amax(dim=1, keepdim=True)
                p = torch.exp(s - m)
                l = p.sum(dim=1, keepdim=True)
                o[b, h, r0:r1] = (p @ vv) / l
                lse[b, h, r0:r1] = (m + torch.log(l)).squeeze(1)
    return o.numpy(), lse.numpy()


def attn_f64(q, k, v, causal: bool, scale: float):
    """Nq = Nk = N form of ``attn_f64_qk``."""
    return attn_f64_qk(q, k, v, causal, scale)


def attn_bf16(q, k, v, causal: bool, scale: float):
    """torch bf16 CPU tensors (q [B,H,Nq,d], k, v [B,H,Nk,d]) -> (o, lse) fp64."""
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
            raise TypeError("expected torch.bfloat16 CPU tensors")
    return attn_f64_qk(q, k, v, causal, scale)


def decode_e4m3(codes, descale: float) -> torch.Tensor:
    """e4m3 codes (uint8 or float8_e4m3fn CPU tensor) -> fp64 values times
    the per-tensor dequantisation scale."""
    if codes.dtype == torch.uint8:
        codes = codes.view(torch.float8_e4m3fn)
    if codes.dtype != torch.float8_e4m3fn:
        raise TypeError("expected uint8 or float8_e4m3fn codes")
    return codes.to(torch.float64) * float(descale)


def attn_e4m3(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float,
              causal: bool, scale: float):
    """e4m3 codes with one dequantisation scale per tensor -> (o, lse) fp64 of
    the attention of the dequantised tensors."""
    return attn_f64_qk(decode_e4m3(q8, descale_q), decode_e4m3(k8, descale_k),
                       decode_e4m3(v8, descale_v), causal, scale)


def attn_bwd_f64(q, k, v, dout, causal: bool, scale: float,
                 rows_per_block: int = ROWS_PER_BLOCK):
    """q, k, v, dO [B,H,N,d] (fp64-convertible CPU arrays; Nq = Nk = N, key
    j visible to query i iff j <= i when causal) -> (dq, dk, dv) fp64 numpy
    arrays.  Query rows go a block at a time; dK and dV add up every block's
    share (sums over i), dQ rows are each block's own."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    if q.dim() != 4 or not (q.shape == k.shape == v.shape == dout.shape):
        raise ValueError("q, k, v, dout must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    dq, dk, dv = (torch.zeros((B, H, N, d), dtype=torch.float64) for _ in range(3))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, N, rows_per_block):
                r1 = min(N, r0 + rows_per_block)
                nvis = r1 if causal else N  # keys [0, nvis) are visible to some row here
                kk, vv = k[b, h, :nvis], v[b, h, :nvis]
                qb, gb = q[b, h, r0:r1], dout[b, h, r0:r1]
                s = scale * (qb @ kk.T)
                if causal:
                    i = torch.arange(r0, r1).unsqueeze(1)
                    j = torch.arange(nvis).unsqueeze(0)
                    s.masked_fill_(j > i, -math.inf)
                p = torch.exp(s - s.amax(dim=1, keepdim=True))
                p = p / p.sum(dim=1, keepdim=True)
                o = p @ vv
                D = (gb * o).sum(dim=1, keepdim=True)
                dp = gb @ vv.T
                ds = p * (dp - D)
                dq[b, h, r0:r1] = scale * (ds @ kk)
                dk[b, h, :nvis] += scale * (ds.T @ qb)
                dv[b, h, :nvis] += p.T @ gb
    return dq.numpy(), dk.numpy(), dv.numpy()


def attn_bwd_bf16(q, k, v, dout, causal: bool, scale: float):
    """torch bf16 CPU tensors -> (dq, dk, dv) fp64."""
    for t in (q, k, v, dout):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
            raise TypeError("expected torch.bfloat16 CPU tensors")
    return attn_bwd_f64(q, k, v, dout, causal, scale)
