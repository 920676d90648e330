"""Pins for the fp64 oracle: checks against things other than the oracle.

Each pin takes an ``oracle.Oracle`` and returns a list of failure strings
(empty = pass), so the same suite runs against the real oracle and against
deliberately broken copies of it (mutation tests).

What pins what:

* ``pin_online_softmax_tiling`` -- an independent fp64 numpy implementation of
  the blocked online softmax (running max and sum, rescaling of the partial
  output at every block: the trick the "Tri Dao: prediction" transcript
  describes) must equal the oracle's plain three-pass definition for every
  block size 1..N, ragged last blocks included.
* ``pin_merge_law`` -- the per-block states (m, l, acc) merge associatively
  (the "algebraic aggregates" view in HN item 40939030) and the merged state
  reproduces the oracle.
* ``pin_identity_values`` -- V = I makes O the probability matrix: rows are
  non-negative and sum to 1, and p_ij / p_ik = exp(s_ij - s_ik).
* ``pin_constant_values``, ``pin_single_key``, ``pin_uniform_queries``,
  ``pin_zero_scale`` -- closed forms.
* ``pin_permutation`` (non-causal set semantics), ``pin_causal_future_blind``
  (the triangular mask), ``pin_key_shift`` (softmax shift invariance and the
  lse offset it produces), ``pin_linearity_in_v`` -- invariants.
* ``pin_library_sdpa`` -- torch's scaled_dot_product_attention (CPU, fp64)
  and scipy's logsumexp on tiny shapes.
* ``pin_golden`` -- hand-derived fixtures under tests/golden/.
* ``pin_bf16_decode`` / ``pin_rows_api`` -- the bf16 entry points agree with
  the fp64 one on torch-decoded inputs, and the row-sampling entry point
  agrees with the whole-tensor one.
"""
from __future__ import annotations

import glob
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Comparisons of two calls that compute every row with the same fp64
# operations are exact for the C oracle.  An implementation built on library
# matrix products groups its sums by the problem's shape, so where the two
# calls differ in shape it may differ in the last bits: such a caller raises
# this (the dense oracle's tests use 1e-13).
SHAPE_REGROUP_ATOL = 0.0


def _rng(seed):
    return np.random.default_rng(seed)


def _close(name, got, want, atol, rtol=0.0):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if got.shape != want.shape:
        return [f"{name}: shape {got.shape} != {want.shape}"]
    if not np.all(np.isfinite(got)):
        return [f"{name}: non-finite output"]
    err = np.abs(got - want)
    tol = atol + rtol * np.abs(want)
    if np.any(err > tol):
        i = int(np.argmax(err - tol))
        return [f"{name}: max err {err.max():.3e} (at flat {i}: got {got.ravel()[i]!r} "
                f"want {want.ravel()[i]!r})"]
    return []


def _scores(q, k, scale, causal):
    """scale * q k^T with -inf above the diagonal when causal (numpy matmul)."""
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    if causal:
        N = q.shape[2]
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    return s


def tiled_online_softmax(q, k, v, scale, causal, block):
    """Blocked online-softmax attention, fp64, written from the description of
    the trick: visit key blocks in order, keep per row the running max m, the
    running sum l of exp(s - m) and the unnormalised output acc; when the max
    grows, rescale l and acc by exp(m_old - m_new)."""
    B, H, N, d = q.shape
    m = np.full((B, H, N), -np.inf)
    l = np.zeros((B, H, N))
    acc = np.zeros((B, H, N, d))
    rows = np.arange(N)[:, None]
    for j0 in range(0, N, block):
        j1 = min(N, j0 + block)
        s = scale * np.einsum("bhic,bhjc->bhij", q, k[:, :, j0:j1])
        if causal:
            keys = np.arange(j0, j1)[None, :]
            s = np.where(keys <= rows, s, -np.inf)
        m_blk = s.max(axis=-1)
        m_new = np.maximum(m, m_blk)
        # rows that have seen no visible key yet keep m = -inf; their alpha is 0
        with np.errstate(invalid="ignore"):
            alpha = np.where(np.isneginf(m_new), 0.0, np.exp(m - m_new))
            p = np.where(np.isneginf(s), 0.0, np.exp(s - m_new[..., None]))
        l = alpha * l + p.sum(-1)
        acc = alpha[..., None] * acc + np.einsum("bhij,bhjc->bhic", p, v[:, :, j0:j1])
        m = m_new
    return acc / l[..., None], m + np.log(l)


def _state(q, k, v, scale, causal, j0, j1):
    """(m, l, acc) of key block [j0, j1) for every row."""
    N = q.shape[2]
    s = scale * np.einsum("bhic,bhjc->bhij", q, k[:, :, j0:j1])
    if causal:
        s = np.where(np.arange(j0, j1)[None, :] <= np.arange(N)[:, None], s, -np.inf)
    m = s.max(-1)
    with np.errstate(invalid="ignore"):
        p = np.where(np.isneginf(s), 0.0, np.exp(s - m[..., None]))
    return m, p.sum(-1), np.einsum("bhij,bhjc->bhic", p, v[:, :, j0:j1])


def _merge(a, b):
    (m1, l1, o1), (m2, l2, o2) = a, b
    m = np.maximum(m1, m2)
    with np.errstate(invalid="ignore"):
        e1 = np.where(np.isneginf(m1), 0.0, np.exp(m1 - m))
        e2 = np.where(np.isneginf(m2), 0.0, np.exp(m2 - m))
    return m, l1 * e1 + l2 * e2, o1 * e1[..., None] + o2 * e2[..., None]


# --------------------------------------------------------------------- pins

def pin_online_softmax_tiling(orc):
    fails = []
    for (B, H, N, d, causal, seed) in [(1, 2, 13, 5, False, 1), (1, 2, 13, 5, True, 2),
                                       (2, 1, 9, 3, True, 3), (1, 1, 16, 8, False, 4)]:
        r = _rng(seed)
        q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
        scale = 0.7
        o, lse = orc.attn_f64(q, k, v, causal, scale)
        for block in range(1, N + 1):
            ot, lt = tiled_online_softmax(q, k, v, scale, causal, block)
            fails += _close(f"tiled o (N={N}, block={block}, causal={causal})", o, ot, 1e-12, 1e-12)
            fails += _close(f"tiled lse (N={N}, block={block}, causal={causal})", lse, lt, 1e-12, 1e-12)
    return fails


def pin_merge_law(orc):
    fails = []
    r = _rng(11)
    B, H, N, d = 1, 2, 12, 4
    q, k, v = (r.standard_normal((B, H, N, d)) * 2 for _ in range(3))
    for causal in (False, True):
        o, lse = orc.attn_f64(q, k, v, causal, 0.9)
        a = _state(q, k, v, 0.9, causal, 0, 5)
        b = _state(q, k, v, 0.9, causal, 5, 9)
        c = _state(q, k, v, 0.9, causal, 9, 12)
        for name, st in (("(ab)c", _merge(_merge(a, b), c)), ("a(bc)", _merge(a, _merge(b, c))),
                         ("(ca)b", _merge(_merge(c, a), b))):
            m, l, acc = st
            fails += _close(f"merge {name} o causal={causal}", acc / l[..., None], o, 1e-12, 1e-12)
            fails += _close(f"merge {name} lse causal={causal}", m + np.log(l), lse, 1e-12, 1e-12)
    return fails


def pin_identity_values(orc):
    fails = []
    r = _rng(21)
    N = 24
    q = r.standard_normal((1, 1, N, 6))
    k = r.standard_normal((1, 1, N, 6))
    # pad the feature dim of q, k up to N so V = I fits the shared [B,H,N,d] shape
    qd = np.zeros((1, 1, N, N)); qd[..., :6] = q
    kd = np.zeros((1, 1, N, N)); kd[..., :6] = k
    v = np.eye(N)[None, None]
    for causal in (False, True):
        P, lse = orc.attn_f64(qd, kd, v, causal, 0.8)
        fails += _close(f"rows of P sum to 1 (causal={causal})", P.sum(-1), np.ones((1, 1, N)), 1e-13)
        if np.any(P < 0):
            fails.append("negative probability")
        s = _scores(q, k, 0.8, causal)[0, 0]
        for i in range(N):
            vis = np.where(np.isfinite(s[i]))[0]
            ratio = P[0, 0, i, vis] / P[0, 0, i, vis[0]]
            fails += _close(f"p ratio row {i} causal={causal}", ratio, np.exp(s[i, vis] - s[i, vis[0]]), 1e-12, 1e-12)
            if causal and np.any(P[0, 0, i, i + 1:] != 0):
                fails.append(f"causal row {i} puts weight on a future key")
    return fails


def pin_constant_values(orc):
    fails = []
    r = _rng(31)
    q, k = r.standard_normal((2, 1, 17, 8)), r.standard_normal((2, 1, 17, 8))
    v = np.full((2, 1, 17, 8), -3.25)
    for causal in (False, True):
        o, _ = orc.attn_f64(q, k, v, causal, 1.3)
        fails += _close(f"constant V -> constant O causal={causal}", o, v, 1e-14)
    return fails


def pin_single_key(orc):
    r = _rng(41)
    q, k, v = (r.standard_normal((2, 3, 1, 5)) for _ in range(3))
    fails = []
    for causal in (False, True):
        o, lse = orc.attn_f64(q, k, v, causal, 0.37)
        fails += _close(f"N=1 O=V causal={causal}", o, v, 1e-15)
        fails += _close(f"N=1 lse causal={causal}", lse, 0.37 * (q * k).sum(-1), 1e-14)
    return fails


def pin_uniform_queries(orc):
    r = _rng(51)
    N = 19
    q = np.zeros((1, 2, N, 4))
    k, v = r.standard_normal((1, 2, N, 4)), r.standard_normal((1, 2, N, 4))
    fails = []
    o, lse = orc.attn_f64(q, k, v, False, 1.0)
    fails += _close("Q=0 O=mean(V)", o, np.broadcast_to(v.mean(2, keepdims=True), o.shape), 1e-14)
    fails += _close("Q=0 lse=ln N", lse, np.full(lse.shape, math.log(N)), 1e-14)
    o, lse = orc.attn_f64(q, k, v, True, 1.0)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    fails += _close("Q=0 causal O=prefix mean", o, prefix, 1e-14)
    fails += _close("Q=0 causal lse=ln(i+1)", lse,
                    np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape), 1e-14)
    fails += _close("causal row 0 O=V0", o[:, :, 0], v[:, :, 0], 1e-15)
    return fails


def pin_zero_scale(orc):
    r = _rng(61)
    q, k, v = (r.standard_normal((1, 1, 11, 3)) * 5 for _ in range(3))
    o, lse = orc.attn_f64(q, k, v, False, 0.0)
    return (_close("scale=0 O=mean V", o, np.broadcast_to(v.mean(2, keepdims=True), o.shape), 1e-14)
            + _close("scale=0 lse=ln N", lse, np.full(lse.shape, math.log(11)), 1e-14))


def pin_permutation(orc):
    r = _rng(71)
    q, k, v = (r.standard_normal((1, 2, 23, 6)) for _ in range(3))
    perm = r.permutation(23)
    o, lse = orc.attn_f64(q, k, v, False, 0.6)
    o2, lse2 = orc.attn_f64(q, k[:, :, perm], v[:, :, perm], False, 0.6)
    return _close("perm O", o2, o, 1e-13) + _close("perm lse", lse2, lse, 1e-13)


def pin_causal_future_blind(orc):
    r = _rng(81)
    N, t = 21, 9
    q, k, v = (r.standard_normal((1, 1, N, 4)) for _ in range(3))
    o, lse = orc.attn_f64(q, k, v, True, 1.1)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:] = r.standard_normal(k2[:, :, t + 1:].shape) * 50
    v2[:, :, t + 1:] = 1e6
    o2, lse2 = orc.attn_f64(q, k2, v2, True, 1.1)
    fails = _close("causal rows <= t unchanged", o2[:, :, :t + 1], o[:, :, :t + 1], 1e-15)
    fails += _close("causal lse <= t unchanged", lse2[:, :, :t + 1], lse[:, :, :t + 1], 1e-15)
    if np.allclose(o2[:, :, t + 1:], o[:, :, t + 1:]):
        fails.append("rows after t ignore keys they can see")
    return fails


def pin_key_shift(orc):
    r = _rng(91)
    q, k, v = (r.standard_normal((1, 2, 15, 5)) for _ in range(3))
    u = r.standard_normal(5)
    fails = []
    for causal in (False, True):
        o, lse = orc.attn_f64(q, k, v, causal, 0.45)
        o2, lse2 = orc.attn_f64(q, k + u, v, causal, 0.45)
        fails += _close(f"key shift O causal={causal}", o2, o, 1e-12)
        fails += _close(f"key shift lse causal={causal}", lse2, lse + 0.45 * (q @ u), 1e-12)
    return fails


def pin_linearity_in_v(orc):
    r = _rng(101)
    q, k, v1, v2 = (r.standard_normal((1, 1, 14, 4)) for _ in range(4))
    fails = []
    for causal in (False, True):
        a, _ = orc.attn_f64(q, k, v1, causal, 0.5)
        b, _ = orc.attn_f64(q, k, v2, causal, 0.5)
        c, _ = orc.attn_f64(q, k, v1 - 2.5 * v2, causal, 0.5)
        fails += _close(f"linear in V causal={causal}", c, a - 2.5 * b, 1e-13)
    return fails


def pin_library_sdpa(orc):
    from scipy.special import logsumexp
    fails = []
    for (B, H, N, d, seed, mag) in [(1, 2, 10, 4, 1, 1.0), (2, 1, 33, 16, 2, 1.0),
                                    (1, 1, 20, 8, 3, 30.0)]:
        r = _rng(200 + seed)
        q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
        k = k * mag  # large scores: the max subtraction must keep exp in range
        for causal in (False, True):
            scale = 1.0 / math.sqrt(d)
            o, lse = orc.attn_f64(q, k, v, causal, scale)
            ot = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
                is_causal=causal, scale=scale).numpy()
            fails += _close(f"sdpa O N={N} mag={mag} causal={causal}", o, ot, 1e-10)
            lt = logsumexp(_scores(q, k, scale, causal), axis=-1)
            fails += _close(f"logsumexp N={N} mag={mag} causal={causal}", lse, lt, 1e-10, 1e-12)
    return fails


def pin_golden(orc):
    fails = []
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    if not files:
        return ["no golden fixtures found"]
    for path in files:
        g = json.load(open(path))
        shp = (g["B"], g["H"], g["N"], g["d"])
        q, k, v = (np.array(g[x], np.float64).reshape(shp) for x in ("q", "k", "v"))
        for key, causal in (("noncausal", False), ("causal", True)):
            o, lse = orc.attn_f64(q, k, v, causal, g["scale"])
            name = os.path.basename(path)
            tol = g.get("tol", 1e-14)
            fails += _close(f"{name} {key} o", o, np.array(g[key]["o"]).reshape(o.shape), tol)
            fails += _close(f"{name} {key} lse", lse, np.array(g[key]["lse"]).reshape(lse.shape), tol)
    return fails


def pin_bf16_decode(orc):
    g = torch.Generator().manual_seed(5)
    shp = (1, 2, 37, 8)
    q, k, v = (torch.randn(shp, generator=g).mul(3).to(torch.bfloat16) for _ in range(3))
    # include bf16 extremes and signed zero
    q.view(-1)[0] = -0.0
    k.view(-1)[1] = torch.tensor(2.0 ** -126, dtype=torch.bfloat16)
    v.view(-1)[2] = torch.tensor(-3.3895e38, dtype=torch.bfloat16)
    v.view(-1)[3] = torch.tensor(2.0 ** -130, dtype=torch.bfloat16)  # subnormal
    fails = []
    for causal in (False, True):
        o, lse = orc.attn_bf16(q, k, v, causal, 0.25)
        o2, lse2 = orc.attn_f64(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                causal, 0.25)
        fails += _close(f"bf16 decode o causal={causal}", o, o2, 0.0)
        fails += _close(f"bf16 decode lse causal={causal}", lse, lse2, 0.0)
    return fails


def pin_rows_api(orc):
    g = torch.Generator().manual_seed(6)
    shp = (2, 3, 29, 8)
    q, k, v = (torch.randn(shp, generator=g).to(torch.bfloat16) for _ in range(3))
    rows = [0, 5, 28, 29, 57, 100, 173, 2 * 3 * 29 - 1, 44]
    fails = []
    for causal in (False, True):
        o, lse = orc.attn_bf16(q, k, v, causal, 0.3)
        orow, lrow = orc.attn_bf16_rows(q, k, v, causal, 0.3, rows)
        fails += _close(f"rows api o causal={causal}", orow, o.reshape(-1, 8)[rows], 0.0)
        fails += _close(f"rows api lse causal={causal}", lrow, lse.reshape(-1)[rows], 0.0)
    return fails


def pin_bottom_right_suffix(orc):
    """Causal with Nk > Nq keeps the diagonal at the bottom-right corner: the
    Nq queries are the last Nq of a causal sequence of length Nk, so their
    result equals the last Nq rows of the square causal attention."""
    r = _rng(131)
    fails = []
    for (Nq, Nk) in [(1, 9), (5, 17), (16, 16), (7, 64)]:
        qf, k, v = (r.standard_normal((1, 2, Nk, 6)) for _ in range(3))
        o_full, lse_full = orc.attn_f64(qf, k, v, True, 0.8)
        o, lse = orc.attn_f64_qk(qf[:, :, Nk - Nq:], k, v, True, 0.8)
        fails += _close(f"bottom-right O Nq={Nq} Nk={Nk}", o, o_full[:, :, Nk - Nq:],
                        SHAPE_REGROUP_ATOL)
        fails += _close(f"bottom-right lse Nq={Nq} Nk={Nk}", lse, lse_full[:, :, Nk - Nq:],
                        SHAPE_REGROUP_ATOL)
    return fails


def pin_rectangular_sdpa(orc):
    """Non-causal Nq != Nk against torch SDPA (fp64) and scipy logsumexp."""
    from scipy.special import logsumexp
    r = _rng(141)
    fails = []
    for (Nq, Nk) in [(3, 40), (40, 3), (1, 1), (33, 17)]:
        q = r.standard_normal((2, 1, Nq, 8))
        k, v = (r.standard_normal((2, 1, Nk, 8)) for _ in range(2))
        o, lse = orc.attn_f64_qk(q, k, v, False, 0.35)
        ot = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=0.35).numpy()
        fails += _close(f"rect sdpa Nq={Nq} Nk={Nk}", o, ot, 1e-12)
        lt = logsumexp(0.35 * np.einsum("bhic,bhjc->bhij", q, k), axis=-1)
        fails += _close(f"rect logsumexp Nq={Nq} Nk={Nk}", lse, lt, 1e-12, 1e-12)
    return fails


def pin_rectangular_bf16_rows(orc):
    g = torch.Generator().manual_seed(7)
    q = torch.randn((2, 2, 13, 8), generator=g).to(torch.bfloat16)
    k, v = (torch.randn((2, 2, 29, 8), generator=g).to(torch.bfloat16) for _ in range(2))
    fails = []
    for causal in (False, True):
        o, lse = orc.attn_bf16_qk(q, k, v, causal, 0.3)
        o2, lse2 = orc.attn_f64_qk(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                   causal, 0.3)
        fails += _close(f"rect bf16 decode causal={causal}", o, o2, 0.0)
        rows = [0, 12, 13, 25, 51, 38]
        orow, lrow = orc.attn_bf16_qk_rows(q, k, v, causal, 0.3, rows)
        fails += _close(f"rect rows o causal={causal}", orow, o.reshape(-1, 8)[rows], 0.0)
        fails += _close(f"rect rows lse causal={causal}", lrow, lse.reshape(-1)[rows], 0.0)
    return fails


def pin_e4m3_decode(orc):
    """The e4m3 decoder against torch's float8_e4m3fn conversion (all 256
    codes) and values the OCP 8-bit format fixes: 0x38 = 1, 0x7e = 448 (the
    largest finite), 0x01 = 2^-9 (the smallest subnormal), 0x08 = 2^-6 (the
    smallest normal), 0x80 = -0, 0x7f / 0xff = NaN."""
    fails = []
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    nan_ok = np.isnan(ref) == np.isnan(got)
    if not nan_ok.all() or not np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)]):
        bad = [c for c in range(256) if not (ref[c] == got[c] or (np.isnan(ref[c]) and np.isnan(got[c])))]
        fails.append(f"e4m3 decode differs from torch at codes {bad[:8]}")
    facts = {0x38: 1.0, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9,
             0xB8: -1.0, 0x40: 2.0, 0x3C: 1.5}
    for c, want in facts.items():
        if orc.e4m3_decode(c) != want:
            fails.append(f"e4m3 code {c:#04x} -> {orc.e4m3_decode(c)} (want {want})")
    if not (orc.e4m3_decode(0x80) == 0.0 and np.signbit(orc.e4m3_decode(0x80))):
        fails.append("e4m3 0x80 is not -0")
    if not (np.isnan(orc.e4m3_decode(0x7F)) and np.isnan(orc.e4m3_decode(0xFF))):
        fails.append("e4m3 0x7f / 0xff are not NaN")
    return fails


def pin_e4m3_attention(orc):
    """Attention on e4m3 codes with per-tensor scales equals the fp64
    attention of the dequantised tensors (torch's decoder times the scales),
    whole and by rows."""
    g = torch.Generator().manual_seed(8)
    shp = (2, 2, 23, 16)
    codes = []
    for _ in range(3):
        c = torch.randint(0, 256, shp, generator=g, dtype=torch.int64).to(torch.uint8)
        c[(c & 0x7F) == 0x7F] = 0x3A  # no NaN codes
        codes.append(c)
    q8, k8, v8 = codes
    sc = (0.5, 0.125, 3.0)
    deq = [c.view(torch.float8_e4m3fn).double().numpy() * s for c, s in zip(codes, sc)]
    fails = []
    rows = [0, 22, 23, 45, 91, 60]
    for causal in (False, True):
        o, lse = orc.attn_e4m3(q8, k8, v8, *sc, causal, 0.02)
        o2, lse2 = orc.attn_f64(*deq, causal, 0.02)
        fails += _close(f"e4m3 attention o causal={causal}", o, o2, 0.0)
        fails += _close(f"e4m3 attention lse causal={causal}", lse, lse2, 0.0)
        orow, lrow = orc.attn_e4m3(q8, k8, v8, *sc, causal, 0.02, rows=rows)
        fails += _close(f"e4m3 rows o causal={causal}", orow, o.reshape(-1, 16)[rows], 0.0)
        fails += _close(f"e4m3 rows lse causal={causal}", lrow, lse.reshape(-1)[rows], 0.0)
    return fails


def pin_e4m3_rectangular(orc):
    """e4m3 attention with Nq != Nk equals the fp64 rectangular attention of
    the dequantised tensors (torch's decoder), whole and by rows."""
    g = torch.Generator().manual_seed(9)
    codes = []
    for shp in ((2, 2, 11, 16), (2, 2, 29, 16), (2, 2, 29, 16)):
        c = torch.randint(0, 256, shp, generator=g, dtype=torch.int64).to(torch.uint8)
        c[(c & 0x7F) == 0x7F] = 0x3A
        codes.append(c)
    q8, k8, v8 = codes
    sc = (0.25, 0.5, 2.0)
    deq = [c.view(torch.float8_e4m3fn).double().numpy() * s for c, s in zip(codes, sc)]
    fails = []
    rows = [0, 10, 11, 43, 25]
    for causal in (False, True):
        o, lse = orc.attn_e4m3_qk(q8, k8, v8, *sc, causal, 0.03)
        o2, lse2 = orc.attn_f64_qk(*deq, causal, 0.03)
        fails += _close(f"e4m3 rect o causal={causal}", o, o2, 0.0)
        fails += _close(f"e4m3 rect lse causal={causal}", lse, lse2, 0.0)
        orow, lrow = orc.attn_e4m3_qk(q8, k8, v8, *sc, causal, 0.03, rows=rows)
        fails += _close(f"e4m3 rect rows o causal={causal}", orow, o.reshape(-1, 16)[rows], 0.0)
        fails += _close(f"e4m3 rect rows lse causal={causal}", lrow, lse.reshape(-1)[rows], 0.0)
    return fails


ALL_PINS = [
    pin_online_softmax_tiling, pin_merge_law, pin_identity_values, pin_constant_values,
    pin_single_key, pin_uniform_queries, pin_zero_scale, pin_permutation,
    pin_causal_future_blind, pin_key_shift, pin_linearity_in_v, pin_library_sdpa,
    pin_golden, pin_bf16_decode, pin_rows_api, pin_bottom_right_suffix, pin_rectangular_sdpa,
    pin_rectangular_bf16_rows, pin_e4m3_decode, pin_e4m3_attention, pin_e4m3_rectangular,
]


def run_all(orc):
    """{pin name: [failures]} for every pin (exceptions count as failures)."""
    out = {}
    for pin in ALL_PINS:
        try:
            out[pin.__name__] = pin(orc)
        except Exception as e:  # a broken oracle may raise, e.g. on bad shapes
            out[pin.__name__] = [f"raised {type(e).__name__}: {e}"]
    return out
