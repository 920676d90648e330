"""The C ABI without a GPU: the library loads, exports exactly what
include/*.h declares, and its host-side argument checks reject bad calls
before anything is launched."""
import ctypes
import glob
import os
import re

import pytest

import exact_attention_51_gb300 as ea
from exact_attention_51_gb300 import build as eabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = "\n".join(l for l in src.splitlines() if not l.lstrip().startswith("#"))
        for m in re.finditer(r"ATTN_API\s+[\w\s\*]*?\b(\w+)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    eabuild.build()
    return ea.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_check_args", "attn_status_string",
            "attn_fwd_device_status", "attn_last_cuda_error"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_only_c_abi_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {ea.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == declared_functions(), exported ^ declared_functions()


def test_status_strings(lib):
    for code in range(7):
        assert ea.attn_status_string(code) not in ("", "unknown status")
    assert ea.attn_status_string(99) == "unknown status"


A = 1 << 20  # fake, 16-byte aligned "device" addresses (never dereferenced)


def ptrs(n_bytes):
    base = [A, A + 4 * n_bytes, A + 8 * n_bytes, A + 12 * n_bytes, A + 16 * n_bytes]
    return base


def chk(q, k, v, o, lse, B=1, H=2, N=128, d=64, scale=0.125, causal=0):
    return ea.attn_fwd_check_args(q, k, v, o, lse, B, H, N, d, scale, causal)


def test_check_args_accepts_valid(lib):
    n = 1 * 2 * 128 * 64 * 2
    assert chk(*ptrs(n)) == ea.ATTN_OK
    assert chk(*ptrs(n), causal=1) == ea.ATTN_OK
    for d in (64, 128, 256):
        assert chk(*ptrs(1 * 2 * 128 * d * 2), d=d) == ea.ATTN_OK
    assert chk(*ptrs(n), scale=0.0) == ea.ATTN_OK
    q = ptrs(n)[0]
    assert chk(q, q, q, *ptrs(n)[3:]) == ea.ATTN_OK  # inputs may alias each other


@pytest.mark.parametrize("field", range(5))
def test_check_args_null_pointer(lib, field):
    p = ptrs(1 << 16)
    p[field] = 0
    assert chk(*p) == ea.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(B=-1), dict(d=32),
                                dict(d=96), dict(d=512), dict(scale=float("nan")),
                                dict(scale=float("inf")), dict(scale=-0.5),
                                dict(B=1 << 20, H=1 << 12), dict(B=1 << 16, H=1 << 8, N=1 << 20)])
def test_check_args_invalid(lib, kw):
    assert chk(*ptrs(1 << 40), **kw) == ea.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("field,off", [(0, 8), (1, 2), (2, 4), (3, 8), (4, 2)])
def test_check_args_misaligned(lib, field, off):
    p = ptrs(1 << 16)
    p[field] += off
    assert chk(*p) == ea.ATTN_ERR_MISALIGNED


def test_check_args_alias(lib):
    n = 1 * 2 * 128 * 64 * 2
    q, k, v, o, lse = ptrs(n)
    assert chk(q, k, v, q, lse) == ea.ATTN_ERR_ALIAS          # o == q
    assert chk(q, k, v, v + 16, lse) == ea.ATTN_ERR_ALIAS     # o overlaps v
    assert chk(q, k, v, o, k + n - 16) == ea.ATTN_ERR_ALIAS   # lse overlaps k's tail
    assert chk(q, k, v, o, o + 64) == ea.ATTN_ERR_ALIAS       # lse inside o
    assert chk(q, k, v, o, o + n) == ea.ATTN_OK               # lse right after o


def test_missing_extension_fails_loudly(tmp_path):
    saved = ea._lib
    ea._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            ea.load_library(str(tmp_path / "nope.so"))
    finally:
        ea._lib = saved


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros((1, 1, 4, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        ea.attn_fwd(x, x, x)


# ------------------------------------------------------------------ split-KV

def test_splitkv_workspace_size(lib):
    def align(x):
        return (x + 255) // 256 * 256
    for (B, H, N, d, S) in [(1, 2, 128, 64, 2), (2, 3, 1000, 128, 5), (1, 1, 7, 256, 64)]:
        rows = B * H * N
        want = align(S * rows * d * 4) + align(S * rows * 4)
        assert ea.attn_fwd_splitkv_workspace_size(B, H, N, d, S) == want
    assert ea.attn_fwd_splitkv_workspace_size(1, 1, 128, 64, 1) == 0
    for bad in [(0, 1, 128, 64, 2), (1, 1, 128, 96, 2), (1, 1, 128, 64, 0), (1, 1, 128, 64, 65)]:
        assert ea.attn_fwd_splitkv_workspace_size(*bad) == 0


def test_splitkv_split_heuristic(lib):
    f = ea.attn_fwd_splitkv_num_splits
    # a launch that already fills the GPU is not split
    assert f(4, 16, 4096, 128, True, 152) == 1
    assert f(1, 32, 16384, 128, True, 152) == 1
    # one head of 8192 keys (32 query blocks of 256 rows): split
    assert 2 <= f(1, 1, 8192, 128, False, 152) <= 16
    # 128 equal blocks already use 84 % of 152 SMs: splitting does not pay
    assert f(1, 4, 8192, 128, False, 152) == 1
    # the same shape causal: the heavy diagonal blocks bound a two-tile
    # launch, but the one-query-tile shape (256 CTAs) already fills the GPU
    assert f(1, 4, 8192, 128, True, 152) == 1
    # one causal head: 64 one-tile CTAs still leave SMs idle, split
    assert 2 <= f(1, 1, 8192, 128, True, 152) <= 16
    # degenerate inputs
    assert f(1, 1, 1024, 64, False, 0) == 1
    assert f(0, 1, 1024, 64, False, 152) == 1
    for args in [(1, 1, 1, 64, False), (1, 2, 100000, 256, True), (2, 3, 777, 128, True)]:
        assert 1 <= f(*args, 152) <= 16


def test_kvcache_split_heuristic(lib):
    f = ea.attn_fwd_kvcache_num_splits
    # a decoding step: 32 heads of one query block against 16384 cached
    # keys leave most SMs idle, so the keys are shared out
    assert 2 <= f(1, 32, 16, 16384, 128, True, 152) <= 16
    assert 2 <= f(1, 32, 1, 16384, 128, True, 152) <= 16
    # the same with enough heads to fill the GPU: no split
    assert f(8, 32, 16, 16384, 128, True, 152) == 1
    # the square case is the attn_fwd model
    for args in [(1, 4, 8192, 8192, 128, True), (1, 1, 8192, 8192, 128, False)]:
        B, H, Nq, Nk, d, c = args
        assert f(*args, 152) == ea.attn_fwd_splitkv_num_splits(B, H, Nq, d, c, 152)
    # causal needs Nk >= Nq; invalid shapes get 1
    assert f(1, 1, 100, 50, 128, True, 152) == 1
    assert f(1, 1, 16, 1024, 96, True, 152) == 1
    # the e4m3 model runs on the same shapes
    assert 2 <= ea.attn_fwd_fp8_kvcache_num_splits(1, 32, 16, 16384, 128, True, 152) <= 16


def _splitkv(lib, p, splits, ws, ws_bytes, **kw):
    B, H, N, d = kw.get("B", 1), kw.get("H", 2), kw.get("N", 128), kw.get("d", 64)
    return lib.attn_fwd_splitkv(*p, B, H, N, d, 0.125, 0, splits, ws, ws_bytes, None)


def test_splitkv_rejects_bad_arguments(lib):
    n = 1 * 2 * 128 * 64 * 2
    p = ptrs(n)
    need = ea.attn_fwd_splitkv_workspace_size(1, 2, 128, 64, 4)
    ws = A + (1 << 30)
    assert _splitkv(lib, p, 0, ws, need) == ea.ATTN_ERR_INVALID_ARG
    assert _splitkv(lib, p, 65, ws, need) == ea.ATTN_ERR_INVALID_ARG
    assert _splitkv(lib, p, 4, None, need) == ea.ATTN_ERR_INVALID_ARG
    assert _splitkv(lib, p, 4, ws, need - 1) == ea.ATTN_ERR_INVALID_ARG
    assert _splitkv(lib, p, 4, ws + 16, need) == ea.ATTN_ERR_MISALIGNED
    assert _splitkv(lib, p, 4, p[1] - (p[1] % 256), need) == ea.ATTN_ERR_ALIAS  # over k
    q = list(p)
    q[0] = 0
    assert _splitkv(lib, q, 4, ws, need) == ea.ATTN_ERR_INVALID_ARG


# ------------------------------------------------------------------ KV cache

def _kvcache(lib, p, Nq, Nk, causal, splits=1, ws=None, ws_bytes=0, d=64):
    return lib.attn_fwd_kvcache(*p, 1, 2, Nq, Nk, d, 0.125, causal, splits, ws, ws_bytes, None)


def test_kvcache_rejects_bad_arguments(lib):
    big = 1 << 24
    p = ptrs(big)
    # causal needs at least as many keys as queries
    assert _kvcache(lib, p, 10, 9, 1) == ea.ATTN_ERR_INVALID_ARG
    assert _kvcache(lib, p, 0, 9, 0) == ea.ATTN_ERR_INVALID_ARG
    assert _kvcache(lib, p, 9, 0, 0) == ea.ATTN_ERR_INVALID_ARG
    assert _kvcache(lib, p, 9, 9, 0, d=80) == ea.ATTN_ERR_INVALID_ARG
    # o may not overlap the (longer) key tensor: keys span 1*2*4096*64*2 bytes
    q, k, v, o, lse = p
    assert _kvcache(lib, [q, k, v, k + 512 * 1024, lse], 16, 4096, 1) == ea.ATTN_ERR_ALIAS
    # a split run needs its workspace
    assert _kvcache(lib, p, 16, 4096, 1, splits=4) == ea.ATTN_ERR_INVALID_ARG


def test_kvcache_split_heuristic(lib):
    f = ea.attn_fwd_kvcache_num_splits
    # decode: one query per head against a long cache -> split
    assert f(1, 8, 1, 32768, 128, True, 152) >= 2
    # Nq = Nk matches the square heuristic
    for args in [(1, 4, 8192, 128, True), (1, 1, 8192, 128, False), (4, 16, 4096, 128, True)]:
        B, H, N, d, c = args
        assert f(B, H, N, N, d, c, 152) == ea.attn_fwd_splitkv_num_splits(B, H, N, d, c, 152)
    assert f(1, 1, 9, 8, 128, True, 152) == 1  # invalid causal shape


# ------------------------------------------------------------------- e4m3

def _fp8(lib, p, ws, ws_bytes, d=128, descales=(1.0, 1.0, 1.0), N=256):
    q, k, v, o, lse = p
    return lib.attn_fwd_fp8(q, k, v, *descales, o, lse, 1, 2, N, d, 0.088, 1, ws, ws_bytes, None)


def test_fp8_workspace_size(lib):
    # the kernel reads V as stored: no workspace without split-KV
    for d in (64, 128, 256):
        assert ea.attn_fwd_fp8_workspace_size(1, 2, 256, d) == 0
    assert ea.attn_fwd_fp8_workspace_size(0, 1, 17, 128) == 0
    assert ea.attn_fwd_fp8_workspace_size(1, 1, 17, 96) == 0


def test_fp8_rejects_bad_arguments(lib):
    # every call below is invalid, so nothing is ever launched
    p = ptrs(1 << 24)
    assert _fp8(lib, p, None, 0, d=96) == ea.ATTN_ERR_INVALID_ARG
    assert _fp8(lib, p, None, 0, d=32) == ea.ATTN_ERR_INVALID_ARG
    for bad in [(0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, float("nan")),
                (float("inf"), 1.0, 1.0)]:
        assert _fp8(lib, p, None, 0, descales=bad) == ea.ATTN_ERR_INVALID_ARG
    assert _fp8(lib, p, None, 0, N=0) == ea.ATTN_ERR_INVALID_ARG
    q, k, v, o, lse = p
    assert _fp8(lib, [q + 8, k, v, o, lse], None, 0) == ea.ATTN_ERR_MISALIGNED
    assert _fp8(lib, [q, k, v, o, lse + 2], None, 0, d=64) == ea.ATTN_ERR_MISALIGNED
    # o overlapping v (v spans 1*2*256*128 one-byte codes)
    assert _fp8(lib, [q, k, v, v + 4096, lse], None, 0) == ea.ATTN_ERR_ALIAS
    # lse overlapping o
    assert _fp8(lib, [q, k, v, o, o + 64], None, 0) == ea.ATTN_ERR_ALIAS


# --------------------------------------------------------------- backward

def test_bwd_rejects_bad_arguments(lib):
    # every call below is invalid, so nothing is ever launched
    N, d = 256, 64
    n = 1 * 2 * N * d * 2
    base = ptrs(1 << 24)
    q, k, v, o, lse = base
    g = A + 40 * (1 << 24)
    dq, dk, dv = g + (1 << 24), g + 2 * (1 << 24), g + 3 * (1 << 24)
    ws = g + 4 * (1 << 24)
    need = ea.attn_bwd_workspace_size(1, 2, N)

    def call(dd=d, w=ws, wb=need, grads=(dq, dk, dv), dout=g):
        return lib.attn_bwd(q, k, v, o, dout, lse, *grads, 1, 2, N, dd, 0.125, 1, w, wb, None)

    for bad_d in (32, 96, 192, 512):
        assert call(dd=bad_d) == ea.ATTN_ERR_INVALID_ARG
    assert call(wb=need - 1) == ea.ATTN_ERR_INVALID_ARG
    assert call(w=None) == ea.ATTN_ERR_INVALID_ARG
    assert call(w=ws + 16) == ea.ATTN_ERR_MISALIGNED
    assert call(dout=None) == ea.ATTN_ERR_INVALID_ARG
    assert call(grads=(dq + 2, dk, dv)) == ea.ATTN_ERR_MISALIGNED
    assert call(grads=(dq, dq + n // 2, dv)) == ea.ATTN_ERR_ALIAS  # dk over dq
    assert call(grads=(q, dk, dv)) == ea.ATTN_ERR_ALIAS  # dq over q
    assert ea.attn_bwd_workspace_size(1, 2, 1) == 2 * 256 * ((2 * 128 * 4 + 255) // 256)


def test_fp8_kvcache_rejects_bad_arguments(lib):
    # every call below is invalid, so nothing is ever launched
    q, k, v, o, lse = ptrs(1 << 24)
    ws = A + (1 << 30)

    def call(Nq=16, Nk=4096, d=128, causal=1, splits=1, w=ws, wb=None):
        need = ea.load_library().attn_fwd_fp8_kvcache_workspace_size(1, 2, Nq, Nk, d, splits)
        return lib.attn_fwd_fp8_kvcache(q, k, v, 1.0, 1.0, 1.0, o, lse, 1, 2, Nq, Nk, d, 0.088,
                                        causal, splits, w, need if wb is None else wb, None)

    assert call(Nq=4097) == ea.ATTN_ERR_INVALID_ARG          # causal needs Nk >= Nq
    assert call(d=96) == ea.ATTN_ERR_INVALID_ARG
    assert call(splits=0) == ea.ATTN_ERR_INVALID_ARG
    assert call(splits=65) == ea.ATTN_ERR_INVALID_ARG
    assert call(splits=4, wb=1024) == ea.ATTN_ERR_INVALID_ARG  # workspace too small
    assert call(splits=4, w=ws + 16) == ea.ATTN_ERR_MISALIGNED
    assert call(splits=4, w=None) == ea.ATTN_ERR_INVALID_ARG
    assert call(splits=4, d=64, w=None) == ea.ATTN_ERR_INVALID_ARG
    # the split-KV workspace overlapping q
    assert call(splits=4, w=q - (q % 256)) == ea.ATTN_ERR_ALIAS
    # o over the (longer) key tensor: keys span 1*2*4096*128 one-byte codes
    assert lib.attn_fwd_fp8_kvcache(q, k, v, 1.0, 1.0, 1.0, k + 4096, lse, 1, 2, 16, 4096, 128,
                                    0.088, 1, 1, ws, 1 << 24, None) == ea.ATTN_ERR_ALIAS
    f = ea.load_library().attn_fwd_fp8_kvcache_workspace_size
    assert f(1, 2, 16, 4096, 128, 1) == ea.attn_fwd_fp8_workspace_size(1, 2, 4096, 128) == 0
    # split-KV partials: splits * B*H*Nq * (d + 1) fp32, each part 256-byte padded
    assert f(1, 2, 16, 4096, 128, 4) == (256 * ((4 * 32 * 128 * 4 + 255) // 256)
                                         + 256 * ((4 * 32 * 4 + 255) // 256))
    assert f(1, 2, 16, 4096, 64, 4) == ea.attn_fwd_splitkv_workspace_size(1, 2, 16, 64, 4)
    assert f(1, 2, 16, 4096, 96, 1) == 0
    assert ea.load_library().attn_fwd_fp8_kvcache_num_splits(1, 8, 1, 32768, 128, 1, 152) >= 2


def _noalloc(lib, p, B, H, N, d, splits, causal=0, scale=0.125):
    vp = ctypes.c_void_p
    return lib.attn_fwd_splitkv_noalloc(vp(p[0]), vp(p[1]), vp(p[2]), vp(p[3]), vp(p[4]), B, H, N,
                                        d, ctypes.c_float(scale), causal, splits, None)


def test_noalloc_host_checks_come_before_the_device(lib):
    """attn_fwd_splitkv_noalloc answers bad arguments, a split count out of
    range and a problem beyond its fixed array before it touches the device
    (these run without a GPU)."""
    n = 1 * 64 * 8192 * 128 * 2
    p = ptrs(n)
    assert _noalloc(lib, p, 1, 64, 8192, 128, 4) == ea.ATTN_ERR_NOALLOC_TOO_LARGE
    for splits in (0, -3, 65):
        assert _noalloc(lib, p, 1, 2, 128, 64, splits) == ea.ATTN_ERR_INVALID_ARG
    assert _noalloc(lib, p, 1, 2, 128, 96, 2) == ea.ATTN_ERR_INVALID_ARG      # d
    assert _noalloc(lib, [A + 2] + p[1:], 1, 2, 128, 64, 2) == ea.ATTN_ERR_MISALIGNED
    assert _noalloc(lib, p, 1, 2, 128, 64, 2, scale=-1.0) == ea.ATTN_ERR_INVALID_ARG
