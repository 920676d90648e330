"""GB300-native fused exact attention forward (sm_103a).

A thin ctypes binding over the C ABI in ``include/attn_fwd.h`` (library
``libexact_attn_gb300.so`` built in place by ``exact_attention_51_gb300.build``).
Every step of the computation runs in the CUDA kernels behind ``attn_fwd``;
this module only marshals torch tensors (device memory) and the current CUDA
stream into the C call.  There is no CPU fallback: without the built library
every call raises.

    O   = softmax(scale * Q K^T [+ causal mask]) V      (bf16 [B,H,N,d])
    LSE = ln sum_j exp(scale * q_i . k_j)                (fp32 [B,H,N])

Sources: "Tri Dao: prediction" (fusion, tiling, online softmax); "Show HN:
Flash Attention in ~100 lines of CUDA" (forward pass, torch only for
bindings); HN item 40939030 (causal = softmax of the triangular matrix).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libexact_attn_gb300.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_MISALIGNED = 2
ATTN_ERR_ALIAS = 3
ATTN_ERR_UNSUPPORTED_DEVICE = 4
ATTN_ERR_LAUNCH = 5
ATTN_ERR_TIMEOUT = 6
ATTN_ERR_NOALLOC_TOO_LARGE = 7
NOALLOC_WORKSPACE_BYTES = 64 * 1024 * 1024  # ATTN_NOALLOC_WORKSPACE_BYTES

SUPPORTED_HEAD_DIMS = (64, 128, 256)
FP8_HEAD_DIMS = (64, 128, 256)  # head dims of attn_fwd_fp8 / attn_fwd_fp8_kvcache

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_int = ctypes.c_int
_flt = ctypes.c_float


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH):
    """Load the CUDA extension (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA extension {path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or python -m exact_attention_51_gb300.build)")
        lib = ctypes.CDLL(path)
        lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _flt, _int, _vp]
        lib.attn_fwd.restype = _int
        lib.attn_fwd_check_args.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _flt,
                                            _int]
        lib.attn_fwd_check_args.restype = _int
        lib.attn_status_string.argtypes = [_int]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_fwd_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint)]
        lib.attn_fwd_device_status.restype = _int
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_last_cuda_error.restype = _int
        lib.attn_fwd_splitkv.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _flt,
                                         _int, _int, _vp, ctypes.c_size_t, _vp]
        lib.attn_fwd_splitkv.restype = _int
        lib.attn_fwd_splitkv_workspace_size.argtypes = [_int, _int, _int, _int, _int]
        lib.attn_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_splitkv_num_splits.argtypes = [_int, _int, _int, _int, _int, _int]
        lib.attn_fwd_splitkv_num_splits.restype = _int
        lib.attn_fwd_splitkv_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int,
                                                 _flt, _int, _int, _vp]
        lib.attn_fwd_splitkv_noalloc.restype = _int
        lib.attn_fwd_kvcache.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int,
                                         _flt, _int, _int, _vp, ctypes.c_size_t, _vp]
        lib.attn_fwd_kvcache.restype = _int
        lib.attn_fwd_kvcache_num_splits.argtypes = [_int, _int, _int, _int, _int, _int, _int]
        lib.attn_fwd_kvcache_num_splits.restype = _int
        lib.attn_bwd.argtypes = [_vp] * 9 + [_int] * 4 + [_flt, _int, _vp, ctypes.c_size_t, _vp]
        lib.attn_bwd.restype = _int
        lib.attn_bwd_workspace_size.argtypes = [_int, _int, _int]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_fp8.argtypes = [_vp, _vp, _vp, _flt, _flt, _flt, _vp, _vp, _int, _int, _int,
                                     _int, _flt, _int, _vp, ctypes.c_size_t, _vp]
        lib.attn_fwd_fp8.restype = _int
        lib.attn_fwd_fp8_workspace_size.argtypes = [_int, _int, _int, _int]
        lib.attn_fwd_fp8_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_fp8_kvcache.argtypes = [_vp, _vp, _vp, _flt, _flt, _flt, _vp, _vp, _int, _int,
                                             _int, _int, _int, _flt, _int, _int, _vp,
                                             ctypes.c_size_t, _vp]
        lib.attn_fwd_fp8_kvcache.restype = _int
        lib.attn_fwd_fp8_kvcache_workspace_size.argtypes = [_int] * 6
        lib.attn_fwd_fp8_kvcache_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_fp8_kvcache_num_splits.argtypes = [_int] * 7
        lib.attn_fwd_fp8_kvcache_num_splits.restype = _int
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp]
        lib.attn_selftest_wait_timeout.restype = _int
        lib.attn_selftest_fwd_dropped_load.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int,
                                                       _int, _flt, _int, _int, ctypes.c_uint, _vp]
        lib.attn_selftest_fwd_dropped_load.restype = _int
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_last_cuda_error() -> int:
    return int(load_library().attn_last_cuda_error())


def attn_fwd_check_args(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                        H: int, N: int, d: int, scale: float, causal: bool) -> int:
    """Host-only argument checks on raw pointers (never dereferenced)."""
    return int(load_library().attn_fwd_check_args(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N,
                                                  d, float(scale), int(bool(causal))))


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def attn_fwd_splitkv_workspace_size(B: int, H: int, N: int, d: int, num_splits: int) -> int:
    return int(load_library().attn_fwd_splitkv_workspace_size(B, H, N, d, num_splits))


def attn_fwd_splitkv_num_splits(B: int, H: int, N: int, d: int, causal: bool,
                                num_sms: int) -> int:
    return int(load_library().attn_fwd_splitkv_num_splits(B, H, N, d, int(bool(causal)),
                                                           num_sms))


def _check_qkv(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, d]")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")


def _outputs(q, out, lse):
    import torch
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor on q's device")
    return out, lse


def _buffer(t):
    """(device pointer, bytes) of an optional scratch tensor; (None, 0) for none."""
    if t is None:
        return None, 0
    return t.data_ptr(), t.numel() * t.element_size()


def attn_fwd_fp8_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_fwd_fp8_workspace_size(B, H, N, d))


def attn_fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float,
                 causal: bool = False, scale: float | None = None, out=None, lse=None,
                 workspace=None, stream=None):
    """Attention forward on e4m3 inputs: q, k, v CUDA tensors [B, H, N, d], d = 64, 128
    or 256, of dtype float8_e4m3fn (or uint8 holding e4m3 codes), element x
    meaning ``descale * x``.  Returns ``(o, lse)``: o bf16 [B,H,N,d], lse fp32
    [B,H,N].  A workspace, if the call needs one
    (``attn_fwd_fp8_workspace_size``), is allocated with torch unless
    given."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda \
                or t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must be a CUDA float8_e4m3fn (or uint8) tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, d]")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor on q's device")
    need = attn_fwd_fp8_workspace_size(B, H, N, d)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = _buffer(workspace)
    with torch.cuda.device(q.device):
        rc = load_library().attn_fwd_fp8(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), float(descale_q), float(descale_k),
            float(descale_v), out.data_ptr(), lse.data_ptr(), B, H, N, d, float(scale),
            int(bool(causal)), ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return out, lse


def attn_fwd_fp8_kvcache(q, k, v, descale_q: float, descale_k: float, descale_v: float,
                         causal: bool = False, scale: float | None = None,
                         num_splits: int | None = None, out=None, lse=None, workspace=None,
                         stream=None):
    """e4m3 forward with q [B,H,Nq,d] and k, v [B,H,Nk,d] (d = 64, 128 or 256):
    the queries are the last Nq positions (causal diagonal at the
    bottom-right).  ``num_splits`` None picks one from the shape and the SM
    count.  Returns ``(o, lse)`` as attn_fwd_fp8."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda \
                or t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must be a CUDA float8_e4m3fn (or uint8) tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k, v must be [B, H, Nk, d] with q's B, H and d")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = int(lib.attn_fwd_fp8_kvcache_num_splits(B, H, Nq, Nk, d, int(bool(causal)),
                                                              sms))
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    elif out.shape != (B, H, Nq, d) or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 [B, H, Nq, d] tensor on q's device")
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor on q's device")
    need = int(lib.attn_fwd_fp8_kvcache_workspace_size(B, H, Nq, Nk, d, num_splits))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = _buffer(workspace)
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_fp8_kvcache(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), float(descale_q), float(descale_k),
            float(descale_v), out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d, float(scale),
            int(bool(causal)), int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8_kvcache")
    return out, lse


def attn_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                     num_splits: int | None = None, out=None, lse=None, workspace=None,
                     stream=None):
    """Split-KV forward (same result as ``attn_fwd``).  ``num_splits`` None
    picks one from the shape and the SM count; the workspace is allocated
    with torch unless given (a uint8 CUDA tensor of enough bytes)."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = attn_fwd_splitkv_num_splits(B, H, N, d, causal, sms)
    out, lse = _outputs(q, out, lse)
    need = attn_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                                  int(num_splits), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv")
    return out, lse


def attn_fwd_kvcache_num_splits(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool,
                                num_sms: int) -> int:
    return int(load_library().attn_fwd_kvcache_num_splits(B, H, Nq, Nk, d, int(bool(causal)),
                                                           num_sms))


def attn_fwd_kvcache(q, k, v, causal: bool = False, scale: float | None = None,
                     num_splits: int | None = None, out=None, lse=None, workspace=None,
                     stream=None):
    """Attention with q [B,H,Nq,d] and k, v [B,H,Nk,d] (KV-cache shapes).

    Causal aligns the diagonal to the bottom-right corner (query i sees keys
    j <= i + Nk - Nq; needs Nk >= Nq).  ``num_splits`` None picks one from the
    shape and the SM count; the split-KV workspace is allocated with torch
    unless given.  Returns ``(o [B,H,Nq,d] bf16, lse [B,H,Nq] fp32)``.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous and 4-D")
    B, H, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k, v must be [B, H, Nk, d] with q's B, H and d")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = attn_fwd_kvcache_num_splits(B, H, Nq, Nk, d, causal, sms)
    out, lse = _outputs(q, out, lse)
    need = attn_fwd_splitkv_workspace_size(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = load_library().attn_fwd_kvcache(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq,
            Nk, d, float(scale), int(bool(causal)), int(num_splits), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_kvcache")
    return out, lse


def attn_fwd_splitkv_noalloc(q, k, v, causal: bool = False, scale: float | None = None,
                             num_splits: int = 2, out=None, lse=None, stream=None):
    """``attn_fwd_splitkv`` whose workspace is the library's fixed device
    array (NOALLOC_WORKSPACE_BYTES): the C call allocates nothing, for
    callers that cannot allocate device memory.  Calls that overlap on the
    GPU race on the shared array; ``out`` / ``lse`` are allocated here with
    torch unless given."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    with torch.cuda.device(q.device):
        rc = load_library().attn_fwd_splitkv_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), int(num_splits), _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv_noalloc")
    return out, lse


def attn_bwd_workspace_size(B: int, H: int, N: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, H, N))


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of the forward pass: ``(dq, dk, dv)`` bf16 [B,H,N,d] for the
    upstream gradient ``dout`` of ``o``, given the forward's ``o`` and ``lse``
    (as returned by ``attn_fwd`` with the same ``causal`` and ``scale``).
    Head dims 64, 128 and 256.  The small fp32 workspace (2 * B*H*ceil128(N) floats)
    is allocated with torch unless given."""
    import torch
    _check_qkv(q, k, v)
    _check_qkv(o, dout, q)
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() \
                or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    need = attn_bwd_workspace_size(B, H, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = load_library().attn_bwd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             stream=None):
    """Fused attention forward on CUDA bf16 tensors [B, H, N, d].

    Returns ``(o, lse)``: o bf16 [B,H,N,d], lse fp32 [B,H,N] (natural log,
    scale included).  ``scale`` defaults to 1/sqrt(d).  ``out`` / ``lse`` may
    be given to write in place.  The call is asynchronous on ``stream``
    (default: torch's current stream of q's device).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, d]")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous bf16 tensor shaped like q on q's device")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor on q's device")
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                          B, H, N, d, float(scale), int(bool(causal)),
                          _stream_handle(stream, q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_selftest_wait_timeout(timeout_ms: int = 100, stream=None, device=None) -> int:
    """Enqueue the bounded-wait self-test kernel (see include/attn_fwd.h)."""
    import torch
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return int(load_library().attn_selftest_wait_timeout(int(timeout_ms),
                                                             _stream_handle(stream, device)))


def attn_selftest_fwd_dropped_load(q, k, v, out, lse, causal: bool, drop_load: int,
                                   timeout_ms: int = 50, scale: float | None = None,
                                   stream=None) -> int:
    """Enqueue the forward's abort-path self-test (see include/attn_fwd.h):
    attn_fwd on these tensors with the copy of ring position ``drop_load``
    left out and every wait limited to ``timeout_ms``.  Returns the C status;
    the outcome is read with ``attn_fwd_device_status``."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    with torch.cuda.device(q.device):
        return int(load_library().attn_selftest_fwd_dropped_load(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), int(drop_load), int(timeout_ms),
            _stream_handle(stream, q.device)))


def attn_fwd_device_status(stream=None, device=None):
    """Synchronise the stream, read and clear the device wait-timeout word.

    Returns ``(status, detail)``; status is ATTN_OK or ATTN_ERR_TIMEOUT.
    """
    import torch
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    detail = ctypes.c_uint(0)
    with torch.cuda.device(device):
        rc = load_library().attn_fwd_device_status(_stream_handle(stream, device),
                                                   ctypes.byref(detail))
    return int(rc), int(detail.value)
