"""exact_attention_30_gb300 -- fused exact attention for GB300 (sm_103a).

A thin Python binding over the C ABI in ``include/fa.h`` (``libfa_gb300.so``).
It only marshals arguments: checks that tensors live on the GPU, are
contiguous and of the right dtype, allocates outputs with PyTorch (device
memory is PyTorch's job here) and passes raw pointers plus the current CUDA
stream to the library. Every step of the computation runs in the library's
CUDA kernels; there is no CPU path. If the shared library has not been built
(``python -m exact_attention_30_gb300.build``), every call raises.

    o, lse = fa_fwd(q, k, v, scale)                 # q,k,v: [B,H,N,d] cuda
    dq, dk, dv = fa_bwd(q, k, v, o, do, lse, scale)
    o, lse = fa_decode(q_new, k_cache, v_cache, scale)   # q_new: [B,H,Nq<=16,d]
    o, lse = fa_fwd(q, k, v, causal=True)            # causal self-attention
    o, lse = fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen)   # packed [total,H,d]
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

__all__ = [
    "fa_fwd", "fa_bwd", "fa_bwd_stage", "fa_bwd_plan", "fa_fwd_varlen", "fa_bwd_varlen",
    "fa_bwd_varlen_workspace_bytes", "FA_CAUSAL", "fa_bwd_workspace_bytes", "fa_softmax_rows", "fa_decode",
    "fa_decode_workspace_bytes", "fa_decode_plan", "fa_check_device_status",
    "fa_debug_timeout_probe", "fa_status_string", "fa_version", "library_path", "load_library",
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
    "FA_F32", "FA_BF16", "FAError", "FA_BWD_PREPROCESS", "FA_BWD_MAIN", "FA_BWD_DQ_CONVERT",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_F32, FA_BF16 = 0, 1
FA_BWD_PREPROCESS, FA_BWD_MAIN, FA_BWD_DQ_CONVERT = 0, 1, 2
FA_CAUSAL = 1
_STAGE_FLAGS = {FA_BWD_PREPROCESS: 1 << 8, FA_BWD_MAIN: 2 << 8, FA_BWD_DQ_CONVERT: 4 << 8}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")
_lib = None

_vp, _ci, _cf, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "fa_fwd": (_ci, [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _ci, _vp]),
    "fa_fwd_ex": (_ci, [_vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp]),
    "fa_fwd_varlen": (_ci, [_vp] * 6 + [_ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp]),
    "fa_fwd_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci]),
    "fa_fwd_ws": (_ci, [_vp] * 6 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp]),
    "fa_fwd_plan": (_ci, [_ci] * 7 + [ctypes.POINTER(_ci)] * 3),
    "fa_bwd_ex": (_ci, [_vp] * 10 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp]),
    "fa_bwd_varlen_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci]),
    "fa_bwd_varlen": (_ci, [_vp] * 11 + [_sz, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _ci, _vp]),
    "fa_bwd_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci]),
    "fa_bwd_plan": (_ci, [_ci] * 7 + [ctypes.POINTER(_ci)] * 3),
    "fa_bwd": (_ci, [_vp] * 10 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci, _vp]),
    "fa_bwd_stage": (_ci, [_ci] + [_vp] * 10 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci, _vp]),
    "fa_bwd_noalloc": (_ci, [_vp] * 9 + [_ci, _ci, _ci, _ci, _cf, _ci, _vp]),
    "fa_softmax_rows": (_ci, [_vp, _vp, _ci, _ci, _cf, _ci, _vp]),
    "fa_decode": (_ci, [_vp] * 6 + [_sz, _ci, _ci, _ci, _ci, _ci, _cf, _ci, _vp]),
    "fa_decode_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci, _ci]),
    "fa_decode_plan": (_ci, [_ci, _ci, _ci, _ci, _ci, _ci, ctypes.POINTER(_ci), ctypes.POINTER(_ci)]),
    "fa_check_device_status": (_ci, [_vp]),
    "fa_debug_timeout_probe": (_ci, [ctypes.c_longlong, _vp]),
    "fa_debug_fwd_skip_load": (_ci, [_vp] * 5 + [_ci, _ci, _ci, _ci, _cf, _ci, ctypes.c_longlong, _vp]),
    "fa_debug_bwd_skip_load": (_ci, [_vp] * 10 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci,
                                                  ctypes.c_longlong, _vp]),
    "fa_debug_bwd_skip_load_ex": (_ci, [_vp] * 10 + [_sz, _ci, _ci, _ci, _ci, _cf, _ci, _ci,
                                                     ctypes.c_longlong, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_ci]),
    "fa_version": (_ci, []),
}


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fa_status_string(code)}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libfa_gb300.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -m exact_attention_30_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(header_path: str | None = None):
    """Names of the functions declared in include/fa.h (for export checks)."""
    path = header_path or os.path.join(os.path.dirname(_HERE), "include", "fa.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def fa_status_string(code: int) -> str:
    return load_library().fa_status_string(int(code)).decode()


def fa_version() -> int:
    return load_library().fa_version()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")


def _check(t: torch.Tensor, name: str, like: torch.Tensor | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B,H,N,d]")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype or t.device != like.device):
        raise ValueError(f"{name} must match q in shape, dtype and device")


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _raise(code: int, where: str):
    if code != FA_OK:
        raise FAError(code, where)


def fa_fwd_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool = False,
                           dtype=torch.bfloat16) -> int:
    """Scratch bytes with which the forward splits its last, partly filled
    wave of CTAs on the current device (0: nothing to gain)."""
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    return int(load_library().fa_fwd_workspace_bytes(B, H, N, d, FA_CAUSAL if causal else 0, code))


def fa_fwd_plan(B: int, H: int, N: int, d: int, causal: bool = False, dtype=torch.bfloat16,
                resident_ctas: int = 0):
    """(n_full, n_tail, splits) of the forward's schedule (fa_fwd_plan in fa.h)."""
    nf, nt, sp = _ci(), _ci(), _ci()
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    rc = load_library().fa_fwd_plan(B, H, N, d, FA_CAUSAL if causal else 0, code, resident_ctas,
                                    ctypes.byref(nf), ctypes.byref(nt), ctypes.byref(sp))
    _raise(rc, "fa_fwd_plan")
    return nf.value, nt.value, sp.value


def fa_bwd_plan(B: int, H: int, N: int, d: int, causal: bool = False, dtype=torch.bfloat16,
                resident_ctas: int = 0):
    """(n_full, n_tail, splits) of the backward main kernel's schedule (fa_bwd_plan in fa.h)."""
    nf, nt, sp = _ci(), _ci(), _ci()
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    rc = load_library().fa_bwd_plan(B, H, N, d, FA_CAUSAL if causal else 0, code, resident_ctas,
                                    ctypes.byref(nf), ctypes.byref(nt), ctypes.byref(sp))
    _raise(rc, "fa_bwd_plan")
    return nf.value, nt.value, sp.value


def fa_fwd(q, k, v, scale: float | None = None, out=None, lse=None, causal: bool = False,
           workspace=None):
    """Forward pass: returns (O [B,H,N,d] like q, LSE [B,H,N] float32).

    When the problem gains from splitting the tail of the schedule
    (fa_fwd_workspace_bytes > 0), the scratch is allocated here unless a
    uint8 CUDA tensor of at least that size is passed as ``workspace``."""
    lib = load_library()
    _check(q, "q")
    _check(k, "k", q)
    _check(v, "v", q)
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "out", q)
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_cuda:
        raise ValueError("lse must be float32 [B,H,N] on the same device")
    flags = FA_CAUSAL if causal else 0
    with torch.cuda.device(q.device):
        ws_bytes = int(lib.fa_fwd_workspace_bytes(B, H, N, d, flags, _dtype_code(q)))
        if ws_bytes > 0 and workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            if workspace.dtype != torch.uint8 or not workspace.is_cuda or workspace.device != q.device:
                raise ValueError("workspace must be a uint8 tensor on q's device")
            rc = lib.fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               workspace.data_ptr(), workspace.numel(), B, H, N, d, scale, flags,
                               _dtype_code(q), _stream_ptr(q.device))
        else:
            rc = lib.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, N, d, scale, flags, _dtype_code(q), _stream_ptr(q.device))
    _raise(rc, "fa_fwd")
    return o, lse


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int, dtype=torch.bfloat16) -> int:
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    return int(load_library().fa_bwd_workspace_bytes(B, H, N, d, code))


def _bwd_call(stage, q, k, v, o, do, lse, scale, workspace, dq, dk, dv, causal=False):
    lib = load_library()
    _check(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n, q)
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B,H,N] on the same device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if workspace is None:
        ws_bytes = fa_bwd_workspace_bytes(B, H, N, d, q.dtype)
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, q)
    if stage is not None and stage not in _STAGE_FLAGS:
        raise ValueError(f"unknown backward stage {stage}")
    flags = (FA_CAUSAL if causal else 0) | (0 if stage is None else _STAGE_FLAGS[stage])
    with torch.cuda.device(q.device):
        rc = lib.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                           lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           B, H, N, d, scale, flags, _dtype_code(q), _stream_ptr(q.device))
    _raise(rc, "fa_bwd" if stage is None else "fa_bwd_stage")
    return dq, dk, dv


def fa_bwd(q, k, v, o, do, lse, scale: float | None = None, workspace=None, dq=None, dk=None,
           dv=None, causal: bool = False):
    """Backward pass: returns (dQ, dK, dV), each like q."""
    return _bwd_call(None, q, k, v, o, do, lse, scale, workspace, dq, dk, dv, causal)


def fa_bwd_stage(stage: int, q, k, v, o, do, lse, scale: float | None = None, workspace=None,
                 dq=None, dk=None, dv=None, causal: bool = False):
    """One backward stage (FA_BWD_PREPROCESS, FA_BWD_MAIN, FA_BWD_DQ_CONVERT) on ``workspace``."""
    return _bwd_call(stage, q, k, v, o, do, lse, scale, workspace, dq, dk, dv, causal)


def _check_varlen(q, cu_seqlens, max_seqlen):
    _check(q, "q")
    if q.dim() != 3:
        raise ValueError("packed tensors are [total, H, d]")
    if not isinstance(cu_seqlens, torch.Tensor) or not cu_seqlens.is_cuda or \
            cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor [B+1]")
    if cu_seqlens.device != q.device:
        raise ValueError("cu_seqlens must be on q's device")
    total, H, d = q.shape
    return cu_seqlens.numel() - 1, H, total, int(max_seqlen), d


def fa_bwd_varlen_workspace_bytes(B: int, H: int, total: int, max_seqlen: int, d: int,
                                  dtype=torch.bfloat16) -> int:
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    return int(load_library().fa_bwd_varlen_workspace_bytes(B, H, total, max_seqlen, d, code))


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, scale: float | None = None,
                  causal: bool = False, out=None, lse=None):
    """Packed variable-length forward: q, k, v [total, H, d]; cu_seqlens int32 [B+1] on the GPU.

    Returns (O [total, H, d] like q, LSE [H, total] float32).
    """
    lib = load_library()
    B, H, total, max_seqlen, d = _check_varlen(q, cu_seqlens, max_seqlen)
    _check(k, "k", q)
    _check(v, "v", q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "out", q)
    if lse.dtype != torch.float32 or lse.shape != (H, total) or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [H, total] on the same device")
    with torch.cuda.device(q.device):
        rc = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               cu_seqlens.data_ptr(), B, H, total, max_seqlen, d, scale,
                               FA_CAUSAL if causal else 0, _dtype_code(q), _stream_ptr(q.device))
    _raise(rc, "fa_fwd_varlen")
    return o, lse


def fa_bwd_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen: int, scale: float | None = None,
                  causal: bool = False, workspace=None):
    """Backward of ``fa_fwd_varlen``: returns (dQ, dK, dV), each [total, H, d] like q."""
    lib = load_library()
    B, H, total, max_seqlen, d = _check_varlen(q, cu_seqlens, max_seqlen)
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n, q)
    if lse.dtype != torch.float32 or lse.shape != (H, total) or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [H, total] on the same device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    with torch.cuda.device(q.device):
        if workspace is None:
            n = fa_bwd_varlen_workspace_bytes(B, H, total, max_seqlen, d, q.dtype)
            workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
        rc = lib.fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                               lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               cu_seqlens.data_ptr(), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), B, H, total, max_seqlen,
                               d, scale, FA_CAUSAL if causal else 0, _dtype_code(q),
                               _stream_ptr(q.device))
    _raise(rc, "fa_bwd_varlen")
    return dq, dk, dv


def fa_softmax_rows(x, scale: float = 1.0, out=None):
    """Row softmax of a CUDA tensor (last dimension = row), fp32 or bf16; returns ``out``."""
    lib = load_library()
    _check(x, "x")
    cols = x.shape[-1]
    rows = x.numel() // max(cols, 1)
    y = torch.empty_like(x) if out is None else out
    _check(y, "out", x)
    with torch.cuda.device(x.device):
        rc = lib.fa_softmax_rows(x.data_ptr(), y.data_ptr(), rows, cols, float(scale),
                                 _dtype_code(x), _stream_ptr(x.device))
    _raise(rc, "fa_softmax_rows")
    return y


def fa_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, dtype=torch.bfloat16) -> int:
    """Scratch bytes fa_decode needs on the current device."""
    code = FA_BF16 if dtype == torch.bfloat16 else FA_F32
    return int(load_library().fa_decode_workspace_bytes(B, H, Nq, Nk, d, code))


def fa_decode_plan(B: int, H: int, Nq: int, Nk: int, d: int, resident_ctas: int = 0):
    """(splits, keys_per_split) that fa_decode uses; resident_ctas > 0 plans without a device."""
    s, k = ctypes.c_int(0), ctypes.c_int(0)
    _raise(load_library().fa_decode_plan(B, H, Nq, Nk, d, int(resident_ctas), ctypes.byref(s),
                                         ctypes.byref(k)), "fa_decode_plan")
    return s.value, k.value


def fa_decode(q, k, v, scale: float | None = None, out=None, lse=None, workspace=None):
    """KV-cache decode: q [B,H,Nq,d] (Nq <= 16) against k, v [B,H,Nk,d], bf16.

    Returns (O like q, LSE [B,H,Nq] float32).
    """
    lib = load_library()
    _check(q, "q")
    _check(k, "k")
    _check(v, "v", k)
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B,H,Nq,d] and k, v [B,H,Nk,d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k, v must be [B,H,Nk,d] with q's B, H, d, dtype and device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "out", q)
    if lse.dtype != torch.float32 or lse.shape != (B, H, Nq) or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be contiguous float32 [B,H,Nq] on the same device")
    with torch.cuda.device(q.device):
        if workspace is None:
            ws_bytes = fa_decode_workspace_bytes(B, H, Nq, Nk, d, q.dtype)
            workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
        rc = lib.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           B, H, Nq, Nk, d, scale, _dtype_code(q), _stream_ptr(q.device))
    _raise(rc, "fa_decode")
    return o, lse


def fa_check_device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().fa_check_device_status(_stream_ptr(dev)))


def fa_debug_timeout_probe(limit_ns: int, device=None) -> int:
    """Launch the bounded-wait probe kernel (see include/fa.h); returns the launch status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().fa_debug_timeout_probe(int(limit_ns), _stream_ptr(dev)))
