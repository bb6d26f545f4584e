"""Exact tiled attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/fa_gb300.h`` (library
``_lib/libfa_gb300.so``, built by ``build.build()``).  Each function here has
the name of the C entry point it calls and only marshals arguments: shape,
dtype and device checks, output allocation through PyTorch when the caller
passes none, the current CUDA stream, and the status code.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path.
If the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# The library the binding loads: the built one, or another build of the same
# C ABI named by FA_GB300_LIBRARY (the bounds-checked debug build,
# _lib/libfa_gb300_debug.so).
LIB_PATH = os.environ.get("FA_GB300_LIBRARY") or os.path.join(_HERE, "_lib", "libfa_gb300.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_lib", "libfa_gb300_debug.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED_ARCH = -2
FA_ERR_LAUNCH = -3
FA_ERR_DEVICE_TIMEOUT = -4
FA_ERR_DEVICE_BOUNDS = -5
FA_ERR_DRIVER = -6
FA_ERR_CUDA = -7
FA_ERR_SCRATCH_CAPACITY = -8
FA_DTYPE_BF16 = 0
FA_DTYPE_F32 = 1

# Every symbol the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_f32": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_fwd_window": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "fa_row_stats": (_I, [_P, _I, _I, _I, _F, _P, _P, _P, _P]),
    "fa_prefix_attention": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P]),
    "fa_prefix_attention_chunked": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P,
                                         _P, _P, _P]),
    "fa_row_stats_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "fa_row_stats_partials": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "fa_row_stats_combine": (_I, [_P, _P, _P, _I, _I, _F, _P, _P, _P, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I,
                           _P]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F,
                           _I, _P]),
    "fa_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "fa_combine_states": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "fa_decode_paged_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                     _P, _P, _P, _P]),
    "fa_decode_splitkv_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _I, _P,
                                       _P]),
    "fa_fwd_fault_inject": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _I, _P]),
    "fa_check_device_status": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_cuda_error": (_I, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fa_status_string(code)} (code {code})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing "
                "(run exact_io_aware_15_gb300.build.build())")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def fa_status_string(code: int) -> str:
    try:
        return load_library().fa_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def _check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FAError(code, where)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _out(t, name, dtype, shape, device):
    """A caller-supplied output buffer, checked (dtype, contiguity, exact
    shape, device), or a new one from torch when t is None.  The kernels write
    every element of the shape they are given, so a smaller buffer would be
    written past its end."""
    shape = tuple(int(x) for x in shape)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _need(t, name, dtype, len(shape))
    if tuple(t.shape) != shape:
        raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    return t


def _workspace(ws, nbytes, device):
    """The caller's fp32 workspace (checked to hold nbytes) or a new one."""
    if ws is None:
        return torch.empty(max(1, (int(nbytes) + 3) // 4), dtype=torch.float32, device=device)
    _need(ws, "workspace", torch.float32, 1)
    if ws.numel() * 4 < nbytes:
        raise ValueError(f"workspace holds {ws.numel() * 4} bytes, needs {nbytes}")
    if ws.device != device:
        raise ValueError(f"workspace must be on {device}")
    return ws


def _same_device(*named):
    """Every tensor on the device of the first one."""
    dev = named[0][0].device
    for t, n in named[1:]:
        if t is not None and t.device != dev:
            raise ValueError(f"{n} is on {t.device}, expected {dev}")


def _scale(scale, D):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


_DT = {torch.bfloat16: FA_DTYPE_BF16, torch.float32: FA_DTYPE_F32}


def fa_fwd_ex(q, k, v, scale=None, causal=False, o_dtype=None, o=None, lse=None):
    """Dense forward.  q, k, v: [B, H, N, D] bf16 (tensor cores) or fp32
    (FFMA kernel).  Returns (o [B, H, N, D] in o_dtype, lse [B, H, N] fp32)."""
    in_dtype = q.dtype
    if in_dtype not in _DT:
        raise TypeError("q, k, v must be bf16 or fp32")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, in_dtype, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    B, H, N, D = q.shape
    o_dtype = in_dtype if o_dtype is None else o_dtype
    if o_dtype not in _DT:
        raise TypeError("o_dtype must be bf16 or fp32")
    _same_device((q, "q"), (k, "k"), (v, "v"))
    o = _out(o, "o", o_dtype, (B, H, N, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H, N), q.device)
    rc = load_library().fa_fwd_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
        _scale(scale, D), int(bool(causal)), _DT[in_dtype], _DT[o_dtype],
        _stream(q))
    _check(rc, "fa_fwd_ex")
    return o, lse


def fa_fwd(q, k, v, scale=None, causal=False, o=None, lse=None):
    """Dense bf16 forward on the tensor cores (fa_fwd)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    B, H, N, D = q.shape
    _same_device((q, "q"), (k, "k"), (v, "v"))
    o = _out(o, "o", torch.bfloat16, (B, H, N, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H, N), q.device)
    rc = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                               B, H, N, D, _scale(scale, D), int(bool(causal)),
                               _stream(q))
    _check(rc, "fa_fwd")
    return o, lse


def fa_fwd_window(q, k, v, window, scale=None, o=None, lse=None):
    """Causal sliding-window forward (bf16): query i sees keys i-window+1 .. i."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    B, H, N, D = q.shape
    _same_device((q, "q"), (k, "k"), (v, "v"))
    o = _out(o, "o", torch.bfloat16, (B, H, N, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H, N), q.device)
    rc = load_library().fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      B, H, N, D, _scale(scale, D), int(window), _stream(q))
    _check(rc, "fa_fwd_window")
    return o, lse


def fa_bwd(q, k, v, o, do, lse, scale=None, causal=False, dq=None, dk=None, dv=None,
           workspace=None):
    """Backward of the dense bf16 forward by recomputation (fa_bwd): returns
    dq, dk, dv (bf16) given the forward's o and lse and the output gradient do."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, n, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q [B, H, N, D]")
    B, H, N, D = q.shape
    _need(lse, "lse", torch.float32, 3)
    if tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be [B, H, N]")
    _same_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (lse, "lse"))
    dq, dk, dv = (_out(t, n, torch.bfloat16, (B, H, N, D), q.device)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    lib = load_library()
    workspace = _workspace(workspace, lib.fa_bwd_workspace_bytes(B, H, N), q.device)
    rc = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                    _ptr(dk), _ptr(dv), _ptr(workspace), B, H, N, D, _scale(scale, D),
                    int(bool(causal)), _stream(q))
    _check(rc, "fa_bwd")
    return dq, dk, dv


def fa_prefix_attention(q, k_cache, v_cache, cu_seqlens_k, scale=None, o=None, lse=None):
    """Attention of q[b, h] over every prefix of sequence b's keys
    (fa_prefix_attention).  q [B, H, D]; caches packed [T, H, D] bf16;
    cu_seqlens_k int32 [B + 1] on the device.  Returns o [T, H, D] bf16 and
    lse [H, T] fp32."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 3)
    _need(v_cache, "v_cache", torch.bfloat16, 3)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    B, H, D = q.shape
    T = k_cache.shape[0]
    if k_cache.shape[1:] != (H, D) or cu_seqlens_k.numel() != B + 1:
        raise ValueError("shapes: q [B, H, D], caches [T, H, D], cu_seqlens_k [B + 1]")
    _same_device((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (cu_seqlens_k, "cu_seqlens_k"))
    o = _out(o, "o", torch.bfloat16, (T, H, D), q.device)
    lse = _out(lse, "lse", torch.float32, (H, T), q.device)
    rc = load_library().fa_prefix_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(cu_seqlens_k), T, B, H, D, _scale(scale, D),
                                            _ptr(o), _ptr(lse), _stream(q))
    _check(rc, "fa_prefix_attention")
    return o, lse


def fa_prefix_attention_chunked(q, k_cache, v_cache, cu_seqlens_k, num_splits, scale=None,
                                o=None, lse=None):
    """Prefix attention with every row cut into num_splits chunks scanned at
    once (fa_prefix_attention_chunked); the chunks' split-KV states go to a
    workspace allocated here.  Returns o [T, H, D] bf16 and lse [H, T]."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 3)
    _need(v_cache, "v_cache", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    B, H, D = q.shape
    T = k_cache.shape[0]
    if k_cache.shape[1:] != (H, D) or v_cache.shape != k_cache.shape or \
            cu_seqlens_k.numel() != B + 1:
        raise ValueError("shapes: q [B, H, D], caches [T, H, D], cu_seqlens_k [B + 1]")
    _same_device((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (cu_seqlens_k, "cu_seqlens_k"))
    S = int(num_splits)
    parts = [torch.empty(s, dtype=torch.float32, device=q.device)
             for s in ((B, H, S), (B, H, S), (B, H, S, D))]
    o = _out(o, "o", torch.bfloat16, (T, H, D), q.device)
    lse = _out(lse, "lse", torch.float32, (H, T), q.device)
    rc = load_library().fa_prefix_attention_chunked(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_k), T, B, H, D, S,
        _scale(scale, D), *(_ptr(p) for p in parts), _ptr(o), _ptr(lse), _stream(q))
    _check(rc, "fa_prefix_attention_chunked")
    return o, lse


def _rows_dtype(x):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [R, C] matrix")
    if x.dtype not in _DT:
        raise TypeError(f"x must be bf16 or fp32, got {x.dtype}")
    return _DT[x.dtype]


def fa_row_stats(x, eps=0.0, mean=None, var=None, rstd=None):
    """Per-row mean, population variance and 1/sqrt(var + eps) of a [R, C]
    bf16 or fp32 matrix (fa_row_stats): Welford states, one pass."""
    dt = _rows_dtype(x)
    R, C = x.shape
    mean, var, rstd = (_out(t, n, torch.float32, (R,), x.device)
                       for t, n in ((mean, "mean"), (var, "var"), (rstd, "rstd")))
    rc = load_library().fa_row_stats(_ptr(x), R, C, dt, float(eps), _ptr(mean), _ptr(var),
                                     _ptr(rstd), _stream(x))
    _check(rc, "fa_row_stats")
    return mean, var, rstd


def fa_row_stats_partials(x, num_splits):
    """Split-K first pass: chunk states (n, mu, M2), each [R, num_splits]."""
    dt = _rows_dtype(x)
    R, C = x.shape
    parts = [torch.empty((R, num_splits), dtype=torch.float32, device=x.device)
             for _ in range(3)]
    rc = load_library().fa_row_stats_partials(_ptr(x), R, C, dt, int(num_splits),
                                              *(_ptr(p) for p in parts), _stream(x))
    _check(rc, "fa_row_stats_partials")
    return tuple(parts)


def fa_row_stats_combine(part_n, part_mu, part_m2, eps=0.0):
    """Split-K second pass: fixed-order fold of each row's chunk states."""
    for t, n in ((part_n, "part_n"), (part_mu, "part_mu"), (part_m2, "part_m2")):
        _need(t, n, torch.float32, 2)
        if t.shape != part_n.shape:
            raise ValueError("chunk state arrays must have the same shape")
    R, S = part_n.shape
    out = [torch.empty(R, dtype=torch.float32, device=part_n.device) for _ in range(3)]
    rc = load_library().fa_row_stats_combine(_ptr(part_n), _ptr(part_mu), _ptr(part_m2), R, S,
                                             float(eps), *(_ptr(o) for o in out),
                                             _stream(part_n))
    _check(rc, "fa_row_stats_combine")
    return tuple(out)


def fa_bwd_window(q, k, v, o, do, lse, window, scale=None, dq=None, dk=None, dv=None,
                  workspace=None):
    """Backward of the causal sliding-window forward (fa_bwd_window): query i
    sees keys i-window+1 .. i.  Same layouts as fa_bwd."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, n, torch.bfloat16, 4)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q [B, H, N, D]")
    B, H, N, D = q.shape
    _need(lse, "lse", torch.float32, 3)
    if tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be [B, H, N]")
    _same_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (lse, "lse"))
    dq, dk, dv = (_out(t, n, torch.bfloat16, (B, H, N, D), q.device)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    workspace = _workspace(workspace, load_library().fa_bwd_workspace_bytes(B, H, N), q.device)
    rc = load_library().fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), B, H, N, D,
                                      _scale(scale, D), int(window), _stream(q))
    _check(rc, "fa_bwd_window")
    return dq, dk, dv


def fa_bwd_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen, scale=None, causal=True,
                  dq=None, dk=None, dv=None, workspace=None):
    """Backward over packed sequences (fa_bwd_varlen): q, k, v, o, do
    [T, H, D] bf16, lse [H, T] fp32 from fa_fwd_varlen, cu_seqlens int32
    [num_seqs + 1] on the device.  Returns dq, dk, dv [T, H, D] bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, n, torch.bfloat16, 3)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q [T, H, D]")
    T, H, D = q.shape
    _need(lse, "lse", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if tuple(lse.shape) != (H, T):
        raise ValueError("lse must be [H, T]")
    _same_device((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do"), (lse, "lse"),
                 (cu_seqlens, "cu_seqlens"))
    dq, dk, dv = (_out(t, n, torch.bfloat16, (T, H, D), q.device)
                  for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")))
    workspace = _workspace(workspace, load_library().fa_bwd_workspace_bytes(1, H, T), q.device)
    rc = load_library().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), H, D,
        _scale(scale, D), int(bool(causal)), _stream(q))
    _check(rc, "fa_bwd_varlen")
    return dq, dk, dv


def fa_fwd_f32(q, k, v, scale=None, causal=False, o=None, lse=None):
    """Dense fp32 forward on the CUDA cores (fa_fwd_f32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.float32, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    B, H, N, D = q.shape
    _same_device((q, "q"), (k, "k"), (v, "v"))
    o = _out(o, "o", torch.float32, (B, H, N, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H, N), q.device)
    rc = load_library().fa_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                   B, H, N, D, _scale(scale, D), int(bool(causal)),
                                   _stream(q))
    _check(rc, "fa_fwd_f32")
    return o, lse


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, scale=None, causal=True,
                  o=None, lse=None):
    """Packed variable-length forward.  q, k, v: [T, H, D] bf16; cu_seqlens:
    int32 [num_seqs + 1] on the same device.  Returns (o [T, H, D] bf16,
    lse [H, T] fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 3)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [T, H, D]")
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, H, D = q.shape
    _same_device((q, "q"), (k, "k"), (v, "v"), (cu_seqlens, "cu_seqlens"))
    o = _out(o, "o", torch.bfloat16, (T, H, D), q.device)
    lse = _out(lse, "lse", torch.float32, (H, T), q.device)
    rc = load_library().fa_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, T, int(max_seqlen), H, D, _scale(scale, D),
        int(bool(causal)), _stream(q))
    _check(rc, "fa_fwd_varlen")
    return o, lse


def fa_decode_workspace_bytes(B: int, H: int, D: int, num_splits: int) -> int:
    return int(load_library().fa_decode_workspace_bytes(B, H, D, num_splits))


def fa_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, N))


def fa_row_stats_workspace_bytes(R: int, num_splits: int) -> int:
    return int(load_library().fa_row_stats_workspace_bytes(R, num_splits))


def fa_decode_splitkv(q, k_cache, v_cache, cu_seqlens_k, num_splits, scale=None,
                      part_m=None, part_d=None, part_o=None):
    """Split-KV first pass.  q [B, H, D] bf16; caches [T_k, H, D] bf16;
    cu_seqlens_k int32 [B + 1] on the device.  Returns the base-2 chunk states
    (part_m [B, H, S], part_d [B, H, S], part_o [B, H, S, D]) in fp32."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 3)
    _need(v_cache, "v_cache", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    B, H, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[1:] != (H, D):
        raise ValueError("caches must be [T_k, H, D] like q's heads and head dim")
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_k must have B + 1 entries")
    S = int(num_splits)
    dev = q.device
    _same_device((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (cu_seqlens_k, "cu_seqlens_k"))
    part_m = _out(part_m, "part_m", torch.float32, (B, H, S), dev)
    part_d = _out(part_d, "part_d", torch.float32, (B, H, S), dev)
    part_o = _out(part_o, "part_o", torch.float32, (B, H, S, D), dev)
    rc = load_library().fa_decode_splitkv(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_k), k_cache.shape[0],
        B, H, D, S, _scale(scale, D), _ptr(part_m), _ptr(part_d), _ptr(part_o),
        _stream(q))
    _check(rc, "fa_decode_splitkv")
    return part_m, part_d, part_o


def fa_decode_paged_splitkv(q, k_pages, v_pages, block_table, seqlens, num_splits,
                            scale=None, part_m=None, part_d=None, part_o=None):
    """Split-KV first pass over a paged cache with grouped query heads.
    q [B, H, D] bf16; pages [P, page_size, H_kv, D] bf16; block_table int32
    [B, max_blocks] and seqlens int32 [B] on the device.  Returns the base-2
    chunk states (part_m, part_d [B, H, S], part_o [B, H, S, D])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, H, D = q.shape
    P, page, Hkv, Dk = k_pages.shape
    if v_pages.shape != k_pages.shape or Dk != D:
        raise ValueError("pages must be [P, page_size, H_kv, D] like q's head dim")
    if block_table.shape[0] != B or seqlens.numel() != B:
        raise ValueError("block_table and seqlens need one row per sequence")
    S = int(num_splits)
    dev = q.device
    _same_device((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"),
                 (block_table, "block_table"), (seqlens, "seqlens"))
    part_m = _out(part_m, "part_m", torch.float32, (B, H, S), dev)
    part_d = _out(part_d, "part_d", torch.float32, (B, H, S), dev)
    part_o = _out(part_o, "part_o", torch.float32, (B, H, S, D), dev)
    rc = load_library().fa_decode_paged_splitkv(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens), P, page,
        block_table.shape[1], B, H, Hkv, D, S, _scale(scale, D), _ptr(part_m), _ptr(part_d),
        _ptr(part_o), _stream(q))
    _check(rc, "fa_decode_paged_splitkv")
    return part_m, part_d, part_o


def fa_combine_states(part_m, part_d, part_o, o_dtype=torch.bfloat16, o=None, lse=None):
    """Split-KV second pass over states [..., S] / [..., S, D] (fp32).
    Returns (o [..., D] in o_dtype, lse [...] fp32)."""
    for t, n in ((part_m, "part_m"), (part_d, "part_d"), (part_o, "part_o")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor")
    lead = tuple(part_m.shape[:-1])
    S = part_m.shape[-1]
    D = part_o.shape[-1]
    if tuple(part_d.shape) != lead + (S,) or tuple(part_o.shape) != lead + (S, D):
        raise ValueError("state shapes do not match")
    rows = 1
    for x in lead:
        rows *= x
    if o_dtype not in _DT:
        raise TypeError("o_dtype must be bf16 or fp32")
    _same_device((part_o, "part_o"), (part_m, "part_m"), (part_d, "part_d"))
    o = _out(o, "o", o_dtype, lead + (D,), part_o.device)
    lse = _out(lse, "lse", torch.float32, lead, part_o.device)
    rc = load_library().fa_combine_states(
        _ptr(part_m), _ptr(part_d), _ptr(part_o), rows, S, D, _ptr(o), _DT[o_dtype],
        _ptr(lse), _stream(part_o))
    _check(rc, "fa_combine_states")
    return o, lse


def fa_decode_splitkv_noalloc(q, k_cache, v_cache, cu_seqlens_k, num_splits, scale=None,
                              o_dtype=torch.bfloat16, o=None, lse=None):
    """Split-KV decode, both passes, for callers that may not allocate device
    memory: the partial states go to the library's static 32 MiB device array
    instead of a workspace (the outputs still come from the caller, or from
    torch here when not given).  Returns (o [B, H, D], lse [B, H])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 3)
    _need(v_cache, "v_cache", torch.bfloat16, 3)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    B, H, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[1:] != (H, D):
        raise ValueError("caches must be [T_k, H, D] like q's heads and head dim")
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_k must have B + 1 entries")
    if o_dtype not in _DT:
        raise TypeError("o_dtype must be bf16 or fp32")
    _same_device((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (cu_seqlens_k, "cu_seqlens_k"))
    o = _out(o, "o", o_dtype, (B, H, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H), q.device)
    rc = load_library().fa_decode_splitkv_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_k), k_cache.shape[0],
        B, H, D, int(num_splits), _scale(scale, D), _ptr(o), _DT[o_dtype], _ptr(lse),
        _stream(q))
    _check(rc, "fa_decode_splitkv_noalloc")
    return o, lse


def fa_fwd_fault_inject(q, k, v, skip_k_tile, wait_limit_us, scale=None, causal=False,
                        o=None, lse=None):
    """Test hook of the failure path (fa_fwd_fault_inject): fa_fwd with key
    tile skip_k_tile never loaded and every device wait limited to
    wait_limit_us; the timeout shows up in fa_check_device_status."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, H, N, D]")
    B, H, N, D = q.shape
    _same_device((q, "q"), (k, "k"), (v, "v"))
    o = _out(o, "o", torch.bfloat16, (B, H, N, D), q.device)
    lse = _out(lse, "lse", torch.float32, (B, H, N), q.device)
    rc = load_library().fa_fwd_fault_inject(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, _scale(scale, D),
        int(bool(causal)), int(skip_k_tile), int(wait_limit_us), _stream(q))
    _check(rc, "fa_fwd_fault_inject")
    return o, lse


def fa_check_device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronises the stream and returns (and clears) the device status:
    FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_DEVICE_BOUNDS."""
    s = torch.cuda.current_stream() if stream is None else stream
    return int(load_library().fa_check_device_status(s.cuda_stream))


def decode(q, k_cache, v_cache, cu_seqlens_k, num_splits=16, scale=None,
           o_dtype=torch.bfloat16):
    """Split-KV decode end to end: fa_decode_splitkv then fa_combine_states."""
    pm, pd, po = fa_decode_splitkv(q, k_cache, v_cache, cu_seqlens_k, num_splits, scale)
    return fa_combine_states(pm, pd, po, o_dtype=o_dtype)


__all__ = [
    "fa_fwd", "fa_fwd_f32", "fa_fwd_ex", "fa_fwd_window", "fa_fwd_varlen", "fa_bwd",
    "fa_bwd_varlen", "fa_bwd_window",
    "fa_bwd_workspace_bytes", "fa_decode_workspace_bytes", "fa_row_stats",
    "fa_row_stats_workspace_bytes", "fa_row_stats_partials", "fa_row_stats_combine",
    "fa_prefix_attention", "fa_prefix_attention_chunked",
    "fa_decode_splitkv", "fa_combine_states", "fa_decode_splitkv_noalloc",
    "fa_decode_paged_splitkv",
    "fa_check_device_status", "fa_fwd_fault_inject",
    "fa_status_string", "decode", "load_library", "FAError", "LIB_PATH", "DEBUG_LIB_PATH",
]
