"""ctypes binding of libfa_gb300.so (include/fa.h).

Argument marshalling only: torch tensors are checked for dtype, device and
layout, and their data pointers are handed to the C entry points, which run
every step on the GPU.  There is no fallback: if the library is missing or a
call fails, a ``FaError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_F16, FA_BF16 = 0, 1
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_WORKSPACE = range(6)

# Symbols include/fa.h declares, with their ctypes signatures.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_qk": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp,
                            _sz, _vp]),
    "fa_fwd_splitkv_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "fa_bwd_qk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                       _i, _i, _vp, _sz, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd_workspace_size_for": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i,
                    _vp, _sz, _vp]),
    "fa_bwd_deterministic": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                  _i, _f, _i, _vp, _sz, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f,
                            _i, _vp]),
    "fa_fwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                                _i, _vp]),
    "fa_bwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                _i, _f, _i, _vp, _i, _i, _vp, _sz, _vp]),
    "fa_fwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_bwd_strided": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                            _f, _i, _vp, _i, _vp, _sz, _vp]),
    "fa_get_device_status": (_i, [_vp]),
    "fa_strerror": (ctypes.c_char_p, [_i]),
    "fa_selftest_expired_wait": (_i, [_i, _vp]),
    "fa_measure_ex2_rate": (_i, [ctypes.POINTER(ctypes.c_double), _vp]),
    "fa_measure_reduce_rate": (_i, [_vp, _sz, ctypes.POINTER(ctypes.c_double), _vp]),
    "fa_timing_enable": (_i, [_i]),
    "fa_timing_read": (_i, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
}
KERNEL_KINDS = ("fwd", "bwd_pre", "bwd_main", "bwd_convert", "bwd_dq")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed with status {status}: {strerror(status)}")


def load(path: str = LIB_PATH):
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise FaError(-1, f"loading {path}: library not built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def strerror(status: int) -> str:
    try:
        return load().fa_strerror(status).decode()
    except Exception:
        return "library not loaded"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FA_F16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; fp16 and bf16 are supported")


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _check(st: int, what: str):
    if st != FA_OK:
        raise FaError(st, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


# ---------------------------------------------------------------- raw entry points
def fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, dtype, stream=None) -> int:
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                         int(causal), float(scale), dtype, _stream_ptr(stream))


def fa_bwd_workspace_size(B, H, Hkv, N, d) -> int:
    return int(load().fa_bwd_workspace_size(B, H, Hkv, N, d))


def fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, deterministic) -> int:
    return int(load().fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, int(bool(deterministic))))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, causal, scale, dtype, workspace,
           workspace_bytes, stream=None) -> int:
    return load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, Hkv, N, d, int(causal), float(scale), dtype,
                         _ptr(workspace), int(workspace_bytes), _stream_ptr(stream))


def fa_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, causal, scale, dtype,
                         workspace, workspace_bytes, stream=None) -> int:
    return load().fa_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                       _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d, int(causal),
                                       float(scale), dtype, _ptr(workspace), int(workspace_bytes),
                                       _stream_ptr(stream))


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, causal, scale, dtype,
                   stream=None) -> int:
    """fa_bwd with the library's own fixed device scratch (no allocation)."""
    return load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d, int(causal),
                                 float(scale), dtype, _stream_ptr(stream))


def fa_get_device_status(stream=None) -> int:
    return load().fa_get_device_status(_stream_ptr(stream))


# ---------------------------------------------------------------- tensor helpers
class FaStrides(ctypes.Structure):
    """struct fa_strides: element strides (batch, head, row) of a [B][heads][N][d] view."""
    _fields_ = [("batch", ctypes.c_longlong), ("head", ctypes.c_longlong),
                ("row", ctypes.c_longlong)]


def _shapes(q, k, v, contiguous=True):
    """(B, H, Hkv, Nq, Nk, d) of q [B,H,Nq,d], k and v [B,Hkv,Nk,d] (views with
    the last dimension contiguous are accepted when contiguous=False)."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,H,Nq,d], k and v [B,Hkv,Nk,d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)}")
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != q.dtype:
            raise ValueError("q, k, v must be CUDA tensors of one dtype")
        if contiguous and not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
        if not contiguous and t.stride(3) != 1:
            raise ValueError("the last (d) dimension must be contiguous")
    return B, H, k.shape[1], Nq, k.shape[2], d


def _strides(*ts):
    """fa_strides[len(ts)] of [B, heads, N, d] views (d contiguous)."""
    arr = (FaStrides * len(ts))()
    for i, t in enumerate(ts):
        if t.dim() != 4 or t.stride(3) != 1:
            raise ValueError("expected a [B, heads, N, d] view with d contiguous")
        arr[i] = FaStrides(t.stride(0), t.stride(1), t.stride(2))
    return arr


def forward_strided(q, k, v, causal: bool, scale: float, out=None, lse=None, stream=None):
    """fa_fwd_strided: q [B,H,Nq,d], k, v [B,Hkv,Nk,d] given as any views whose
    d elements are contiguous (e.g. x.transpose(1, 2) of a [B, N, H, d]
    tensor); out (allocated like q's layout unless given) likewise.  Returns
    (o, lse)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v, contiguous=False)
    if out is None:
        out = torch.empty_like(q)   # same strides as q when q is dense in memory
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check(load().fa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, Nq,
                                 Nk, d, int(causal), float(scale), _dtype_code(q),
                                 _strides(q, k, v, out), _stream_ptr(stream)), "fa_fwd_strided")
    return out, lse


def backward_strided(q, k, v, o, lse, dout, causal: bool, scale: float, dq=None, dk=None,
                     dv=None, workspace=None, stream=None, deterministic: bool = False):
    """fa_bwd_strided: the gradients of forward_strided; every tensor may be a
    strided view (d contiguous); dq, dk, dv are allocated like q, k, v unless
    given.  Returns (dq, dk, dv)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v, contiguous=False)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(load().fa_bwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, Nq, Nk, d, int(causal),
                                 float(scale), _dtype_code(q),
                                 _strides(q, k, v, o, dout, dq, dk, dv), int(bool(deterministic)),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "fa_bwd_strided")
    return dq, dk, dv


def forward(q, k, v, causal: bool, scale: float, out=None, lse=None, stream=None):
    """(o, lse) of exact attention; outputs are allocated unless given.  The
    key length may differ from the query length (causal mask bottom-right)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if Nq == Nk:
        st = fa_fwd(q, k, v, out, lse, B, H, Hkv, Nq, d, causal, scale, _dtype_code(q), stream)
    else:
        st = load().fa_fwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, Nq, Nk,
                              d, int(causal), float(scale), _dtype_code(q), _stream_ptr(stream))
    _check(st, "fa_fwd")
    return out, lse


def backward(q, k, v, o, lse, dout, causal: bool, scale: float, dq=None, dk=None, dv=None,
             workspace=None, stream=None, deterministic: bool = False):
    """(dq, dk, dv) of sum(O o dO); outputs and scratch are allocated unless given.
    deterministic=True uses fa_bwd_deterministic (bitwise reproducible dQ)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if Nq == Nk:
        fn = fa_bwd_deterministic if deterministic else fa_bwd
        st = fn(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, d, causal, scale,
                _dtype_code(q), workspace, ws_bytes, stream)
    else:
        st = load().fa_bwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, H, Hkv, Nq, Nk, d, int(causal), float(scale),
                              _dtype_code(q), int(bool(deterministic)), _ptr(workspace),
                              ws_bytes, _stream_ptr(stream))
    _check(st, "fa_bwd_deterministic" if deterministic else "fa_bwd")
    return dq, dk, dv


def device_status(stream=None):
    """Synchronise the stream and raise if a kernel reported a bounded-wait timeout."""
    _check(fa_get_device_status(stream), "fa_get_device_status")


def measure_ex2_rate(stream=None) -> float:
    """Exponentials per second of the device's ex2 unit (fa_measure_ex2_rate)."""
    out = ctypes.c_double(0.0)
    _check(load().fa_measure_ex2_rate(ctypes.byref(out), _stream_ptr(stream)),
           "fa_measure_ex2_rate")
    return out.value


def measure_reduce_rate(scratch: torch.Tensor, stream=None) -> float:
    """Bytes per second of fp32 bulk reduce-adds from every SM into `scratch`
    (a device tensor of at least 1 MiB, 256-byte aligned; zeros are added:
    fa_measure_reduce_rate)."""
    out = ctypes.c_double(0.0)
    _check(load().fa_measure_reduce_rate(ctypes.c_void_p(scratch.data_ptr()),
                                         scratch.numel() * scratch.element_size(),
                                         ctypes.byref(out), _stream_ptr(stream)),
           "fa_measure_reduce_rate")
    return out.value


def timing_enable(capacity: int):
    """Start (capacity > 0) or stop (0) per-kernel event timing inside the library."""
    _check(load().fa_timing_enable(int(capacity)), "fa_timing_enable")


def timing_read():
    """{kind: (summed ms, launches)} of the kernels timed since the last read."""
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    n = (ctypes.c_int * len(KERNEL_KINDS))()
    _check(load().fa_timing_read(ms, n), "fa_timing_read")
    return {k: (ms[i], n[i]) for i, k in enumerate(KERNEL_KINDS)}


def forward_splitkv(q, k, v, causal: bool, scale: float, num_splits: int = 0, out=None, lse=None,
                    workspace=None, stream=None):
    """(o, lse) through fa_fwd_splitkv (key axis split, partials merged on the GPU)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = int(load().fa_fwd_splitkv_workspace_size(B, H, Hkv, Nq, Nk, d, int(num_splits)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(load().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, Nq,
                                 Nk, d, int(causal), float(scale), _dtype_code(q), int(num_splits),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "fa_fwd_splitkv")
    return out, lse


def _check_mask(block_mask, H, Nq, Nk, device):
    """A block mask [1 or H, ceil(Nq/128), ceil(Nk/128)] as a contiguous uint8
    CUDA tensor (nonzero = computed); returns (mask, mask_heads)."""
    nbr, nbc = -(-Nq // 128), -(-Nk // 128)
    if (block_mask.dim() != 3 or block_mask.shape[0] not in (1, H)
            or tuple(block_mask.shape[1:]) != (nbr, nbc)):
        raise ValueError(f"block mask must be [1 or {H}, {nbr}, {nbc}], got "
                         f"{tuple(block_mask.shape)}")
    if block_mask.dtype not in (torch.uint8, torch.bool):
        raise TypeError("block mask must be uint8 or bool")
    if not block_mask.is_cuda or block_mask.device != device or not block_mask.is_contiguous():
        raise ValueError("block mask must be a contiguous tensor on the inputs' device")
    return block_mask, int(block_mask.shape[0])


def forward_blocksparse(q, k, v, block_mask, causal: bool, scale: float, out=None, lse=None,
                        stream=None):
    """(o, lse) of exact attention restricted to the kept 128 x 128 blocks of
    block_mask [1 or H, ceil(Nq/128), ceil(Nk/128)] (fa_fwd_blocksparse)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v)
    mask, mh = _check_mask(block_mask, H, Nq, Nk, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check(load().fa_fwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv,
                                     Nq, Nk, d, int(causal), float(scale), _dtype_code(q),
                                     _ptr(mask), mh, _stream_ptr(stream)), "fa_fwd_blocksparse")
    return out, lse


def backward_blocksparse(q, k, v, o, lse, dout, block_mask, causal: bool, scale: float, dq=None,
                         dk=None, dv=None, workspace=None, stream=None,
                         deterministic: bool = False):
    """(dq, dk, dv) of the block-sparse forward above (fa_bwd_blocksparse)."""
    B, H, Hkv, Nq, Nk, d = _shapes(q, k, v)
    mask, mh = _check_mask(block_mask, H, Nq, Nk, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(load().fa_bwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, Nq, Nk, d,
                                     int(causal), float(scale), _dtype_code(q), _ptr(mask), mh,
                                     int(bool(deterministic)), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _stream_ptr(stream)), "fa_bwd_blocksparse")
    return dq, dk, dv
