"""fp64 CPU oracle for exact softmax attention (forward and analytic backward).

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU
baseline leg of ``bench.py`` use this package; the product library never
imports or calls it, and it imports nothing from the product package.

The arithmetic lives in ``attention_oracle.c`` (plain C, fp64, OpenMP over
rows); this module builds it with gcc and marshals numpy arrays through
ctypes.  Every entry point takes fp64 arrays in the [B, H, N, d] layout
(keys/values [B, Hkv, N, d]) and returns fp64 results.

What is computed, and where each step comes from on the pages, is stated in
the C file's header: O = softmax(scale * Q K^T [+ causal mask]) V, the row
logsumexp L = m + ln(l) ("FlashAttention-2: Faster Attention with Better
Parallelism and Work Partitioning", paper digest, section 3 "Target
operation" and the section 4 notation table) and the five-product gradient
with D = rowsum(dO o O) (same digest, section 3 "FLOPs" and section 4).

Every function here is pinned by the CPU tests in ``tests/test_oracle_*.py``
(closed forms, invariants, finite differences and fp64 library routines).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C file into a shared library with gcc (+OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its C signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or build()
    lib = ctypes.CDLL(p)
    lib.oracle_fwd_group.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                     ctypes.c_long, ctypes.c_int, ctypes.c_double, _dp, _dp]
    lib.oracle_fwd_group.restype = None
    lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                    ctypes.c_long, ctypes.c_int, ctypes.c_double, ctypes.c_long,
                                    _lp, _dp, _dp]
    lib.oracle_fwd_rows.restype = None
    lib.oracle_bwd_group.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                     ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                     _dp, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_bwd_group.restype = None
    lib.oracle_bwd_rows.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                    ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                    ctypes.c_long, ctypes.c_long, _dp, _dp, _dp]
    lib.oracle_bwd_rows.restype = None
    _bp = ctypes.POINTER(ctypes.c_ubyte)
    lib.oracle_fwd_group_blockmask.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                               ctypes.c_long, ctypes.c_long, ctypes.c_int, _bp,
                                               ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                               ctypes.c_double, _dp, _dp]
    lib.oracle_fwd_group_blockmask.restype = None
    lib.oracle_bwd_group_blockmask.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                               ctypes.c_long, ctypes.c_long, ctypes.c_int, _bp,
                                               ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                               ctypes.c_double, _dp, _dp, _dp]
    lib.oracle_bwd_group_blockmask.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _f64(a) -> np.ndarray:
    """Widen any array-like (numpy or CPU torch tensor, any float dtype) to contiguous fp64."""
    if hasattr(a, "detach"):  # torch tensor: widen with torch (numpy has no bf16)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _shapes(q, k):
    B, H, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d or Hkv < 1 or H % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape}")
    return B, H, Hkv, Nq, Nk, d


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())


def forward(q, k, v, causal: bool, scale: float, lib=None):
    """O [B,H,Nq,d] and L [B,H,Nq] (natural log) of exact attention, fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, Nq, Nk, d = _shapes(q, k)
    G = H // Hkv
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for kh in range(Hkv):
            qs = np.ascontiguousarray(q[b, kh * G:(kh + 1) * G])
            og = np.zeros((G, Nq, d))
            lg = np.zeros((G, Nq))
            lib.oracle_fwd_group(_ptr(qs), _ptr(np.ascontiguousarray(k[b, kh])),
                                 _ptr(np.ascontiguousarray(v[b, kh])), G, Nq, Nk, d,
                                 int(bool(causal)), float(scale), _ptr(og), _ptr(lg))
            o[b, kh * G:(kh + 1) * G] = og
            lse[b, kh * G:(kh + 1) * G] = lg
    return o, lse


def forward_group(q_group, k_head, v_head, causal: bool, scale: float, lib=None):
    """One key/value group: q [G,Nq,d], k/v [Nk,d] -> O [G,Nq,d], L [G,Nq]."""
    lib = lib or load()
    qg, kh, vh = _f64(q_group), _f64(k_head), _f64(v_head)
    G, Nq, d = qg.shape
    Nk = kh.shape[0]
    o = np.zeros((G, Nq, d))
    lse = np.zeros((G, Nq))
    lib.oracle_fwd_group(_ptr(qg), _ptr(kh), _ptr(vh), G, Nq, Nk, d, int(bool(causal)),
                         float(scale), _ptr(o), _ptr(lse))
    return o, lse


def forward_rows(q_group, k_head, v_head, rows, causal: bool, scale: float, lib=None):
    """Selected rows of one group: rows = [(g, i), ...] -> O [n,d], L [n]."""
    lib = lib or load()
    qg, kh, vh = _f64(q_group), _f64(k_head), _f64(v_head)
    G, Nq, d = qg.shape
    Nk = kh.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    if r.size and (r[:, 0].min() < 0 or r[:, 0].max() >= G or r[:, 1].min() < 0
                   or r[:, 1].max() >= Nq):
        raise ValueError("row index out of range")
    n = r.shape[0]
    o = np.zeros((n, d))
    lse = np.zeros((n,))
    lib.oracle_fwd_rows(_ptr(qg), _ptr(kh), _ptr(vh), G, Nq, Nk, d, int(bool(causal)),
                        float(scale), n, r.ctypes.data_as(_lp), _ptr(o), _ptr(lse))
    return o, lse


def backward_group(q_group, k_head, v_head, dout_group, causal: bool, scale: float, lib=None,
                   extras: bool = False):
    """One group's gradients: dQ [G,Nq,d], dK [Nk,d], dV [Nk,d] (+ O, L, D if extras)."""
    lib = lib or load()
    qg, kh, vh, dg = _f64(q_group), _f64(k_head), _f64(v_head), _f64(dout_group)
    G, Nq, d = qg.shape
    Nk = kh.shape[0]
    dq = np.zeros((G, Nq, d))
    dk = np.zeros((Nk, d))
    dv = np.zeros((Nk, d))
    o = np.zeros((G, Nq, d))
    lse = np.zeros((G, Nq))
    delta = np.zeros((G, Nq))
    lib.oracle_bwd_group(_ptr(qg), _ptr(kh), _ptr(vh), _ptr(dg), G, Nq, Nk, d,
                         int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                         _ptr(o), _ptr(lse), _ptr(delta))
    if extras:
        return dq, dk, dv, o, lse, delta
    return dq, dk, dv


def backward(q, k, v, dout, causal: bool, scale: float, lib=None):
    """dQ [B,H,Nq,d], dK/dV [B,Hkv,Nk,d] of sum(O o dO), fp64."""
    lib = lib or load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Hkv, Nq, Nk, d = _shapes(q, k)
    G = H // Hkv
    dq = np.zeros((B, H, Nq, d))
    dk = np.zeros((B, Hkv, Nk, d))
    dv = np.zeros((B, Hkv, Nk, d))
    for b in range(B):
        for kh in range(Hkv):
            sl = slice(kh * G, (kh + 1) * G)
            g_dq, g_dk, g_dv = backward_group(q[b, sl], k[b, kh], v[b, kh], dout[b, sl],
                                              causal, scale, lib)
            dq[b, sl] = g_dq
            dk[b, kh] = g_dk
            dv[b, kh] = g_dv
    return dq, dk, dv


def backward_rows(q_group, k_head, v_head, dout_group, r0: int, r1: int, causal: bool,
                  scale: float, dk=None, dv=None, lib=None):
    """Rows [r0, r1) of the flattened G*Nq query rows of one group: their dQ
    [r1-r0, d], and their contributions added into dk, dv [Nk, d] (new zero
    arrays unless given).  Returns (dq_rows, dk, dv)."""
    lib = lib or load()
    qg, kh, vh, dg = _f64(q_group), _f64(k_head), _f64(v_head), _f64(dout_group)
    G, Nq, d = qg.shape
    Nk = kh.shape[0]
    if not (0 <= r0 <= r1 <= G * Nq):
        raise ValueError("row range out of bounds")
    dq = np.zeros((r1 - r0, d))
    dk = np.zeros((Nk, d)) if dk is None else dk
    dv = np.zeros((Nk, d)) if dv is None else dv
    assert dk.dtype == np.float64 and dk.flags.c_contiguous and dk.shape == (Nk, d)
    assert dv.dtype == np.float64 and dv.flags.c_contiguous and dv.shape == (Nk, d)
    lib.oracle_bwd_rows(_ptr(qg), _ptr(kh), _ptr(vh), _ptr(dg), G, Nq, Nk, d, int(bool(causal)),
                        float(scale), int(r0), int(r1), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def _block_mask(block_mask, H: int, Nq: int, Nk: int, bs: int) -> np.ndarray:
    """Check a block mask [mask_heads, ceil(Nq/bs), ceil(Nk/bs)] (mask_heads 1 or H)
    and return it as contiguous uint8 (nonzero = the block is kept)."""
    m = np.ascontiguousarray(np.asarray(block_mask) != 0, dtype=np.uint8)
    nbr, nbc = -(-Nq // bs), -(-Nk // bs)
    if m.ndim != 3 or m.shape[0] not in (1, H) or m.shape[1:] != (nbr, nbc):
        raise ValueError(f"block mask shape {m.shape} does not fit H={H} "
                         f"[{nbr}, {nbc}] blocks of {bs}")
    return m


def forward_blocksparse(q, k, v, block_mask, causal: bool, scale: float, bs: int = 128,
                        lib=None):
    """Exact attention restricted to a block pattern: key k is visible to query i
    of head h only where block_mask[h or 0, i // bs, k // bs] != 0 (and, if
    causal, k <= i + Nk - Nq).  Returns O [B,H,Nq,d], L [B,H,Nq] in fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, Nq, Nk, d = _shapes(q, k)
    G = H // Hkv
    m = _block_mask(block_mask, H, Nq, Nk, bs)
    per_head = m.shape[0] == H
    nbc = m.shape[2]
    hstride = m.shape[1] * nbc if per_head else 0
    o = np.zeros((B, H, Nq, d))
    lse = np.zeros((B, H, Nq))
    for b in range(B):
        for kh in range(Hkv):
            sl = slice(kh * G, (kh + 1) * G)
            qs = np.ascontiguousarray(q[b, sl])
            mg = np.ascontiguousarray(m[sl] if per_head else m[0:1])
            og = np.zeros((G, Nq, d))
            lg = np.zeros((G, Nq))
            lib.oracle_fwd_group_blockmask(
                _ptr(qs), _ptr(np.ascontiguousarray(k[b, kh])),
                _ptr(np.ascontiguousarray(v[b, kh])), G, Nq, Nk, d, int(bool(causal)),
                mg.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), bs, nbc, hstride,
                float(scale), _ptr(og), _ptr(lg))
            o[b, sl] = og
            lse[b, sl] = lg
    return o, lse


def backward_blocksparse(q, k, v, dout, block_mask, causal: bool, scale: float,
                         bs: int = 128, lib=None):
    """Gradients of sum(O o dO) for the block-restricted attention of
    forward_blocksparse: dQ [B,H,Nq,d], dK/dV [B,Hkv,Nk,d] in fp64."""
    lib = lib or load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Hkv, Nq, Nk, d = _shapes(q, k)
    G = H // Hkv
    m = _block_mask(block_mask, H, Nq, Nk, bs)
    per_head = m.shape[0] == H
    nbc = m.shape[2]
    hstride = m.shape[1] * nbc if per_head else 0
    dq = np.zeros((B, H, Nq, d))
    dk = np.zeros((B, Hkv, Nk, d))
    dv = np.zeros((B, Hkv, Nk, d))
    for b in range(B):
        for kh in range(Hkv):
            sl = slice(kh * G, (kh + 1) * G)
            mg = np.ascontiguousarray(m[sl] if per_head else m[0:1])
            g_dq = np.zeros((G, Nq, d))
            g_dk = np.zeros((Nk, d))
            g_dv = np.zeros((Nk, d))
            lib.oracle_bwd_group_blockmask(
                _ptr(np.ascontiguousarray(q[b, sl])), _ptr(np.ascontiguousarray(k[b, kh])),
                _ptr(np.ascontiguousarray(v[b, kh])), _ptr(np.ascontiguousarray(dout[b, sl])),
                G, Nq, Nk, d, int(bool(causal)),
                mg.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), bs, nbc, hstride,
                float(scale), _ptr(g_dq), _ptr(g_dk), _ptr(g_dv))
            dq[b, sl] = g_dq
            dk[b, kh] = g_dk
            dv[b, kh] = g_dv
    return dq, dk, dv
