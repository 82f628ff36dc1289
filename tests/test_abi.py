"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from exact_io_aware_20_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from exact_io_aware_20_gb300 import build
        build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(binding.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr), name


def test_measure_reduce_rate_rejects_bad_buffers(lib):
    """Refused on the host, before any launch: no buffer, less than 1 MiB,
    or not 256-byte aligned."""
    out = ctypes.c_double(0.0)
    for ptr, size in ((None, 1 << 24), (FAKE, (1 << 20) - 16), (FAKE + 16, 1 << 24)):
        st = lib.fa_measure_reduce_rate(ptr, size, ctypes.byref(out), None)
        assert st == binding.FA_ERR_INVALID_ARG, (ptr, size)
    assert lib.fa_measure_reduce_rate(FAKE, 1 << 24, None, None) == binding.FA_ERR_INVALID_ARG


def test_strerror(lib):
    for st in range(6):
        assert binding.strerror(st)
    assert binding.strerror(99) == "unknown status"


def test_workspace_size(lib):
    B, H, N, d = 2, 4, 100, 64
    # D, the fp32 dQ accumulator (each padded to 256 bytes), the work counter
    want = (-(-B * H * N * 4 // 256)) * 256 + (-(-B * H * N * d * 4 // 256)) * 256 + 256
    assert binding.fa_bwd_workspace_size(B, H, 2, N, d) == want
    assert binding.fa_bwd_workspace_size(B, H, 3, N, d) == 0   # H % Hkv
    assert binding.fa_bwd_workspace_size(0, H, 2, N, d) == 0
    assert binding.fa_bwd_workspace_size(B, H, 2, N, 96) == 0


def test_workspace_size_for_the_path(lib):
    """The deterministic path needs only D (dQ is written directly); the
    default path D and the fp32 dQ accumulator, which is the upper bound."""
    B, H, N = 2, 32, 8192
    delta = -(-B * H * N * 4 // 256) * 256
    for d in (64, 128, 256):
        assert binding.fa_bwd_workspace_size_for(B, H, 8, N, d, True) == delta
        assert binding.fa_bwd_workspace_size_for(B, H, 8, N, d, False) == \
            binding.fa_bwd_workspace_size(B, H, 8, N, d)
    assert binding.load().fa_bwd_workspace_size_for(B, H, 8, N, 128, 2) == 0
    assert binding.fa_bwd_workspace_size_for(B, H, 3, N, 128, True) == 0


def test_backward_rejects_a_workspace_too_small_for_its_path(lib):
    """With only D's bytes the default (accumulating) path is refused before
    anything is enqueued; the deterministic path accepts them (checked on the
    GPU in test_bwd_gpu.py)."""
    B, H, Hkv, N, d = 1, 4, 4, 256, 128
    only_d = binding.fa_bwd_workspace_size_for(B, H, Hkv, N, d, True)
    st = lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv, N, d, 1,
                    0.088, binding.FA_BF16, FAKE, only_d, None)
    assert st == binding.FA_ERR_WORKSPACE
    st = lib.fa_bwd_deterministic(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv,
                                  N, d, 1, 0.088, binding.FA_BF16, FAKE, only_d - 256, None)
    assert st == binding.FA_ERR_WORKSPACE


FAKE = 1 << 20   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("case,expect", [
    (dict(B=0), binding.FA_ERR_INVALID_ARG),
    (dict(N=0), binding.FA_ERR_INVALID_ARG),
    (dict(Hkv=3), binding.FA_ERR_INVALID_ARG),
    (dict(causal=2), binding.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), binding.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), binding.FA_ERR_INVALID_ARG),
    (dict(B=65536), binding.FA_ERR_INVALID_ARG),
    (dict(d=96), binding.FA_ERR_UNSUPPORTED),
    (dict(d=32), binding.FA_ERR_UNSUPPORTED),
    (dict(dtype=2), binding.FA_ERR_UNSUPPORTED),
    (dict(q=None), binding.FA_ERR_INVALID_ARG),
    (dict(lse=None), binding.FA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), binding.FA_ERR_INVALID_ARG),   # not 16-byte aligned
])
def test_fwd_rejects(lib, case, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=4, Hkv=2, N=64, d=64, causal=0,
             scale=0.125, dtype=binding.FA_BF16)
    a.update(case)
    st = lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["N"],
                    a["d"], a["causal"], a["scale"], a["dtype"], None)
    assert st == expect


@pytest.mark.parametrize("case,expect", [
    (dict(H=5), binding.FA_ERR_INVALID_ARG),
    (dict(dout=None), binding.FA_ERR_INVALID_ARG),
    (dict(dk=FAKE + 4), binding.FA_ERR_INVALID_ARG),
    (dict(ws=None), binding.FA_ERR_WORKSPACE),
    (dict(ws_bytes=16), binding.FA_ERR_WORKSPACE),
    (dict(ws=FAKE + 16), binding.FA_ERR_WORKSPACE),   # not 256-byte aligned
    (dict(d=48), binding.FA_ERR_UNSUPPORTED),
])
def test_bwd_rejects(lib, case, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, H=4, Hkv=2, N=64, d=64, causal=1, scale=0.125, dtype=binding.FA_F16,
             ws=FAKE, ws_bytes=1 << 30)
    a.update(case)
    st = lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"],
                    a["dv"], a["B"], a["H"], a["Hkv"], a["N"], a["d"], a["causal"], a["scale"],
                    a["dtype"], a["ws"], a["ws_bytes"], None)
    assert st == expect


def test_splitkv_workspace_checks(lib):
    B, H, Hkv, Nq, Nk, d = 2, 8, 2, 1, 4096, 128
    need = binding.load().fa_fwd_splitkv_workspace_size(B, H, Hkv, Nq, Nk, d, 4)
    assert need == 4 * B * H * Nq * d * 4 + 256   # partial O + (padded) partial L
    assert binding.load().fa_fwd_splitkv_workspace_size(B, H, Hkv, Nq, Nk, d, 1) == 0
    assert binding.load().fa_fwd_splitkv_workspace_size(B, H, 3, Nq, Nk, d, 4) == 0
    st = lib.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv, Nq, Nk, d, 1, 0.088,
                            binding.FA_BF16, 4, FAKE, 16, None)
    assert st == binding.FA_ERR_WORKSPACE
    st = lib.fa_fwd_splitkv(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, Hkv, Nq, Nk, d, 1, 0.088,
                            binding.FA_BF16, -1, FAKE, 1 << 30, None)
    assert st == binding.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("case,expect", [
    (dict(mask=None), binding.FA_ERR_INVALID_ARG),
    (dict(mask_heads=3), binding.FA_ERR_INVALID_ARG),      # neither 1 nor H
    (dict(mask_heads=0), binding.FA_ERR_INVALID_ARG),
    (dict(Nk=8193 * 128), binding.FA_ERR_INVALID_ARG),     # forward key-tile list
    (dict(d=256, Nk=8193 * 128), binding.FA_ERR_INVALID_ARG),   # 128-key tiles at every d
    (dict(q=FAKE + 2), binding.FA_ERR_INVALID_ARG),
    (dict(d=80), binding.FA_ERR_UNSUPPORTED),
])
def test_fwd_blocksparse_rejects(lib, case, expect):
    a = dict(q=FAKE, Nk=512, d=128, mask=FAKE, mask_heads=1)
    a.update(case)
    st = lib.fa_fwd_blocksparse(a["q"], FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 256, a["Nk"], a["d"], 0,
                                0.1, binding.FA_BF16, a["mask"], a["mask_heads"], None)
    assert st == expect


@pytest.mark.parametrize("case,expect", [
    (dict(mask=None), binding.FA_ERR_INVALID_ARG),
    (dict(mask_heads=2), binding.FA_ERR_INVALID_ARG),
    (dict(det=2), binding.FA_ERR_INVALID_ARG),
    # (H / Hkv) * ceil(Nq / 128) above the d = 128 step list (8192)
    (dict(H=8, Hkv=2, Nq=128 * 2049), binding.FA_ERR_INVALID_ARG),
    (dict(d=256, H=4, Hkv=1, Nq=64 * 1025), binding.FA_ERR_INVALID_ARG),   # 4096 at d = 256
    (dict(det=1, Nk=64 * 8193), binding.FA_ERR_INVALID_ARG),   # dQ kernel key-tile list
    (dict(ws=None), binding.FA_ERR_WORKSPACE),
])
def test_bwd_blocksparse_rejects(lib, case, expect):
    a = dict(H=4, Hkv=4, Nq=256, Nk=256, d=128, mask=FAKE, mask_heads=1, det=0, ws=FAKE)
    a.update(case)
    st = lib.fa_bwd_blocksparse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, a["H"],
                                a["Hkv"], a["Nq"], a["Nk"], a["d"], 1, 0.1, binding.FA_F16,
                                a["mask"], a["mask_heads"], a["det"], a["ws"], 1 << 40, None)
    assert st == expect


def _fa_strides(vals):
    arr = (binding.FaStrides * len(vals))()
    for i, v in enumerate(vals):
        arr[i] = binding.FaStrides(*v)
    return arr


@pytest.mark.parametrize("bad", [None, (0, 64, 8192), (8192, 64, 12), (-64, 64, 8192),
                                 (1 << 40, 64, 8192)])
def test_strided_rejects(lib, bad):
    good = (4 * 256 * 64, 256 * 64, 64)
    fwd = None if bad is None else _fa_strides([good, good, bad, good])
    st = lib.fa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 4, 256, 256, 64, 0, 0.1,
                            binding.FA_BF16, fwd, None)
    assert st == binding.FA_ERR_INVALID_ARG
    bwd = None if bad is None else _fa_strides([good] * 7 + [bad])
    st = lib.fa_bwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 4, 256,
                            256, 64, 0, 0.1, binding.FA_BF16, bwd, 0, FAKE, 1 << 30, None)
    assert st == binding.FA_ERR_INVALID_ARG
