"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (plugins handed only inputs and outputs, processes that must not call
cudaMalloc after start-up).  It must give fa_bwd's gradients, call after
call, from the library's fixed scratch array.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from parity import check_grads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("w", [
    Workload("noalloc", 2, 8, 2, 1000, 128, "bf16", True, 42),
    Workload("noalloc64", 1, 4, 4, 777, 64, "f16", False, 43),
], ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_twice(w):
    q, k, v, do = make_inputs(w, DEV)
    o, lse = binding.forward(q, k, v, w.causal, w.scale)
    dq_ref, dk_ref, dv_ref = binding.backward(q, k, v, o, lse, do, w.causal, w.scale)
    code = binding.FA_BF16 if w.dtype == "bf16" else binding.FA_F16
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = binding.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, w.B, w.H, w.Hkv, w.N, w.d,
                                    w.causal, w.scale, code)
        assert st == binding.FA_OK, binding.strerror(st)
        binding.device_status()
        check_grads([("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)],
                    f"noalloc call {call}")
        # dK and dV have no atomics: the same bits as fa_bwd
        assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)


def test_noalloc_rejects_problems_above_its_scratch():
    B, H, Hkv, N, d = 1, 32, 8, 8192, 128     # needs ~129 MiB of scratch
    assert binding.fa_bwd_workspace_size(B, H, Hkv, N, d) > 64 * 2**20
    fake = 1 << 20                           # never dereferenced: rejected on the host
    st = binding.load().fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                       B, H, Hkv, N, d, 1, 0.088, binding.FA_BF16, None)
    assert st == binding.FA_ERR_WORKSPACE


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second GPU")
def test_noalloc_on_a_second_device():
    """The scratch address is looked up per device, with that device current:
    a call under device 1 gives fa_bwd's gradients there."""
    w = Workload("noalloc_dev1", 1, 4, 2, 300, 128, "bf16", True, 44)
    dev = torch.device("cuda", 1)
    with torch.cuda.device(dev):
        q, k, v, do = make_inputs(w, dev)
        o, lse = binding.forward(q, k, v, w.causal, w.scale)
        dq_ref, dk_ref, dv_ref = binding.backward(q, k, v, o, lse, do, w.causal, w.scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = binding.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, w.B, w.H, w.Hkv, w.N, w.d,
                                    w.causal, w.scale, binding.FA_BF16)
        assert st == binding.FA_OK, binding.strerror(st)
        binding.device_status()
        check_grads([("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)], "noalloc dev1")
