"""Failure detection on the GPU without a fault: an expired bounded wait is
reported as FA_ERR_TIMEOUT by fa_get_device_status, once, and the context
keeps working afterwards."""
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from parity import check_forward

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    lib = binding.load()
    assert binding.fa_get_device_status() == binding.FA_OK
    stream = torch.cuda.current_stream().cuda_stream or None
    assert lib.fa_selftest_expired_wait(20000, stream) == binding.FA_OK
    assert binding.fa_get_device_status() == binding.FA_ERR_TIMEOUT
    assert binding.fa_get_device_status() == binding.FA_OK     # the word was cleared
    w = Workload("after", 1, 2, 1, 300, 64, "bf16", True, 5)
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.cuda(), k.cuda(), v.cuda(), w.causal, w.scale)
    binding.device_status()
    o_ref, lse_ref = oracle.forward(q, k, v, w.causal, w.scale)
    check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref, "forward after an expired wait")


def test_selftest_rejects_bad_limits():
    lib = binding.load()
    assert lib.fa_selftest_expired_wait(0, None) == binding.FA_ERR_INVALID_ARG
    assert lib.fa_selftest_expired_wait(3000000, None) == binding.FA_ERR_INVALID_ARG
