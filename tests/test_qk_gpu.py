"""Separate query and key lengths (prefix / decode / cross-attention shapes):
forward and both backward paths against the fp64 oracle, whose mask is
anchored at the bottom-right corner (query i sees keys k <= i + Nk - Nq)."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from parity import check_forward, check_grads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SHAPES = [(1, 1000), (5, 300), (77, 500), (300, 1000), (129, 129), (500, 200), (260, 64),
          (1000, 300)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
def test_qk_forward_backward(d, causal, Nq, Nk):
    w = Workload("qk", 1, 4, 2, Nq, d, "bf16", causal, 7 + Nq + 3 * Nk + d)
    q, k, v, do = make_inputs(w, Nk=Nk)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = binding.forward(qd, kd, vd, causal, w.scale)
    res = [binding.backward(qd, kd, vd, o, lse, dod, causal, w.scale, deterministic=det)
           for det in (False, True)]
    binding.device_status()
    o_r, lse_r = oracle.forward(q, k, v, causal, w.scale)
    lse_c, lse_rc = lse.cpu().double().numpy(), lse_r.copy()
    empty = np.isneginf(lse_rc)
    # rows that see no key: O = 0 and L = -inf exactly
    assert np.array_equal(np.isneginf(lse_c), empty)
    assert torch.all(o.cpu()[torch.from_numpy(empty)] == 0)
    lse_c[empty] = 0.0
    lse_rc[empty] = 0.0
    check_forward(o.cpu(), lse_c, o_r, lse_rc, f"qk fwd d{d} c{causal} {Nq}x{Nk}")
    dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, causal, w.scale)
    for det, (dq, dk, dv) in zip((False, True), res):
        check_grads([("dq", dq.cpu(), dq_r), ("dk", dk.cpu(), dk_r), ("dv", dv.cpu(), dv_r)],
                    f"qk bwd det{det} d{d} c{causal} {Nq}x{Nk}")
