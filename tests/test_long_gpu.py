"""Sequences four times the longest workload's (N = 65,573 queries and keys,
so the last 128-row tile is ragged), causal, two query heads on one kv head,
at every head dim, through the forward and both backward entry points.

The oracle cannot form these gradients whole, so the test takes what it can
compute one row at a time, plus two identities that hold at any size:
  - O and L on sampled rows (forward_rows);
  - dQ of the first query tile and of the last rows (backward_rows);
  - dK and dV of the last key tile exactly: under the causal mask with
    Nq = Nk only the rows from that tile's first key on see its keys, so
    those rows' contributions (backward_rows) are the whole gradient there;
  - sum over keys of dV = sum over the group's rows of dO: each softmax row
    sums to one ("FlashAttention-2" paper digest, section 3 backward: dV =
    P^T dO);
  - sum over keys of dK = 0: each row of dS = P o (dP - D) sums to zero,
    because sum_j P_ij dP_ij = dO_i . O_i = D_i (section 4, the D term).
The identities are checked with the gradients' relative L2 bound (2e-2):
with P and the outputs rounded to bf16 (unit roundoff u = 2^-8) the expected
error is about u times the norm of the terms, a few 1e-3, while a missing or
misplaced block of the sum moves it by far more.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from parity import GRAD_REL_L2, check_forward, check_grads, rel_l2, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
N = 65536 + 37


@pytest.mark.parametrize("d", [64, 128, 256])
def test_long_sequence_sampled_and_identities(d):
    w = Workload("long", 1, 2, 1, N, d, "bf16", True, 907 + d)
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = binding.forward(qd, kd, vd, True, w.scale)
    res = {det: binding.backward(qd, kd, vd, o, lse, dod, True, w.scale, deterministic=det)
           for det in (False, True)}
    binding.device_status()
    o, lse = o.cpu(), lse.cpu()
    G = w.H // w.Hkv
    qg, kh, vh, dog = (to_np(t) for t in (q[0], k[0, 0], v[0, 0], do[0]))   # fp64 once

    # forward: sampled rows of both heads
    idx = [0, 1, 127, 128, 4097, 40000, N - 38, N - 37, N - 1]
    rows = [(g, i) for g in range(G) for i in idx]
    o_r, lse_r = oracle.forward_rows(qg, kh, vh, rows, True, w.scale)
    o_g = torch.stack([o[0, g, i] for g, i in rows])
    lse_g = np.array([float(lse[0, g, i]) for g, i in rows])
    check_forward(o_g, lse_g, o_r, lse_r, f"long d{d} fwd rows")

    # the oracle's rows: the first query tile of head 0 and, for every head,
    # the rows from the last key tile's first key on (their dK / dV
    # contributions are that tile's whole gradient)
    last0 = (N - 1) // 128 * 128
    dq_first, _, _ = oracle.backward_rows(qg, kh, vh, dog, 0, 128, True, w.scale)
    dk_last = np.zeros((N, d))
    dv_last = np.zeros((N, d))
    dq_last = []
    for g in range(G):
        dq_g, _, _ = oracle.backward_rows(qg, kh, vh, dog, g * N + last0, (g + 1) * N, True,
                                          w.scale, dk=dk_last, dv=dv_last)
        dq_last.append(dq_g)
    sum_do = dog.sum(axis=(0, 1))                      # sum over the group's rows

    for det, (dq, dk, dv) in res.items():
        what = f"long d{d} det{int(det)}"
        dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
        for t in (dq, dk, dv):
            assert torch.isfinite(t.float()).all(), what
        check_grads([("dq first tile", dq[0, 0, :128], dq_first)]
                    + [(f"dq last rows h{g}", dq[0, g, last0:], dq_last[g]) for g in range(G)]
                    + [("dk last tile", dk[0, 0, last0:], dk_last[last0:]),
                       ("dv last tile", dv[0, 0, last0:], dv_last[last0:])], what)
        dv_np, dk_np = to_np(dv[0, 0]), to_np(dk[0, 0])
        e_v = rel_l2(dv_np.sum(axis=0), sum_do)
        e_k = float(np.linalg.norm(dk_np.sum(axis=0))) / float(np.linalg.norm(dk_np))
        assert e_v <= GRAD_REL_L2, f"{what}: sum of dV against sum of dO, rel_l2 {e_v:.3e}"
        assert e_k <= GRAD_REL_L2, f"{what}: sum of dK against its norm {e_k:.3e}"
