"""Block-sparse attention (exact attention restricted to the kept 128 x 128
blocks of a mask) through fa_fwd_blocksparse / fa_bwd_blocksparse, against
the fp64 oracle with the same block mask."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_block_mask, make_inputs
from parity import check_forward, check_grads, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _mask(heads, Nq, Nk, density, seed):
    m = make_block_mask(heads, Nq, Nk, density, seed)
    m[0, 0, :] = 0          # a query block that sees nothing: O = 0, L = -inf
    if m.shape[2] > 1:
        m[:, :, 1] = 0      # a key block no query sees: dK = dV = 0
    return m


def _run(w, Nk, mask, causal):
    q, k, v, do = make_inputs(w, Nk=Nk)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    md = mask.to(DEV)
    o, lse = binding.forward_blocksparse(qd, kd, vd, md, causal, w.scale)
    grads = [binding.backward_blocksparse(qd, kd, vd, o, lse, dod, md, causal, w.scale,
                                          deterministic=det) for det in (False, True)]
    binding.device_status()
    return (q, k, v, do), (o, lse), grads


def _check(w, Nk, mask, causal, inputs, fwd, grads, what):
    q, k, v, do = inputs
    o, lse = fwd
    mnp = mask.numpy()
    o_r, lse_r = oracle.forward_blocksparse(q, k, v, mnp, causal, w.scale)
    lse_c, lse_rc = lse.cpu().double().numpy(), lse_r.copy()
    empty = np.isneginf(lse_rc)
    assert np.array_equal(np.isneginf(lse_c), empty), f"{what}: empty rows differ"
    assert torch.all(o.cpu()[torch.from_numpy(empty)] == 0)
    lse_c[empty] = 0.0
    lse_rc[empty] = 0.0
    check_forward(o.cpu(), lse_c, o_r, lse_rc, f"{what} fwd")
    dq_r, dk_r, dv_r = oracle.backward_blocksparse(q, k, v, do, mnp, causal, w.scale)
    # keys that no query of their group sees under the mask: dK = dV = 0 exactly
    B, H, Nq = lse_r.shape
    Hkv = k.shape[1]
    keep = np.repeat(np.repeat(mnp.astype(bool), 128, axis=1), 128, axis=2)[:, :Nq, :Nk]
    if causal:
        keep = keep & (np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq))[None]
    keep = np.broadcast_to(keep, (H, Nq, Nk))
    unseen = ~keep.reshape(Hkv, H // Hkv, Nq, Nk).any(axis=(1, 2))       # [Hkv, Nk]
    unseen = torch.from_numpy(np.broadcast_to(unseen, (B, Hkv, Nk)).copy())
    for det, (dq, dk, dv) in zip((False, True), grads):
        assert torch.all(dq.cpu()[torch.from_numpy(empty)] == 0), f"{what}: dq of empty rows"
        assert torch.all(dk.cpu()[unseen] == 0) and torch.all(dv.cpu()[unseen] == 0), \
            f"{what}: dk/dv of unseen keys"
        check_grads([("dq", dq.cpu(), dq_r), ("dk", dk.cpu(), dk_r), ("dv", dv.cpu(), dv_r)],
                    f"{what} bwd det{det}")


SHAPES = [(512, 512), (300, 700), (700, 300), (1000, 1000)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
@pytest.mark.parametrize("per_head", [False, True])
def test_blocksparse_matches_oracle(d, causal, Nq, Nk, per_head):
    w = Workload("bs", 1, 4, 2, Nq, d, "bf16", causal, 11 + Nq + 5 * Nk + d + per_head)
    mask = _mask(w.H if per_head else 1, Nq, Nk, 0.5, w.seed)
    inputs, fwd, grads = _run(w, Nk, mask, causal)
    _check(w, Nk, mask, causal, inputs, fwd, grads,
           f"blocksparse d{d} c{causal} {Nq}x{Nk} heads{mask.shape[0]}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_the_dense_kernel(d, causal):
    """Every block kept: the same tiles in the same order as the dense path,
    so the forward and the deterministic backward agree with it bit for bit.
    (The dense forward at d = 128 runs the two-tile kernel, which sums the
    row weights on the ALU and divides by their exact sum: there the forward
    is compared within the parity tolerances.  The dense backward at d = 256
    runs its own kernels (the cluster pair for dK and dV, with 128-row steps
    and dS from the 16-bit weights; a dQ kernel with 128-key tiles summed in a
    staggered order): there the gradients are compared within the rounding of
    the weights and of the 16-bit outputs.)"""
    w = Workload("bs1", 2, 4, 1, 640, d, "f16", causal, 90 + d)
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    ones = torch.ones((1, 5, 5), dtype=torch.uint8, device=DEV)
    o_s, l_s = binding.forward_blocksparse(q, k, v, ones, causal, w.scale)
    o_d, l_d = binding.forward(q, k, v, causal, w.scale)
    g_s = binding.backward_blocksparse(q, k, v, o_d, l_d, do, ones, causal, w.scale,
                                       deterministic=True)
    g_d = binding.backward(q, k, v, o_d, l_d, do, causal, w.scale, deterministic=True)
    binding.device_status()
    if d == 128:
        assert (o_s.float() - o_d.float()).abs().max().item() <= 2e-3
        assert (l_s - l_d).abs().max().item() <= 1e-5
    else:
        assert torch.equal(o_s, o_d) and torch.equal(l_s, l_d)
    if d == 256:
        for a, b in zip(g_s, g_d):
            assert rel_l2(a, b) <= 1e-2
    else:
        for a, b in zip(g_s, g_d):
            assert torch.equal(a, b)


def test_empty_mask_gives_zeros():
    w = Workload("bs0", 1, 2, 2, 300, 128, "bf16", False, 5)
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    zero = torch.zeros((2, 3, 3), dtype=torch.uint8, device=DEV)
    o, lse = binding.forward_blocksparse(q, k, v, zero, False, w.scale)
    for det in (False, True):
        dq, dk, dv = binding.backward_blocksparse(q, k, v, o, lse, do, zero, False, w.scale,
                                                  deterministic=det)
        binding.device_status()
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
        assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


def test_gqa_per_head_masks_long():
    """GQA group of 8 heads with their own masks, 2048 queries over 4096 keys
    (16 x 32 blocks, 30 % kept), causal, against the oracle everywhere."""
    w = Workload("bsl", 1, 8, 1, 2048, 128, "bf16", True, 77)
    Nk = 4096
    mask = _mask(8, 2048, Nk, 0.3, 77)
    inputs, fwd, grads = _run(w, Nk, mask, True)
    _check(w, Nk, mask, True, inputs, fwd, grads, "blocksparse gqa8 2048x4096")
