"""fa_fwd_splitkv (key axis split, partials merged by their logsumexps) and the
packed short-query path of fa_fwd_qk, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from parity import check_forward

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

SHAPES = [(1, 4096), (1, 300), (4, 1000), (16, 2000), (64, 517), (100, 900)]


def _check(o, lse, q, k, v, causal, scale, what):
    o_r, lse_r = oracle.forward(q, k, v, causal, scale)
    lse_c, lse_rc = lse.cpu().double().numpy(), lse_r.copy()
    empty = np.isneginf(lse_rc)
    assert np.array_equal(np.isneginf(lse_c), empty), what
    lse_c[empty] = 0.0
    lse_rc[empty] = 0.0
    check_forward(o.cpu(), lse_c, o_r, lse_rc, what)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 4)])
@pytest.mark.parametrize("Nq,Nk", SHAPES)
@pytest.mark.parametrize("splits", [0, 3])
def test_splitkv_matches_oracle(d, causal, H, Hkv, Nq, Nk, splits):
    w = Workload("split", 2, H, Hkv, Nq, d, "bf16", causal, 900 + Nq + Nk + d)
    q, k, v, _ = make_inputs(w, Nk=Nk)
    o, lse = binding.forward_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), causal, w.scale, splits)
    binding.device_status()
    _check(o, lse, q, k, v, causal, w.scale, f"splitkv{splits} d{d} c{causal} H{H}/{Hkv} {Nq}x{Nk}")


@pytest.mark.parametrize("Nq,Nk", [(1, 2048), (3, 700), (64, 1000)])
def test_packed_short_query_and_split_agree(Nq, Nk):
    """fa_fwd_qk (packed, one pass) and fa_fwd_splitkv give the same result up
    to rounding, for causal GQA short queries."""
    w = Workload("pack", 1, 16, 4, Nq, 128, "f16", True, 31)
    q, k, v, _ = make_inputs(w, Nk=Nk)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o1, l1 = binding.forward(qd, kd, vd, True, w.scale)
    o2, l2 = binding.forward_splitkv(qd, kd, vd, True, w.scale, 4)
    binding.device_status()
    _check(o1, l1, q, k, v, True, w.scale, "packed fa_fwd_qk")
    assert (o1.float() - o2.float()).abs().max().item() < 4e-3
    assert (l1 - l2).abs().max().item() < 1e-4


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("Nq,Nk", [(1000, 1000), (1000, 300), (700, 2000)])
def test_splitkv_splits_without_keys(d, Nq, Nk):
    """Causal with many query rows: the first query tiles see only the first
    key tiles, so the later splits hold no key for them.  Those splits' partials
    must carry weight 0 in the merge; the workspace starts filled with a finite
    non-zero pattern so that an unwritten partial would show."""
    w = Workload("split-empty", 1, 4, 2, Nq, d, "bf16", True, 41 + Nq + Nk + d)
    q, k, v, _ = make_inputs(w, Nk=Nk)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for splits in (3, 8):
        need = int(binding.load().fa_fwd_splitkv_workspace_size(1, 4, 2, Nq, Nk, d, splits))
        ws = torch.full((max(need, 256),), 0x3F, dtype=torch.uint8, device=DEV)
        o, lse = binding.forward_splitkv(qd, kd, vd, True, w.scale, splits, workspace=ws)
        binding.device_status()
        _check(o, lse, q, k, v, True, w.scale, f"splitkv{splits} empty splits d{d} {Nq}x{Nk}")
