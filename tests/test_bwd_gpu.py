"""GPU backward parity against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import WORKLOADS, Workload, make_inputs
from parity import check_forward, check_grads, check_grads_tiled

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_fwd_bwd(w: Workload):
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = binding.forward(qd, kd, vd, w.causal, w.scale)
    dq, dk, dv = binding.backward(qd, kd, vd, o, lse, dod, w.causal, w.scale)
    binding.device_status()
    return (q, k, v, do), (o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu())


SWEEP = []
for d in (64, 128, 256):
    for causal in (False, True):
        for dtype in ("bf16", "f16"):
            for (H, Hkv) in ((2, 2), (4, 1)):
                for N in (1, 17, 128, 129, 300):
                    SWEEP.append((d, causal, dtype, H, Hkv, N))


@pytest.mark.parametrize("d,causal,dtype,H,Hkv,N", SWEEP)
def test_backward_sweep(d, causal, dtype, H, Hkv, N):
    w = Workload("sweep", 1, H, Hkv, N, d, dtype, causal, 101 + N + d)
    (q, k, v, do), (o, lse, dq, dk, dv) = run_fwd_bwd(w)
    dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, causal, w.scale)
    check_grads([("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)],
                f"bwd d{d} causal{causal} {dtype} H{H}/{Hkv} N{N}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [383, 640, 1000])
def test_backward_several_tiles_gqa(N, d):
    """Several key and query tiles, three query heads per kv head, two
    batches: every head dim's unit walk (key tiles x heads x query tiles, the
    heavy-first order under the mask) and its ragged last tiles."""
    for causal in (False, True):
        w = Workload("multi", 2, 6, 2, N, d, "bf16", causal, 7 + N + d)
        (q, k, v, do), (o, lse, dq, dk, dv) = run_fwd_bwd(w)
        dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, causal, w.scale)
        check_grads([("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)], f"bwd d{d} N{N} c{causal}")


def test_backward_tiny_workload():
    w = WORKLOADS["tiny"]
    (q, k, v, do), (o, lse, dq, dk, dv) = run_fwd_bwd(w)
    dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, w.causal, w.scale)
    check_grads([("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)], "bwd tiny")


def test_backward_dk_dv_deterministic_and_workspace_contents_ignored():
    w = Workload("det", 1, 8, 2, 900, 128, "bf16", True, 4)
    q, k, v, do = make_inputs(w, DEV)
    o, lse = binding.forward(q, k, v, w.causal, w.scale)
    need = binding.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device=DEV)   # garbage contents
    r1 = binding.backward(q, k, v, o, lse, do, w.causal, w.scale, workspace=ws)
    ws.fill_(0xFF)
    r2 = binding.backward(q, k, v, o, lse, do, w.causal, w.scale, workspace=ws)
    binding.device_status()
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])
    # dQ: equal up to the order of the atomic additions
    assert (r1[0].float() - r2[0].float()).abs().max().item() < 1e-2


@pytest.mark.parametrize("deterministic", [False, True])
def test_backward_with_exactly_the_workspace_of_its_path(deterministic):
    """d = 128: the deterministic path runs in D's bytes alone, the default
    path in D plus the accumulator; both against the oracle."""
    w = Workload("ws", 1, 8, 2, 700, 128, "bf16", True, 21)
    q, k, v, do = make_inputs(w)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = binding.forward(qd, kd, vd, w.causal, w.scale)
    need = binding.fa_bwd_workspace_size_for(w.B, w.H, w.Hkv, w.N, w.d, deterministic)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    dq, dk, dv = binding.backward(qd, kd, vd, o, lse, dod, w.causal, w.scale, workspace=ws,
                                  deterministic=deterministic)
    binding.device_status()
    dq_r, dk_r, dv_r = oracle.backward(q, k, v, do, w.causal, w.scale)
    check_grads([("dq", dq.cpu(), dq_r), ("dk", dk.cpu(), dk_r), ("dv", dv.cpu(), dv_r)],
                f"exact workspace det{deterministic}")


FULL = ["gpt_layer", "gpt_layer_causal", "long_seq", "head256", "gqa8k"]


@pytest.mark.parametrize("name", FULL)
def test_backward_full_size_group(name):
    """Full-size workloads: every gradient of the first and the last (batch,
    kv-head) groups against the oracle, over each whole group and over every
    (head, 128-row) tile of dQ and (128-key) tile of dK and dV on its own
    (the forward outputs of those groups too)."""
    w = WORKLOADS[name]
    (q, k, v, do), (o, lse, dq, dk, dv) = run_fwd_bwd(w)
    G = w.H // w.Hkv
    for b, kh in {(0, 0), (w.B - 1, w.Hkv - 1)}:
        sl = slice(kh * G, (kh + 1) * G)
        dq_r, dk_r, dv_r, o_r, lse_r, _ = oracle.backward_group(
            q[b, sl], k[b, kh], v[b, kh], do[b, sl], w.causal, w.scale, extras=True)
        what = f"{name} (b{b}, kvh{kh})"
        check_forward(o[b, sl], lse[b, sl], o_r, lse_r, what + " fwd")
        check_grads([("dq", dq[b, sl], dq_r), ("dk", dk[b, kh], dk_r), ("dv", dv[b, kh], dv_r)],
                    what + " bwd")
        check_grads_tiled([("dq", dq[b, sl], dq_r), ("dk", dk[b, kh][None], dk_r[None]),
                           ("dv", dv[b, kh][None], dv_r[None])], 128, what + " bwd tiles")
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_reduce_rate_diagnostic():
    """fa_measure_reduce_rate: a plausible rate (0.5 to 50 TB/s over all SMs)
    and finite scratch contents left unchanged (zeros are added)."""
    scratch = torch.full((8 << 20,), 1.5, dtype=torch.float32, device="cuda")
    rate = binding.measure_reduce_rate(scratch)
    assert 5e11 < rate < 5e13, rate
    assert bool((scratch == 1.5).all())
