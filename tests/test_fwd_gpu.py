"""GPU forward parity against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_20_gb300 import binding
from exact_io_aware_20_gb300.inputs import WORKLOADS, Workload, make_inputs
from parity import check_forward, max_abs, record, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_fwd(w: Workload):
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), w.causal, w.scale)
    binding.device_status()
    return (q, k, v), o.cpu(), lse.cpu()


SWEEP = []
for d in (64, 128, 256):
    for causal in (False, True):
        for dtype in ("bf16", "f16"):
            for (H, Hkv) in ((2, 2), (4, 1)):
                for N in (1, 17, 128, 129, 300):
                    SWEEP.append((d, causal, dtype, H, Hkv, N))


@pytest.mark.parametrize("d,causal,dtype,H,Hkv,N", SWEEP)
def test_forward_sweep(d, causal, dtype, H, Hkv, N):
    w = Workload("sweep", 1, H, Hkv, N, d, dtype, causal, 77 + N + d)
    (q, k, v), o, lse = run_fwd(w)
    o_ref, lse_ref = oracle.forward(q, k, v, causal, w.scale)
    check_forward(o, lse, o_ref, lse_ref, f"d{d} causal{causal} {dtype} H{H}/{Hkv} N{N}")


@pytest.mark.parametrize("N", [383, 640, 1000])
def test_forward_several_tiles_gqa(N):
    for causal in (False, True):
        w = Workload("multi", 2, 6, 2, N, 128, "bf16", causal, 5 + N)
        (q, k, v), o, lse = run_fwd(w)
        o_ref, lse_ref = oracle.forward(q, k, v, causal, w.scale)
        check_forward(o, lse, o_ref, lse_ref, f"N{N} causal{causal}")


def test_forward_tiny_workload():
    w = WORKLOADS["tiny"]
    (q, k, v), o, lse = run_fwd(w)
    o_ref, lse_ref = oracle.forward(q, k, v, w.causal, w.scale)
    check_forward(o, lse, o_ref, lse_ref, "tiny")


def test_forward_deterministic():
    w = Workload("det", 2, 4, 2, 700, 128, "bf16", True, 3)
    q, k, v, _ = make_inputs(w, DEV)
    o1, l1 = binding.forward(q, k, v, w.causal, w.scale)
    o2, l2 = binding.forward(q, k, v, w.causal, w.scale)
    binding.device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_large_scores_f16():
    """Scores spread far apart (scale 4, values x3): exercises the running-max
    rescale path, checked with the stated O / L bounds.  Runs in f16: with
    values x3 |O| reaches ~10, where one bf16 half-ulp (0.031) is above the O
    bound."""
    w = Workload("wide", 1, 2, 2, 517, 64, "f16", False, 9, 3.0)
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), False, 4.0)
    binding.device_status()
    o_ref, lse_ref = oracle.forward(q, k, v, False, 4.0)
    check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref, "wide scores f16")


@pytest.mark.parametrize("causal", [False, True])
def test_forward_large_scores_two_tile_f16(causal):
    """The d = 128 two-query-tile kernel under spread-out scores (scale 4,
    values x3): its running-max rescale of O runs on many key tiles."""
    w = Workload("wide", 2, 4, 2, 1100, 128, "f16", causal, 19, 3.0)
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal, 4.0)
    binding.device_status()
    o_ref, lse_ref = oracle.forward(q, k, v, causal, 4.0)
    check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref, f"wide scores two-tile causal{causal}")


def test_forward_large_scores_bf16():
    """Peaky softmax (scale 3, N(0,1) values) in bf16: the rescale path in bf16.

    The stated O bound (1e-2) is for the 1/sqrt(d)-scaled workloads.  Here a few
    keys dominate each row, so the error is the bf16 floor: with an 8-bit
    significand, rounding each weight P costs up to 2^-8 relative (after the
    normalisation by the rounded sum, up to 2 * 2^-8 of |V_k - O| per weight)
    and rounding O up to 2^-8 |O|, so |err| <= 2^-7 max|V| + 2^-8 max|O| (both
    <= max|V|).  That bound, rel_L2 <= 5e-3 and the L bound are checked."""
    w = Workload("wide", 1, 2, 2, 517, 64, "bf16", False, 9, 1.0)
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), False, 3.0)
    binding.device_status()
    o_ref, lse_ref = oracle.forward(q, k, v, False, 3.0)
    vmax = float(v.float().abs().max())
    err = max_abs(o.cpu(), o_ref)
    record("wide scores bf16", o_max_abs=err, o_rel_l2=rel_l2(o.cpu(), o_ref),
           lse_max_abs=max_abs(lse.cpu(), lse_ref))
    assert err <= (2.0 ** -7 + 2.0 ** -8) * vmax, (err, vmax)
    assert rel_l2(o.cpu(), o_ref) <= 5e-3
    assert max_abs(lse.cpu(), lse_ref) <= 1e-3


FULL = ["gpt_layer", "gpt_layer_causal", "long_seq", "head256", "gqa8k"]


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(name):
    """Full-size workloads: whole outputs of two (batch, kv-head) groups and
    sampled rows of others against the oracle."""
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), w.causal, w.scale)
    binding.device_status()
    o, lse = o.cpu(), lse.cpu()
    G = w.H // w.Hkv
    rng = np.random.default_rng(w.seed)
    groups = [(0, 0), (w.B - 1, w.Hkv - 1)]
    for (b, kh) in groups:
        sl = slice(kh * G, (kh + 1) * G)
        o_ref, lse_ref = oracle.forward_group(q[b, sl], k[b, kh], v[b, kh], w.causal, w.scale)
        check_forward(o[b, sl], lse[b, sl], o_ref, lse_ref, f"{name} group b{b} kh{kh}")
    for _ in range(4):
        b, kh = int(rng.integers(w.B)), int(rng.integers(w.Hkv))
        rows = [(int(rng.integers(G)), int(i)) for i in rng.integers(0, w.N, 16)]
        rows += [(0, w.N - 1), (G - 1, 0)]
        o_ref, lse_ref = oracle.forward_rows(q[b, kh * G:(kh + 1) * G], k[b, kh], v[b, kh], rows,
                                             w.causal, w.scale)
        got_o = torch.stack([o[b, kh * G + g, i] for g, i in rows])
        got_l = torch.stack([lse[b, kh * G + g, i] for g, i in rows])
        check_forward(got_o, got_l, o_ref, lse_ref, f"{name} rows b{b} kh{kh}")


# (B, H, Hkv, Nq, Nk, causal): several 256-row units per CTA (300 units), and
# with Nk = 40000 (20 MB of K and V per KV head) causal (batch, head) pairs
# split over two sections of the longest-first order
PERSISTENT = [(3, 20, 5, 1100, 1100, False), (3, 20, 5, 1100, 1100, True),
              (1, 8, 4, 700, 40000, True), (2, 8, 2, 1500, 1300, True)]


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,causal", PERSISTENT)
def test_forward_every_unit_sampled(B, H, Hkv, Nq, Nk, causal):
    """The two-query-tile forward walks (batch, head, 256-row block) units in
    a persistent loop: rows from every unit (first, last and random rows of
    both 128-row tiles) against the oracle, plus one whole group."""
    w = Workload("units", B, H, Hkv, Nq, 128, "bf16", causal, 31 + Nq + Nk + B)
    q, k, v, _ = make_inputs(w, Nk=Nk)
    o, lse = binding.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal, w.scale)
    binding.device_status()
    o, lse = o.cpu(), lse.cpu()
    G = H // Hkv
    rng = np.random.default_rng(B * 1000 + Nq)

    def check(got_o, got_l, o_ref, lse_ref, what):
        # rows that see no key (Nq > Nk under the mask): O = 0 and L = -inf
        got_l, lse_ref = got_l.double().numpy().copy(), np.asarray(lse_ref).copy()
        empty = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(got_l), empty), what
        assert torch.all(got_o[torch.from_numpy(empty)] == 0), what
        got_l[empty] = 0.0
        lse_ref[empty] = 0.0
        check_forward(got_o, got_l, o_ref, lse_ref, what)

    if Nk <= 2000:
        o_ref, lse_ref = oracle.forward_group(q[0, :G], k[0, 0], v[0, 0], causal, w.scale)
        check(o[0, :G], lse[0, :G], o_ref, lse_ref, "units whole group b0 kh0")
    for b in range(B):
        for kh in range(Hkv):
            rows = []
            for g in range(G):
                for start in range(0, Nq, 128):
                    end = min(start + 128, Nq)
                    rows += [(g, start), (g, end - 1), (g, int(rng.integers(start, end)))]
            o_ref, lse_ref = oracle.forward_rows(q[b, kh * G:(kh + 1) * G], k[b, kh], v[b, kh],
                                                 rows, causal, w.scale)
            got_o = torch.stack([o[b, kh * G + g, i] for g, i in rows])
            got_l = torch.stack([lse[b, kh * G + g, i] for g, i in rows])
            check(got_o, got_l, o_ref, lse_ref, f"units b{b} kh{kh} {Nq}x{Nk}")
