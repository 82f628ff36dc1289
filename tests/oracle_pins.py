"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes a loaded oracle library (so the same checks can
be run against deliberately broken copies of the oracle, see
``test_oracle_mutants.py``) and raises ``AssertionError`` on a mismatch.

What pins what:
  closed forms      identical keys, zero queries, one dominant score, the
                    first causal row, the hand-solved d=1, N=2 case (forward
                    and gradients, from the two-key sigmoid form)
  invariants        rows of P sum to 1 and P = exp(S - L) (read off with
                    V = I), L equals a long-double logsumexp, permutation of
                    keys, shift of all keys by one vector, GQA equals MHA with
                    repeated K/V, D = rowsum(dO o O); summed over the keys,
                    dV equals the summed dO of the rows that see a key and
                    dK is zero
  derivatives       central finite differences of sum(O o dO)
  library routines  torch fp64 softmax/matmul and torch.autograd gradients
  bottom-right mask Nq != Nk rows, including rows with no allowed key
  block mask        an all-ones mask is the dense result bit for bit; a query
                    block that keeps one key block is dense attention over
                    that key slice; torch fp64 with the block mask expanded
                    to an element mask (shared and per-head masks, GQA,
                    causal, ragged edges, fully masked rows)

Block-sparse attention ("FlashAttention: Fast and Memory-Efficient Exact
Attention with IO-Awareness", abstract and "Key contributions") is read as
exact attention restricted to the kept blocks of a given pattern.

The attention definition these follow: "FlashAttention-2: Faster Attention
with Better Parallelism and Work Partitioning" (paper digest), section 3
"Target operation", section 4 notation table (L = m + log l, D) and the GQA
line of section 4 "six checks".
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _allowed(i, k, Nq, Nk, causal):
    return (not causal) or k <= i + (Nk - Nq)


def pin_identical_keys(lib):
    """All key rows equal -> uniform weights over the allowed keys."""
    rng = _rng(1)
    for causal in (False, True):
        G, N, d = 2, 13, 8
        q = _rand(rng, G, N, d)
        krow = _rand(rng, d)
        k = np.tile(krow, (N, 1))
        v = _rand(rng, N, d)
        scale = 0.7
        o, lse = oracle.forward_group(q, k, v, causal, scale, lib)
        for g in range(G):
            for i in range(N):
                n_allowed = (i + 1) if causal else N
                s = scale * float(q[g, i] @ krow)
                np.testing.assert_allclose(o[g, i], v[:n_allowed].mean(axis=0), rtol=0, atol=1e-12)
                assert abs(lse[g, i] - (s + math.log(n_allowed))) < 1e-12


def pin_zero_queries(lib):
    """Q = 0 -> L = ln(#allowed keys), O = mean of allowed V rows."""
    rng = _rng(2)
    for causal in (False, True):
        N, d = 17, 4
        q = np.zeros((1, N, d))
        k = _rand(rng, N, d)
        v = _rand(rng, N, d)
        o, lse = oracle.forward_group(q, k, v, causal, 1.3, lib)
        for i in range(N):
            n = (i + 1) if causal else N
            assert abs(lse[0, i] - math.log(n)) < 1e-13
            np.testing.assert_allclose(o[0, i], v[:n].mean(axis=0), rtol=0, atol=1e-12)


def pin_dominant_score(lib):
    """One key with a score 60 above every other selects its value row."""
    rng = _rng(3)
    N, d, kstar = 24, 6, 5
    k = _rand(rng, N, d)
    k[:, 0] = 0.0
    k[kstar, 0] = 1.0
    v = _rand(rng, N, d)
    scale = 0.25
    q = np.zeros((1, N, d))
    q[0, :, 0] = 60.0 / scale
    for causal in (False, True):
        o, lse = oracle.forward_group(q, k, v, causal, scale, lib)
        for i in range(kstar, N):
            n = (i + 1) if causal else N
            # weight of every other key is exp(-60) / (1 + (n-1) exp(-60))
            tail = (n - 1) * math.exp(-60.0) * float(np.abs(v).max()) * 2
            np.testing.assert_allclose(o[0, i], v[kstar], rtol=0, atol=tail + 1e-13)
            assert abs(lse[0, i] - 60.0) < n * math.exp(-60.0) + 1e-12


def pin_causal_first_row(lib):
    """Under the causal mask query 0 sees only key 0: O_0 = V_0, L_0 = S_00."""
    rng = _rng(4)
    G, N, d = 3, 9, 5
    q = _rand(rng, G, N, d)
    k = _rand(rng, N, d)
    v = _rand(rng, N, d)
    o, lse = oracle.forward_group(q, k, v, True, 0.9, lib)
    for g in range(G):
        np.testing.assert_allclose(o[g, 0], v[0], rtol=0, atol=1e-14)
        assert abs(lse[g, 0] - 0.9 * float(q[g, 0] @ k[0])) < 1e-14


def _two_key_case():
    # d = 1, N = 2, scale = 1: row i has scores (q_i k_0, q_i k_1), so the
    # weight of key 0 is sigmoid(q_i (k_0 - k_1)).
    q = np.array([1.0, -2.0])
    k = np.array([0.5, 1.5])
    v = np.array([2.0, -1.0])
    dout = np.array([1.0, -0.5])
    return q, k, v, dout


def pin_two_keys_forward(lib):
    """d=1, N=2 by hand, and the printed values in tests/golden/two_keys.txt."""
    q, k, v, _ = _two_key_case()
    o, lse = oracle.forward_group(q.reshape(1, 2, 1), k.reshape(2, 1), v.reshape(2, 1),
                                  False, 1.0, lib)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    for i in range(2):
        w0 = sig(q[i] * (k[0] - k[1]))
        assert abs(o[0, i, 0] - (w0 * v[0] + (1 - w0) * v[1])) < 1e-15
        a, b = q[i] * k[0], q[i] * k[1]
        assert abs(lse[0, i] - (max(a, b) + math.log1p(math.exp(-abs(a - b))))) < 1e-15
    # values worked out by hand (tests/golden/two_keys.txt)
    assert abs(o[0, 0, 0] - (-0.1931757358900147)) < 1e-15
    assert abs(o[0, 1, 0] - 1.642391233933647) < 1e-15
    assert abs(lse[0, 0] - 1.8132616875182228) < 1e-15
    assert abs(lse[0, 1] - (-0.8730719889570275)) < 1e-15
    # causal: row 0 sees key 0 only
    oc, lc = oracle.forward_group(q.reshape(1, 2, 1), k.reshape(2, 1), v.reshape(2, 1),
                                  True, 1.0, lib)
    assert oc[0, 0, 0] == 2.0 and lc[0, 0] == 0.5
    assert abs(oc[0, 1, 0] - o[0, 1, 0]) < 1e-15


def pin_two_keys_backward(lib):
    """Gradients of the d=1, N=2 case from the sigmoid form, by hand.

    O_i = w_i v_0 + (1 - w_i) v_1, w_i = sigmoid(q_i (k_0 - k_1)), so with
    c_i = dO_i (v_0 - v_1) w_i (1 - w_i):
      dV_0 = sum_i dO_i w_i, dV_1 = sum_i dO_i (1 - w_i),
      dQ_i = c_i (k_0 - k_1), dK_0 = sum_i c_i q_i = -dK_1.
    """
    q, k, v, dout = _two_key_case()
    dq, dk, dv = oracle.backward_group(q.reshape(1, 2, 1), k.reshape(2, 1), v.reshape(2, 1),
                                       dout.reshape(1, 2, 1), False, 1.0, lib)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    w = [sig(q[i] * (k[0] - k[1])) for i in range(2)]
    c = [dout[i] * (v[0] - v[1]) * w[i] * (1 - w[i]) for i in range(2)]
    assert abs(dv[0, 0] - sum(dout[i] * w[i] for i in range(2))) < 1e-15
    assert abs(dv[1, 0] - sum(dout[i] * (1 - w[i]) for i in range(2))) < 1e-15
    for i in range(2):
        assert abs(dq[0, i, 0] - c[i] * (k[0] - k[1])) < 1e-15
    dk0 = sum(c[i] * q[i] for i in range(2))
    assert abs(dk[0, 0] - dk0) < 1e-15 and abs(dk[1, 0] + dk0) < 1e-15


def pin_rows_are_probabilities(lib):
    """With V = I the output rows are the weights: sum to 1, equal exp(S - L)."""
    rng = _rng(5)
    for causal in (False, True):
        N = d = 16
        q = _rand(rng, 2, N, d)
        k = _rand(rng, N, d)
        v = np.eye(N)
        scale = 0.5
        o, lse = oracle.forward_group(q, k, v, causal, scale, lib)
        np.testing.assert_allclose(o.sum(axis=-1), 1.0, rtol=0, atol=1e-13)
        for g in range(2):
            s = scale * (q[g].astype(np.longdouble) @ k.astype(np.longdouble).T)
            for i in range(N):
                row = [s[i, kk] for kk in range(N) if _allowed(i, kk, N, N, causal)]
                m = max(row)
                L = m + np.log(sum(np.exp(x - m) for x in row))
                assert abs(float(L) - lse[g, i]) < 1e-13
                for kk in range(N):
                    want = float(np.exp(s[i, kk] - L)) if _allowed(i, kk, N, N, causal) else 0.0
                    assert abs(o[g, i, kk] - want) < 1e-14


def pin_permutation_and_shift(lib):
    """Non-causal O is invariant under a joint permutation of K and V rows;
    adding one vector c to every key row leaves O alone and moves L_i by
    scale * q_i . c (masked or not)."""
    rng = _rng(6)
    G, N, d = 2, 21, 8
    q = _rand(rng, G, N, d)
    k = _rand(rng, N, d)
    v = _rand(rng, N, d)
    scale = 0.35
    o, lse = oracle.forward_group(q, k, v, False, scale, lib)
    perm = rng.permutation(N)
    op, lp = oracle.forward_group(q, k[perm], v[perm], False, scale, lib)
    np.testing.assert_allclose(op, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, lse, rtol=0, atol=1e-12)
    c = _rand(rng, d)
    for causal in (False, True):
        o1, l1 = oracle.forward_group(q, k, v, causal, scale, lib)
        o2, l2 = oracle.forward_group(q, k + c, v, causal, scale, lib)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-11)
        np.testing.assert_allclose(l2 - l1, scale * (q @ c), rtol=0, atol=1e-11)


def pin_gqa_equals_repeated_mha(lib):
    """GQA with G heads per KV head equals MHA with K, V repeated; the GQA
    dK/dV are the sums of the G per-head MHA gradients."""
    rng = _rng(7)
    B, H, Hkv, N, d = 2, 4, 2, 11, 6
    q = _rand(rng, B, H, N, d)
    k = _rand(rng, B, Hkv, N, d)
    v = _rand(rng, B, Hkv, N, d)
    do = _rand(rng, B, H, N, d)
    G = H // Hkv
    kr = np.repeat(k, G, axis=1)
    vr = np.repeat(v, G, axis=1)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, causal, 0.4, lib)
        o2, l2 = oracle.forward(q, kr, vr, causal, 0.4, lib)
        np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, l2, rtol=0, atol=1e-13)
        dq, dk, dv = oracle.backward(q, k, v, do, causal, 0.4, lib)
        dq2, dk2, dv2 = oracle.backward(q, kr, vr, do, causal, 0.4, lib)
        np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, G, N, d).sum(axis=2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, G, N, d).sum(axis=2), rtol=0, atol=1e-12)


def pin_delta_and_extras(lib):
    """The backward's own O and L match the forward; D = rowsum(dO o O)."""
    rng = _rng(8)
    G, N, d = 2, 10, 4
    q, k, v, do = _rand(rng, G, N, d), _rand(rng, N, d), _rand(rng, N, d), _rand(rng, G, N, d)
    for causal in (False, True):
        _, _, _, o, lse, delta = oracle.backward_group(q, k, v, do, causal, 0.6, lib, extras=True)
        of, lf = oracle.forward_group(q, k, v, causal, 0.6, lib)
        np.testing.assert_allclose(o, of, rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse, lf, rtol=0, atol=1e-14)
        np.testing.assert_allclose(delta, (do * of).sum(-1), rtol=0, atol=1e-13)


def pin_gradient_sums(lib):
    """Sums over the keys of a group's gradients: sum_k dV_k = the sum of dO
    over the rows that see a key (every row of P sums to 1, dV = P^T dO) and
    sum_k dK_k = 0 (every row of dS = P o (dP - D) sums to 0, because
    sum_k P_ik dP_ik = dO_i . O_i = D_i), with and without the mask, Nq != Nk
    included."""
    rng = _rng(21)
    for causal, Nq, Nk in ((False, 11, 11), (True, 11, 11), (True, 9, 6), (True, 6, 9)):
        G, d = 3, 5
        q, k, v = _rand(rng, G, Nq, d), _rand(rng, Nk, d), _rand(rng, Nk, d)
        do = _rand(rng, G, Nq, d)
        _, dk, dv = oracle.backward_group(q, k, v, do, causal, 0.7, lib)
        seen = np.array([any(_allowed(i, kk, Nq, Nk, causal) for kk in range(Nk))
                         for i in range(Nq)], dtype=np.float64)
        np.testing.assert_allclose(dv.sum(0), (do * seen[None, :, None]).sum((0, 1)), rtol=0,
                                   atol=1e-12)
        np.testing.assert_allclose(dk.sum(0), np.zeros(d), rtol=0, atol=1e-12)


def _fd_check(lib, G, Nq, Nk, d, causal, seed):
    rng = _rng(seed)
    q, k, v = _rand(rng, G, Nq, d), _rand(rng, Nk, d), _rand(rng, Nk, d)
    do = _rand(rng, G, Nq, d)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = oracle.backward_group(q, k, v, do, causal, scale, lib)

    def f(q_, k_, v_):
        o, _ = oracle.forward_group(q_, k_, v_, causal, scale, lib)
        return float((o * do).sum())

    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        err = np.abs(num - grad).max() / max(1.0, np.abs(grad).max())
        assert err < 1e-6, f"finite differences d{name}: rel err {err}"


def pin_finite_differences(lib):
    for (G, Nq, Nk, d, causal, seed) in ((1, 7, 7, 4, False, 10), (2, 9, 9, 3, True, 11),
                                         (2, 5, 8, 4, True, 12), (1, 16, 16, 8, True, 13)):
        _fd_check(lib, G, Nq, Nk, d, causal, seed)


def _torch_reference(q, k, v, do, causal, scale, keep=None):
    """torch fp64: explicit matmul + torch.softmax, autograd for the gradients.
    keep (optional, bool [H or 1, Nq, Nk]): element mask; rows it empties get
    O = 0, L = -inf and zero gradients."""
    q = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    G = q.shape[1] // k.shape[1]
    kr = k.repeat_interleave(G, dim=1)
    vr = v.repeat_interleave(G, dim=1)
    s = scale * torch.matmul(q, kr.transpose(-1, -2))
    Nq, Nk = s.shape[-2], s.shape[-1]
    if causal:
        i = torch.arange(Nq).view(-1, 1)
        kk = torch.arange(Nk).view(1, -1)
        s = s.masked_fill(kk > i + (Nk - Nq), float("-inf"))
    if keep is not None:
        s = s.masked_fill(~torch.as_tensor(keep), float("-inf"))
    empty = torch.isneginf(s).all(dim=-1, keepdim=True)
    p = torch.softmax(s.masked_fill(empty, 0.0), dim=-1).masked_fill(empty, 0.0)
    lse = torch.logsumexp(s, dim=-1)
    o = torch.matmul(p, vr)
    (o * torch.tensor(do)).sum().backward()
    return (o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(),
            v.grad.numpy())


def pin_torch_fp64(lib):
    """Agreement with torch fp64 softmax/autograd on small inputs (1e-12)."""
    rng = _rng(20)
    for (B, H, Hkv, Nq, Nk, d, causal) in ((1, 2, 2, 9, 9, 8, False), (2, 4, 1, 13, 13, 16, True),
                                           (1, 4, 2, 33, 33, 8, True), (1, 2, 1, 6, 11, 4, True),
                                           (1, 1, 1, 1, 7, 4, True)):
        q, k, v = _rand(rng, B, H, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
        do = _rand(rng, B, H, Nq, d)
        scale = 1.0 / math.sqrt(d)
        o_t, l_t, dq_t, dk_t, dv_t = _torch_reference(q, k, v, do, causal, scale)
        o, lse = oracle.forward(q, k, v, causal, scale, lib)
        dq, dk, dv = oracle.backward(q, k, v, do, causal, scale, lib)
        for a, b in ((o, o_t), (lse, l_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def pin_bottom_right_mask(lib):
    """Nq != Nk under the mask: query i sees keys k <= i + Nk - Nq; a query
    with no key left has O = 0, L = -inf and zero gradient."""
    rng = _rng(21)
    # Nq < Nk (decode-like): the last query sees every key.
    q, k, v = _rand(rng, 1, 3, 4), _rand(rng, 8, 4), _rand(rng, 8, 4)
    o, lse = oracle.forward_group(q, k, v, True, 0.5, lib)
    of, lf = oracle.forward_group(q[:, 2:], k, v, False, 0.5, lib)
    np.testing.assert_allclose(o[:, 2], of[:, 0], rtol=0, atol=1e-14)
    o0, l0 = oracle.forward_group(q[:, :1], k[:6], v[:6], False, 0.5, lib)
    np.testing.assert_allclose(o[:, 0], o0[:, 0], rtol=0, atol=1e-14)
    # Nq > Nk: the first Nq - Nk queries have no key.
    q, k, v = _rand(rng, 1, 6, 4), _rand(rng, 4, 4), _rand(rng, 4, 4)
    do = _rand(rng, 1, 6, 4)
    o, lse = oracle.forward_group(q, k, v, True, 0.5, lib)
    assert np.all(o[0, :2] == 0.0) and np.all(np.isneginf(lse[0, :2]))
    assert abs(lse[0, 2] - 0.5 * float(q[0, 2] @ k[0])) < 1e-14
    dq, dk, dv = oracle.backward_group(q, k, v, do, True, 0.5, lib)
    assert np.all(dq[0, :2] == 0.0) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def pin_rows_match_group(lib):
    """forward_rows returns the same rows as the whole-group forward."""
    rng = _rng(22)
    G, N, d = 3, 40, 8
    q, k, v = _rand(rng, G, N, d), _rand(rng, N, d), _rand(rng, N, d)
    rows = [(0, 0), (2, 39), (1, 17), (2, 5)]
    for causal in (False, True):
        o, lse = oracle.forward_group(q, k, v, causal, 0.3, lib)
        orows, lrows = oracle.forward_rows(q, k, v, rows, causal, 0.3, lib)
        for t, (g, i) in enumerate(rows):
            assert np.array_equal(orows[t], o[g, i]) and lrows[t] == lse[g, i]


def pin_row_slabs_sum_to_group(lib):
    """backward_rows over a partition of the query rows reproduces the whole
    group's gradients (the sums over rows split exactly)."""
    rng = _rng(23)
    G, N, d = 2, 19, 5
    q, k, v, do = _rand(rng, G, N, d), _rand(rng, N, d), _rand(rng, N, d), _rand(rng, G, N, d)
    for causal in (False, True):
        dq, dk, dv = oracle.backward_group(q, k, v, do, causal, 0.45, lib)
        dk_s, dv_s = np.zeros((N, d)), np.zeros((N, d))
        dq_s = []
        for (r0, r1) in ((0, 7), (7, 8), (8, 30), (30, 38)):
            dq_part, _, _ = oracle.backward_rows(q, k, v, do, r0, r1, causal, 0.45, dk_s, dv_s, lib)
            dq_s.append(dq_part)
        np.testing.assert_allclose(np.concatenate(dq_s).reshape(G, N, d), dq, rtol=0, atol=1e-13)
        np.testing.assert_allclose(dk_s, dk, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv_s, dv, rtol=0, atol=1e-12)


def _expand_blocks(mask, Nq, Nk, bs):
    """Element mask [h, Nq, Nk] from a block mask [h, ceil(Nq/bs), ceil(Nk/bs)]."""
    m = np.asarray(mask, dtype=bool)
    return np.repeat(np.repeat(m, bs, axis=1), bs, axis=2)[:, :Nq, :Nk]


def pin_blockmask_all_ones_is_dense(lib):
    """An all-ones block mask changes nothing: outputs equal the dense ones bit for bit."""
    rng = _rng(30)
    B, H, Hkv, Nq, Nk, d, bs = 1, 4, 2, 21, 26, 8, 4
    q, k, v = _rand(rng, B, H, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
    do = _rand(rng, B, H, Nq, d)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, causal, 0.4, lib)
        dq, dk, dv = oracle.backward(q, k, v, do, causal, 0.4, lib)
        for heads in (1, H):
            ones = np.ones((heads, -(-Nq // bs), -(-Nk // bs)), dtype=np.uint8)
            ob, lb = oracle.forward_blocksparse(q, k, v, ones, causal, 0.4, bs, lib)
            gb = oracle.backward_blocksparse(q, k, v, do, ones, causal, 0.4, bs, lib)
            assert np.array_equal(ob, o) and np.array_equal(lb, lse)
            for a, b in zip(gb, (dq, dk, dv)):
                assert np.array_equal(a, b)


def pin_blockmask_single_block(lib):
    """A query block that keeps only key block j is dense attention of those
    queries over keys [j*bs, (j+1)*bs); a query block that keeps none has
    O = 0, L = -inf and zero dQ."""
    rng = _rng(31)
    H, N, d, bs = 2, 24, 4, 6
    q, k, v = _rand(rng, 1, H, N, d), _rand(rng, 1, 1, N, d), _rand(rng, 1, 1, N, d)
    do = _rand(rng, 1, H, N, d)
    nb = N // bs
    mask = np.zeros((H, nb, nb), dtype=np.uint8)
    mask[0, 1, 3] = 1     # head 0: query block 1 sees key block 3 only
    mask[1, 2, 0] = 1     # head 1: query block 2 sees key block 0 only
    mask[1, 0, 2] = 1
    o, lse = oracle.forward_blocksparse(q, k, v, mask, False, 0.7, bs, lib)
    for h, qb, kb in ((0, 1, 3), (1, 2, 0), (1, 0, 2)):
        qs = q[0, h, qb * bs:(qb + 1) * bs][None]
        ks, vs = k[0, 0, kb * bs:(kb + 1) * bs], v[0, 0, kb * bs:(kb + 1) * bs]
        od, ld = oracle.forward_group(qs, ks, vs, False, 0.7, lib)
        np.testing.assert_allclose(o[0, h, qb * bs:(qb + 1) * bs], od[0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[0, h, qb * bs:(qb + 1) * bs], ld[0], rtol=0, atol=1e-14)
    assert np.all(o[0, 0, :bs] == 0.0) and np.all(np.isneginf(lse[0, 0, :bs]))
    dq, dk, dv = oracle.backward_blocksparse(q, k, v, do, mask, False, 0.7, bs, lib)
    assert np.all(dq[0, 0, :bs] == 0.0) and np.all(dq[0, 1, bs:2 * bs] == 0.0)
    # key block 1 is kept by no query block of either head
    assert np.all(dk[0, 0, bs:2 * bs] == 0.0) and np.all(dv[0, 0, bs:2 * bs] == 0.0)


def pin_blockmask_torch(lib):
    """Agreement with torch fp64 under the element mask a block mask expands to."""
    rng = _rng(32)
    for (B, H, Hkv, Nq, Nk, d, bs, heads, causal) in (
            (1, 2, 2, 17, 23, 8, 4, 2, False), (2, 4, 2, 20, 20, 4, 4, 4, True),
            (1, 4, 1, 13, 30, 8, 8, 1, True), (1, 3, 3, 30, 11, 4, 5, 3, True),
            (1, 2, 1, 300, 260, 16, 128, 2, False)):
        q, k, v = _rand(rng, B, H, Nq, d), _rand(rng, B, Hkv, Nk, d), _rand(rng, B, Hkv, Nk, d)
        do = _rand(rng, B, H, Nq, d)
        mask = (rng.random((heads, -(-Nq // bs), -(-Nk // bs))) < 0.5).astype(np.uint8)
        mask[0, 0, :] = 0  # one query block with no key at all
        keep = _expand_blocks(mask, Nq, Nk, bs)
        o_t, l_t, dq_t, dk_t, dv_t = _torch_reference(q, k, v, do, causal, 0.35, keep)
        o, lse = oracle.forward_blocksparse(q, k, v, mask, causal, 0.35, bs, lib)
        dq, dk, dv = oracle.backward_blocksparse(q, k, v, do, mask, causal, 0.35, bs, lib)
        np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(l_t))
        fin = np.isfinite(l_t)
        np.testing.assert_allclose(lse[fin], l_t[fin], rtol=0, atol=1e-12)
        for a, b in ((o, o_t), (dq, dq_t), (dk, dk_t), (dv, dv_t)):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


ALL_PINS = [pin_identical_keys, pin_zero_queries, pin_dominant_score, pin_causal_first_row,
            pin_two_keys_forward, pin_two_keys_backward, pin_rows_are_probabilities,
            pin_permutation_and_shift, pin_gqa_equals_repeated_mha, pin_delta_and_extras,
            pin_gradient_sums,
            pin_finite_differences, pin_torch_fp64, pin_bottom_right_mask, pin_rows_match_group,
            pin_row_slabs_sum_to_group, pin_blockmask_all_ones_is_dense,
            pin_blockmask_single_block, pin_blockmask_torch]
