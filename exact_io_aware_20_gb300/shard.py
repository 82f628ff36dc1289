"""Splitting one attention problem across ranks (one process per GPU).

The work units of both passes are the (batch, key/value head) groups: a key/
value head and the G = H / Hkv query heads that read it.  Forward query tiles
are independent ("FlashAttention-2: Faster Attention with Better Parallelism
and Work Partitioning", paper digest, section 4 "six checks": no dependence
between query blocks), and a group carries all of its dK/dV sums (same
section, GQA/MQA line), so groups need no exchange: ranks take contiguous
ranges of groups and no collective runs on the data path.

In the [B, H, N, d] / [B, Hkv, N, d] layouts the groups are contiguous in
memory in (b, kv-head) order, so a range of groups is a plain view shaped as
one batch with (u1 - u0) key/value heads.
"""
from __future__ import annotations


def unit_range(B: int, Hkv: int, rank: int, world: int):
    """Contiguous, balanced range [u0, u1) of the B*Hkv groups for `rank`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    units = B * Hkv
    base, extra = divmod(units, world)
    u0 = rank * base + min(rank, extra)
    return u0, u0 + base + (1 if rank < extra else 0)


def shard_views(q, k, v, u0: int, u1: int, *more_q):
    """Views of groups [u0, u1): q-like tensors [B,H,N,d] -> [1, (u1-u0)*G, N, d],
    k, v [B,Hkv,N,d] -> [1, u1-u0, N, d].  Extra q-shaped tensors (o, dO, dQ, ...)
    and lse-shaped [B,H,N] tensors in `more_q` are cut the same way."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    n = u1 - u0

    def cut_q(t):
        if t.dim() == 4:
            return t.reshape(B * Hkv, G, N, t.shape[-1])[u0:u1].reshape(1, n * G, N, t.shape[-1])
        return t.reshape(B * Hkv, G, N)[u0:u1].reshape(1, n * G, N)

    def cut_kv(t):
        return t.reshape(B * Hkv, N, t.shape[-1])[u0:u1].reshape(1, n, N, t.shape[-1])

    return (cut_q(q), cut_kv(k), cut_kv(v)) + tuple(cut_q(t) for t in more_q)
