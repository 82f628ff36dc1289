"""Model of the d = 256 cluster-pair backward kernel's barrier protocol,
checked on random step counts and interleavings (no GPU).

Two CTAs, each with its own in-order tensor pipe (a commit arrives once every
product queued before it in that CTA has completed), its own TMA loads
(completing in any order) and its own barriers; remote arrivals and stores
cross between them.  Rank 0 forms S^T, writes P^T over it (TMEM) and sends
P^T to rank 1's shared memory; rank 1 forms dP^T, reads the received P^T and
writes dS^T over dP^T; each CTA's accumulator product reads the 16-bit tile
from TMEM and its Z operand (dO on rank 0, Q on rank 1).  Every region
carries a label of what was last written there, and each reader (a product
when it runs, a warp when it reads) asserts the label of the step it works on.
Each CTA's two streamed operands pass through one ring of chunk slots (ten
on rank 0; on rank 1 what the P^T buffers leave) in the order its MMA warp
reads them (the accumulator product reads an aligned pair of slots).  The
exchange runs warp to warp through one or two buffers: sender warp (h, w) of
rank 0 writes step t's rows into its own copy of buffer t % PBUF and sends
them as one bulk copy into rank 1's, which receiver warp (h, w) of rank 1
reads (the copy's source must hold the rows until the copy lands, and only
rank 1's release of the buffer tells rank 0 that it has); the bytes complete
on the receiver's IN_FULL of that buffer, whose phase also needs the receiver's own expect_tx (made for step
t + PBUF before it releases step t's rows on rank 0's OUT_FREE).  The model is at
warp granularity: OUT_FREE, which the kernel counts in threads, counts the
warp here.
"""
import random

import pytest

from test_bwd_protocol_cpu import Bar


def run_pair(n, seed, plant=None, ld_slots=3, ring=(10, 6), pbuf=2, slow=False, land_p=0.1,
             limit=400_000):
    """Returns True when both CTAs finish; False on a hang (the roles stop
    making progress); raises AssertionError on a wrong read.  slow: rank 1's
    dS warps get a fifth of the other roles' turns; land_p: the chance per
    turn that an exchanged block of rows lands."""
    rnd = random.Random(seed)
    B = {}
    for r in (0, 1):
        B[r, "Stat"] = Bar(1)
        for c in range(ring[r]):
            B[r, f"RF{c}"] = Bar(1)
            B[r, f"RE{c}"] = Bar(1)
        for s in (0, 1):
            B[r, f"SF{s}"] = Bar(1)
            B[r, f"PF{s}"] = Bar(8)
        for h in (0, 1):
            for w in range(4):
                for pb in range(pbuf):
                    B[r, f"IN{h}{w}{pb}"] = Bar(2)   # the receiver's expect_tx, the bytes landing
                    B[r, f"OUT{h}{w}{pb}"] = Bar(1)
        B[r, "Final"] = Bar(1)
    content = {}
    loads = {0: [], 1: []}
    pipes = {0: [], 1: []}
    tag16 = {0: "P16", 1: "dS16"}
    rx = []                                    # sent rows whose bytes have not landed
    expect = {(h, w, pb): 0 for h in (0, 1) for w in range(4) for pb in range(pbuf)}

    def wait(key, parity):
        while not B[key].done(parity):
            yield

    def queued(r, region, write_only):
        for op in pipes[r]:
            if op[0] != "mma":
                continue
            if region in op[2] or (not write_only and region in op[1]):
                return True
        return False

    def producer(r):
        content[r, "stat"] = None
        loads[r].append(((r, "Stat"), (r, "stat"), "unit"))
        ci = 0

        def tile(kind, t):
            nonlocal ci
            for c in range(4):
                slot = ci % ring[r]
                if ci >= ring[r]:
                    yield from wait((r, f"RE{slot}"), ((ci // ring[r]) - 1) & 1)
                loads[r].append(((r, f"RF{slot}"), (r, "ring", slot), (kind, t, c)))
                ci += 1
                yield
        for t in range(n):
            yield from tile("A", t)
            if t >= 1:
                yield from tile("B", t - 1)
        if n > 0:
            yield from tile("B", n - 1)

    def mma(r):
        ci = 0

        def score(t):
            nonlocal ci
            buf = [(r, "buf", t & 1, h, w) for h in (0, 1) for w in range(4)]
            for c in range(4):
                slot = ci % ring[r]
                yield from wait((r, f"RF{slot}"), (ci // ring[r]) & 1)
                checks = {(r, "stat"): "unit", (r, "ring", slot): ("A", t, c)}
                sets = {x: ("S", t) for x in buf} if c == 3 else {}
                pipes[r].append(("mma", [(r, "stat"), (r, "ring", slot)], buf, checks, sets))
                pipes[r].append(("commit", (r, f"RE{slot}")))
                ci += 1
            pipes[r].append(("commit", (r, f"SF{t & 1}")))

        def acc(t):
            nonlocal ci
            yield from wait((r, f"PF{t & 1}"), (t >> 1) & 1)
            buf = [(r, "buf", t & 1, h, w) for h in (0, 1) for w in range(4)]
            for dh in (0, 1):
                slot = ci % ring[r]
                assert slot + 1 < ring[r], "an operand pair straddles the end of the ring"
                yield from wait((r, f"RF{slot}"), (ci // ring[r]) & 1)
                yield from wait((r, f"RF{slot + 1}"), ((ci + 1) // ring[r]) & 1)
                checks = {x: (tag16[r], t) for x in buf}
                checks[r, "ring", slot] = ("B", t, 2 * dh)
                checks[r, "ring", slot + 1] = ("B", t, 2 * dh + 1)
                pipes[r].append(("mma", buf + [(r, "ring", slot), (r, "ring", slot + 1)],
                                 [(r, "acc")], checks, {}))
                pipes[r].append(("commit", (r, f"RE{slot}")))
                pipes[r].append(("commit", (r, f"RE{slot + 1}")))
                ci += 2

        yield from wait((r, "Stat"), 0)
        for t in range(n):
            if plant == "score_early" and r == 0 and t >= 1:
                # the next scores before this step's accumulator product
                if t == 1:
                    yield from score(0)
                    yield from score(1)
                elif t + 1 < n:
                    yield from score(t + 1)
                yield from acc(t - 1)
                continue
            yield from score(t)
            if t >= 1:
                yield from acc(t - 1)
        if plant == "score_early" and n == 1:
            yield from score(0)
        if n > 0:
            yield from acc(n - 1)
        pipes[r].append(("commit", (r, "Final")))

    def warp(r, h, w):
        ld = lambda t: (r, "ld", h, t % ld_slots)
        content[ld(0)] = ("LD", 0)
        for t in range(n):
            pb, use = t % pbuf, t // pbuf
            assert content.get(ld(t)) == ("LD", t), "L / D values of another step"
            buf = (r, "buf", t & 1, h, w)   # this warp's lane quarter and half

            def read_scores():
                assert content.get(buf) == ("S", t), "scores of another step in TMEM"
                assert not queued(r, buf, write_only=True), "TMEM read while a product writes it"
            if r == 0:
                yield from wait((r, f"SF{t & 1}"), (t >> 1) & 1)
                read_scores()
                yield
                assert not queued(r, buf, write_only=False), "TMEM write while a product uses it"
                content[buf] = ("P16", t)
                # the L / D values are read until here
                assert content.get(ld(t)) == ("LD", t), "L / D values of another step"
                B[r, f"PF{t & 1}"].arrive()       # before the rows are sent
                yield
                if plant == "stage_before_outfree":
                    content[0, "stage", h, w, pb] = ("P", t)
                    yield
                if t >= pbuf and plant != "no_outfree_wait":
                    yield from wait((0, f"OUT{h}{w}{pb}"), (use - 1) & 1)
                content[0, "stage", h, w, pb] = ("P", t)   # this CTA's copy of the rows
                rx.append((h, w, pb, t))       # one bulk copy: reads that copy, lands later
                yield
            else:
                if plant != "no_infull_wait":
                    yield from wait((1, f"IN{h}{w}{pb}"), use & 1)
                assert content.get((1, "pin", h, w, pb)) == ("P", t), "P^T of another step received"
                yield
                if plant == "release_first":
                    B[0, f"OUT{h}{w}{pb}"].arrive()
                    yield
                if t + pbuf < n:
                    expect[h, w, pb] += 1
                    B[1, f"IN{h}{w}{pb}"].arrive()    # expect_tx of step t + pbuf
                if plant != "release_first":
                    B[0, f"OUT{h}{w}{pb}"].arrive()
                yield from wait((1, f"SF{t & 1}"), (t >> 1) & 1)
                read_scores()
                yield
                if plant == "early_pfull":
                    B[r, f"PF{t & 1}"].arrive()
                    yield
                assert not queued(r, buf, write_only=False), "TMEM write while a product uses it"
                content[buf] = ("dS16", t)
                yield
            if r == 1:
                # the L / D values are read until here
                assert content.get(ld(t)) == ("LD", t), "L / D values of another step"
                if plant != "early_pfull":
                    B[r, f"PF{t & 1}"].arrive()
            if t + 1 < n:
                content[ld(t + 1)] = ("LD", t + 1)
            yield
        yield from wait((r, "Final"), 0)
        assert not queued(r, (r, "acc"), write_only=True), "accumulator read before its last product"

    def land(i):
        h, w, pb, t = rx.pop(i)
        assert expect[h, w, pb] >= t // pbuf + 1, "rows landed before the receiver expected them"
        assert content.get((0, "stage", h, w, pb)) == ("P", t), \
            "the bulk copy's source was overwritten before the copy had read it"
        content[1, "pin", h, w, pb] = ("P", t)
        B[1, f"IN{h}{w}{pb}"].arrive()

    def run_pipe(r):
        op = pipes[r].pop(0)
        if op[0] == "commit":
            B[op[1]].arrive()
        else:
            for region, label in op[3].items():
                assert content.get(region) == label, f"{region} holds {content.get(region)}"
            content.update(op[4])

    def land_load(r, i):
        bar, region, label = loads[r].pop(i)
        content[region] = label
        B[bar].arrive()

    # rank 1 expects the rows of steps 0 and 1 before the cluster meets
    for h in (0, 1):
        for w in range(4):
            for pb in range(min(n, pbuf)):
                expect[h, w, pb] += 1
                B[1, f"IN{h}{w}{pb}"].arrive()
    roles = []
    for r in (0, 1):
        roles += [producer(r), mma(r)]
        roles += [warp(r, h, w) for h in (0, 1) for w in range(4)]
    alive = list(range(len(roles)))
    slow_roles = set(range(len(roles) - 8, len(roles)))     # rank 1's dS warps
    for _ in range(limit):
        if not alive and not any(loads.values()) and not any(pipes.values()) and not rx:
            return True
        x = rnd.random()
        r = rnd.randrange(2)
        if rx and rnd.random() < land_p:
            land(rnd.randrange(len(rx)))
        elif loads[r] and x < 0.2:
            land_load(r, rnd.randrange(len(loads[r])))
        elif pipes[r] and x < 0.45:
            run_pipe(r)
        elif alive:
            k = rnd.choice(alive)
            if slow and k in slow_roles and rnd.random() > 0.2:
                others = [i for i in alive if i not in slow_roles]
                if others:
                    k = rnd.choice(others)
            try:
                next(roles[k])
            except StopIteration:
                alive.remove(k)
        elif rx:
            land(0)
        elif loads[r]:
            land_load(r, 0)
        elif pipes[r]:
            run_pipe(r)
    return False


@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("ring,pbuf", [((10, 6), 2), ((10, 8), 1), ((8, 8), 1), ((6, 6), 2)])
def test_pair_protocol(seed, ring, pbuf):
    n = [1, 2, 3, 5, 8][seed % 5]
    assert run_pair(n, seed, ring=ring, pbuf=pbuf, slow=seed % 4 == 3)


@pytest.mark.parametrize("plant", ["no_outfree_wait", "no_infull_wait", "early_pfull",
                                   "score_early", "two_ld_slots", "release_first", "odd_ring",
                                   "stage_before_outfree"])
def test_pair_protocol_catches(plant):
    """Each planted mistake produces a wrong read or a hang on some seed."""
    caught = False
    for seed in range(60):
        try:
            ok = run_pair(6, seed, plant=None if plant in ("two_ld_slots", "odd_ring") else plant,
                          ld_slots=2 if plant == "two_ld_slots" else 3,
                          ring=(10, 5) if plant == "odd_ring" else (10, 6), slow=seed % 2 == 1,
                          land_p=0.1 if seed % 3 else 0.01)
        except AssertionError:
            caught = True
            break
        if not ok:
            caught = True
            break
    assert caught, plant
