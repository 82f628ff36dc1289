"""Models of the d = 128 backward kernels' barrier protocols, checked on
random step counts and interleavings (no GPU).

Same conventions as the forward model: the roles step by step, tensor-core
products and commits through one in-order queue (a commit arrives once every
product issued before it has completed), mbarrier phase/parity semantics,
TMA loads completing in any order.  Each product records which TMEM region
it reads and writes; a warp reading or writing TMEM asserts that no queued
product writes that region (or, for its writes, reads it).

Key-outer kernel, dK/dV only (TMEM: dV | dK | S^T, with P^T written over it |
dP^T, with dS^T written over it): issue order dV(t), S^T(t+1), dK(t),
dP^T(t+1).  Query-outer dQ kernel (TMEM: two S buffers, with dS written over
them | dP | dQ): issue order S(j+1), [DP_READ(j)] dP(j+1), [DS_FULL(j)]
dQ(j).  This model found that with one DS_FULL barrier a fast dS warp could
arrive for tile j + 1 (dP_{j+1} is issued once every warp has read dP_j)
before a slow one arrived for tile j, completing the phase early; the kernel
alternates two DS_FULL barriers."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def simulate(roles, loads, pipe, B, rnd, content=None, slow=(), limit=2_000_000):
    """content: optional dict, region (TMEM columns or a shared-memory tile)
    -> label of what was last written there: by products given as ("mma",
    reads, writes, label), by loads given as (barrier, tile, label); a queued
    ("check", region, label) asserts, in queue order, that the region holds
    that label when the products after it run.  slow: roles that get a tenth
    of the others' turns (a warp starved by the scheduler).  Returns False
    (a hang) if the roles have not finished after `limit` moves."""
    alive = list(range(len(roles)))
    for _ in range(limit):
        if not alive and not loads and not pipe:
            return True
        r = rnd.random()
        if loads and (r < 0.2 or not alive):
            ld = loads.pop(rnd.randrange(len(loads)))
            if isinstance(ld, tuple):
                content[ld[1]] = ld[2]
                ld = ld[0]
            B[ld].arrive()
        elif pipe and (r < 0.45 or not alive):
            op = pipe.pop(0)
            if op[0] == "commit":
                B[op[1]].arrive()
            elif op[0] == "check":
                what = "K / V of another unit" if op[1] == "KV" else f"{op[1]} of another step"
                assert content.get(op[1]) == op[2], what + " in shared memory or TMEM"
            elif content is not None and len(op) == 4:
                content[op[2]] = op[3]
        elif alive:
            k = rnd.choice(alive)
            fast = [i for i in alive if i not in slow]
            if k in slow and fast and rnd.random() > 0.1:
                k = rnd.choice(fast)
            try:
                next(roles[k])
            except StopIteration:
                alive.remove(k)
    return False


def touches(pipe, region):
    """A queued product reads or writes this TMEM region."""
    return any(op[0] == "mma" and region in op[1:] for op in pipe)


def run_key_outer(n, qs, seed, with_dq=False):
    """with_dq: the block-sparse form, with dS^T in shared memory, dQ^T formed
    in the dP columns and drained by four dQ warps (DQ_FULL / DQ_EMPTY), and
    the dS^T tile released by DS_EMPTY."""
    rnd = random.Random(seed)
    B = {"KV": Bar(1), "DOF": Bar(1), "DOE": Bar(1), "SF": Bar(1), "DPF": Bar(1),
         "Final": Bar(1), "PF": Bar(8), "DSF": Bar(8), "DQF": Bar(1), "DQE": Bar(4),
         "DSE": Bar(1)}
    for s in range(qs):
        B[f"QF{s}"] = Bar(1)
        B[f"QE{s}"] = Bar(1)
    loads, pipe = [], []

    def producer():
        loads.append("KV")
        for t in range(n):
            s = t % qs
            if t >= qs:
                while not B[f"QE{s}"].done(((t // qs) + 1) & 1):
                    yield
            loads.append(f"QF{s}")
            if t >= 1:
                while not B["DOE"].done((t - 1) & 1):
                    yield
            loads.append("DOF")

    def mma():
        def issue_s(t):
            while not B[f"QF{t % qs}"].done((t // qs) & 1):
                yield
            pipe.append(("mma", "S"))                 # S^T(t) writes the S columns
            pipe.append(("commit", "SF"))

        def issue_dp(t):
            while not B["DOF"].done(t & 1):
                yield
            pipe.append(("mma", "dP"))                # dP^T(t) writes the dP columns
            pipe.append(("commit", "DPF"))
        while not B["KV"].done(0):
            yield
        if n > 0:
            yield from issue_s(0)
            yield from issue_dp(0)
        for t in range(n):
            while not B["PF"].done(t & 1):
                yield
            pipe.append(("mma", "S", "dV"))           # dV(t) reads P^T from S
            pipe.append(("commit", "DOE"))
            if t + 1 < n:
                yield from issue_s(t + 1)
            while not B["DSF"].done(t & 1):
                yield
            if with_dq:
                pipe.append(("mma", "dS", "dP"))      # dQ^T(t): dS^T (smem) into the dP columns
                pipe.append(("commit", "DQF"))
                pipe.append(("mma", "dS", "dK"))      # dK(t) reads dS^T from shared memory
            else:
                pipe.append(("mma", "dP", "dK"))      # dK(t) reads dS^T from dP
            pipe.append(("commit", f"QE{t % qs}"))
            if with_dq:
                pipe.append(("commit", "DSE"))
            if t + 1 < n:
                if with_dq:
                    while not B["DQE"].done(t & 1):
                        yield
                yield from issue_dp(t + 1)
        pipe.append(("commit", "Final"))

    def pwarp():
        for t in range(n):
            while not B["SF"].done(t & 1):
                yield
            assert not touches(pipe, "S"), "S read / P written while a product uses S"
            yield
            B["PF"].arrive()
            while not B["DPF"].done(t & 1):
                yield
            if with_dq:
                if t > 0:
                    while not B["DSE"].done((t - 1) & 1):
                        yield
                assert not touches(pipe, "dS"), "dS^T written while a product reads it"
            assert not touches(pipe, "dP"), "dP read / dS written while a product uses dP"
            yield
            B["DSF"].arrive()
        while not B["Final"].done(0):
            yield
        assert not touches(pipe, "dV") and not touches(pipe, "dK")

    def dqwarp():
        for t in range(n if with_dq else 0):
            while not B["DQF"].done(t & 1):
                yield
            assert not touches(pipe, "dP"), "dQ^T read while a product writes the dP columns"
            yield
            B["DQE"].arrive()

    roles = [producer(), mma()] + [pwarp() for _ in range(8)] + [dqwarp() for _ in range(4)]
    return simulate(roles, loads, pipe, B, rnd)


def run_query_outer(n, kst, seed):
    rnd = random.Random(seed)
    B = {"QD": Bar(1), "DPF": Bar(1), "DPR": Bar(8), "Done": Bar(1)}
    for s in range(2):
        # one arrival per dS warp, alternating between two barriers (a warp
        # can arrive for tile j + 1 before a slower one has for tile j)
        B[f"DSF{s}"] = Bar(8)
    for s in range(kst):
        B[f"KF{s}"] = Bar(1)
        B[f"KE{s}"] = Bar(1)
    for s in range(2):
        B[f"VF{s}"] = Bar(1)
        B[f"VE{s}"] = Bar(1)
        B[f"SF{s}"] = Bar(1)
    loads, pipe = [], []

    def producer():
        loads.append("QD")
        for j in range(n):
            sk, sv = j % kst, j & 1
            if j >= kst:
                while not B[f"KE{sk}"].done(((j // kst) + 1) & 1):
                    yield
            loads.append(f"KF{sk}")
            if j >= 2:
                while not B[f"VE{sv}"].done(((j >> 1) + 1) & 1):
                    yield
            loads.append(f"VF{sv}")

    def mma():
        def issue_s(j):
            while not B[f"KF{j % kst}"].done((j // kst) & 1):
                yield
            pipe.append(("mma", f"S{j & 1}"))
            pipe.append(("commit", f"SF{j & 1}"))

        def issue_dp(j):
            while not B[f"VF{j & 1}"].done((j >> 1) & 1):
                yield
            pipe.append(("mma", "dP"))
            pipe.append(("commit", "DPF"))
            pipe.append(("commit", f"VE{j & 1}"))
        while not B["QD"].done(0):
            yield
        if n > 0:
            yield from issue_s(0)
            yield from issue_dp(0)
        for j in range(n):
            if j + 1 < n:
                yield from issue_s(j + 1)
                while not B["DPR"].done(j & 1):
                    yield
                yield from issue_dp(j + 1)
            while not B[f"DSF{j & 1}"].done((j >> 1) & 1):
                yield
            pipe.append(("mma", f"S{j & 1}", "dQ"))   # dQ(j) reads dS from S buffer j & 1
            pipe.append(("commit", f"KE{j % kst}"))
        pipe.append(("commit", "Done"))

    def dswarp():
        for j in range(n):
            while not B[f"SF{j & 1}"].done((j >> 1) & 1):
                yield
            assert not touches(pipe, f"S{j & 1}"), "S read while a product uses its buffer"
            yield
            while not B["DPF"].done(j & 1):
                yield
            assert not touches(pipe, "dP"), "dP read while a product writes it"
            B["DPR"].arrive()
            yield
            assert not touches(pipe, f"S{j & 1}"), "dS written while a product uses its buffer"
            B[f"DSF{j & 1}"].arrive()
        while not B["Done"].done(0):
            yield
        assert not touches(pipe, "dQ")

    return simulate([producer(), mma()] + [dswarp() for _ in range(8)], loads, pipe, B, rnd)


@pytest.mark.parametrize("seed", range(30))
def test_key_outer_protocol(seed):
    rnd = random.Random(seed)
    assert run_key_outer(rnd.choice([0, 1, 2, 3, 7, 12]), rnd.choice([2, 3]), seed)


@pytest.mark.parametrize("seed", range(30))
def test_key_outer_protocol_with_dq(seed):
    rnd = random.Random(seed)
    assert run_key_outer(rnd.choice([0, 1, 2, 3, 7, 12]), 2, seed, with_dq=True)


@pytest.mark.parametrize("seed", range(30))
def test_query_outer_protocol(seed):
    rnd = random.Random(seed)
    assert run_query_outer(rnd.choice([0, 1, 2, 3, 7, 12]), rnd.choice([2, 3]), seed)



def run_fused(units, seed, plant=None, slow_dq=False):
    """The persistent fused d = 128 kernel (all five products, dQ added to the
    fp32 accumulator): one CTA takes the units (key tiles) of `units` (their
    step counts, each >= 1) one after another.  Per step the key-outer
    protocol with two Q stages and dQ^T formed in the dP columns, read out by
    four dQ warps (DQ_FULL, then one DQ_EMPTY arrival per warp before the
    next dP^T may overwrite the columns).  Per unit: a record published in a
    two-slot ring (UNIT_FULL, one UNIT_EMPTY arrival per reading warp), K and
    V loaded once the previous unit's last products that read them have
    completed (KV_EMPTY), and dV / dK read out by the dQ warps after FINAL,
    before the next unit's first dV overwrites them (ACC_EMPTY).  Step and
    unit barriers run on across units (parities from the CTA's global step
    and unit counts).
    Besides the checks of the other models, every product finds the K / V,
    Q and dO tiles of its own unit and step in shared memory, every read of
    S^T, dP^T or dQ^T finds the product of the same step, the dK / dV
    read-out finds the unit's last step, and every warp reads the record of
    its own unit.  slow_dq: the dQ warps get few turns.  plant: None, or a
    mistake to plant: "no_acc_wait" (dV(0)
    without waiting for the read-out), "no_kv_empty" (K / V loaded without
    waiting for KV_EMPTY), "no_unit_empty" (a record written without waiting
    for UNIT_EMPTY), "no_readout_wait" (dQ^T read without DQ_FULL)."""
    rnd = random.Random(seed)
    B = {"KV": Bar(1), "KVE": Bar(1), "DOF": Bar(1), "DOE": Bar(1), "SF": Bar(1),
         "DPF": Bar(1), "Final": Bar(1), "AccE": Bar(4), "PF": Bar(8), "DSF": Bar(8),
         "DQF": Bar(1), "DQE": Bar(4), "DSE": Bar(1)}
    qs = 2
    for s_ in range(qs):
        B[f"QF{s_}"] = Bar(1)
        B[f"QE{s_}"] = Bar(1)
    for s_ in range(2):
        B[f"UF{s_}"] = Bar(1)
        B[f"UE{s_}"] = Bar(13)
    loads, pipe, slots, content = [], [], [None, None], {}
    n_units = len(units)

    def wait(bar, parity):
        while not B[bar].done(parity):
            yield

    def producer():
        g = 0
        for k in range(n_units + 1):
            n = units[k] if k < n_units else 0
            if k >= 2 and plant != "no_unit_empty":
                yield from wait(f"UE{k & 1}", ((k >> 1) - 1) & 1)
            slots[k & 1] = (k, n)
            B[f"UF{k & 1}"].arrive()
            if n == 0:
                return
            for t in range(n):
                gs, s_ = g + t, (g + t) % qs
                if gs >= qs:
                    yield from wait(f"QE{s_}", ((gs // qs) + 1) & 1)
                loads.append((f"QF{s_}", f"Q{s_}", (k, t)))
                if gs >= 1:
                    yield from wait("DOE", (gs - 1) & 1)
                loads.append(("DOF", "dO", (k, t)))
                if t == 0:
                    if k >= 1 and plant != "no_kv_empty":
                        yield from wait("KVE", (k - 1) & 1)
                    loads.append(("KV", "KV", k))
            g += n

    def read_unit(k):
        yield from wait(f"UF{k & 1}", (k >> 1) & 1)
        rec = slots[k & 1]
        assert rec is not None and rec[0] == k, "unit record overwritten before it was read"
        B[f"UE{k & 1}"].arrive()
        return rec[1]

    def mma():
        def issue_s(gs, k, t):
            yield from wait(f"QF{gs % qs}", (gs // qs) & 1)
            pipe.append(("check", "KV", k))
            pipe.append(("check", f"Q{gs % qs}", (k, t)))
            pipe.append(("mma", "K", "S", ("S", gs)))
            pipe.append(("commit", "SF"))

        def issue_dp(gs, k, t):
            yield from wait("DOF", gs & 1)
            pipe.append(("check", "KV", k))
            pipe.append(("check", "dO", (k, t)))
            pipe.append(("mma", "V", "dP", ("dP", gs)))
            pipe.append(("commit", "DPF"))
        g = 0
        for k in range(n_units + 1):
            n = yield from read_unit(k)
            if n == 0:
                break
            yield from wait("KV", k & 1)
            yield from issue_s(g, k, 0)
            if g >= 1:
                yield from wait("DQE", (g - 1) & 1)
            yield from issue_dp(g, k, 0)
            for t in range(n):
                gs = g + t
                yield from wait("PF", gs & 1)
                if t == 0 and k >= 1 and plant != "no_acc_wait":
                    yield from wait("AccE", (k - 1) & 1)
                pipe.append(("check", "S", ("P", gs)))
                pipe.append(("check", "dO", (k, t)))
                pipe.append(("mma", "S", "dV", ("dV", k, t)))
                pipe.append(("commit", "DOE"))
                if t + 1 < n:
                    yield from issue_s(gs + 1, k, t + 1)
                yield from wait("DSF", gs & 1)
                pipe.append(("check", "KV", k))
                pipe.append(("mma", "dS", "dP", ("dQ", gs)))   # dQ^T into the dP columns
                pipe.append(("commit", "DQF"))
                if t + 1 == n:
                    pipe.append(("commit", "KVE"))
                pipe.append(("check", f"Q{gs % qs}", (k, t)))
                pipe.append(("mma", "dS", "dK", ("dK", k, t)))
                pipe.append(("commit", f"QE{gs % qs}"))
                pipe.append(("commit", "DSE"))
                if t + 1 == n:
                    pipe.append(("commit", "Final"))
                else:
                    yield from wait("DQE", gs & 1)
                    yield from issue_dp(gs + 1, k, t + 1)
            g += n

    def pwarp():
        g = 0
        for k in range(n_units + 1):
            n = yield from read_unit(k)
            if n == 0:
                return
            for t in range(n):
                gs = g + t
                yield from wait("SF", gs & 1)
                assert not touches(pipe, "S")
                assert content.get("S") in (("S", gs), ("P", gs)), "S^T read before its product"
                yield
                content["S"] = ("P", gs)
                B["PF"].arrive()
                yield from wait("DPF", gs & 1)
                if gs > 0:
                    yield from wait("DSE", (gs - 1) & 1)
                assert not touches(pipe, "dS") and not touches(pipe, "dP")
                assert content.get("dP") == ("dP", gs), "dP^T read before its product"
                yield
                B["DSF"].arrive()
            g += n

    def dqwarp():
        g = 0
        for k in range(n_units + 1):
            n = yield from read_unit(k)
            if n == 0:
                return
            for t in range(n):
                gs = g + t
                if plant != "no_readout_wait":
                    yield from wait("DQF", gs & 1)
                assert not touches(pipe, "dP"), "dQ^T read while a product writes the dP columns"
                assert content.get("dP") == ("dQ", gs), "dQ^T read before the product that forms it"
                yield
                B["DQE"].arrive()
                yield                      # the step's reduce-adds
            yield from wait("Final", k & 1)
            assert not touches(pipe, "dV") and not touches(pipe, "dK"), \
                "dK / dV read out while a product writes them"
            assert content.get("dV") == ("dV", k, n - 1) and content.get("dK") == ("dK", k, n - 1), \
                "dK / dV read out without the unit's last step, or after the next unit's first"
            yield
            B["AccE"].arrive()
            yield                          # the dK store
            g += n

    return simulate([producer(), mma()] + [pwarp() for _ in range(8)] +
                    [dqwarp() for _ in range(4)], loads, pipe, B, rnd, content,
                    slow=range(10, 14) if slow_dq else (), limit=100_000)


def random_units(rnd):
    return [rnd.choice([1, 1, 2, 3, 5]) for _ in range(rnd.randint(1, 6))]


@pytest.mark.parametrize("seed", range(60))
def test_fused_protocol(seed):
    rnd = random.Random(seed)
    assert run_fused(random_units(rnd), seed, slow_dq=seed % 3 == 0)


@pytest.mark.parametrize("plant,message", [
    ("no_readout_wait", "dQ^T read"),
    ("no_acc_wait", "dK / dV read out"),
    ("no_kv_empty", "K / V"),
    ("no_unit_empty", "unit record"),
])
def test_fused_model_catches_a_planted_mistake(plant, message):
    caught = 0
    for seed in range(60):
        rnd = random.Random(1000 + seed)
        units = [rnd.choice([1, 1, 2, 3]) for _ in range(rnd.randint(3, 6))]
        try:
            finished = run_fused(units, seed, plant=plant, slow_dq=seed % 2 == 0)
        except AssertionError as e:
            assert message in str(e), (plant, e)
            caught += 1
            continue
        if not finished:       # a hang: a barrier phase completed twice unseen
            caught += 1
    assert caught > 0
