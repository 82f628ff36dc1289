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


def simulate(roles, loads, pipe, B, rnd, content=None):
    """content: optional dict, TMEM region -> label of the product that last
    wrote it (products given as ("mma", reads, writes, label))."""
    alive = list(range(len(roles)))
    for _ in range(2_000_000):
        if not alive and not loads and not pipe:
            return True
        r = rnd.random()
        if loads and (r < 0.2 or not alive):
            B[loads.pop(rnd.randrange(len(loads)))].arrive()
        elif pipe and (r < 0.45 or not alive):
            op = pipe.pop(0)
            if op[0] == "commit":
                B[op[1]].arrive()
            elif content is not None and len(op) == 4:
                content[op[2]] = op[3]
        elif alive:
            k = rnd.choice(alive)
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



def run_fused(n, seed, readout_wait=True):
    """The fused d = 128 kernel (all five products, dQ added to the fp32
    accumulator): the key-outer protocol with two Q stages, dQ^T formed in
    the dP columns and read out by four dQ warps (DQ_FULL, then one DQ_EMPTY
    arrival per warp before dP^T(t+1) may overwrite the columns); their
    staging and bulk reduce-add are ordered among themselves by named
    barriers and touch no barrier here.  Besides the checks of the other
    models, each read of dQ^T must find the product of the same step in the
    dP columns.  readout_wait=False plants a mistake: the dQ warps read
    without waiting for DQ_FULL."""
    rnd = random.Random(seed)
    B = {"KV": Bar(1), "DOF": Bar(1), "DOE": Bar(1), "SF": Bar(1), "DPF": Bar(1),
         "Final": Bar(1), "PF": Bar(8), "DSF": Bar(8), "DQF": Bar(1), "DQE": Bar(4),
         "DSE": Bar(1)}
    qs = 2
    for s_ in range(qs):
        B[f"QF{s_}"] = Bar(1)
        B[f"QE{s_}"] = Bar(1)
    loads, pipe = [], []

    def producer():
        loads.append("KV")
        for t in range(n):
            s_ = t % qs
            if t >= qs:
                while not B[f"QE{s_}"].done(((t // qs) + 1) & 1):
                    yield
            loads.append(f"QF{s_}")
            if t >= 1:
                while not B["DOE"].done((t - 1) & 1):
                    yield
            loads.append("DOF")

    def mma():
        def issue_s(t):
            while not B[f"QF{t % qs}"].done((t // qs) & 1):
                yield
            pipe.append(("mma", "S"))
            pipe.append(("commit", "SF"))

        def issue_dp(t):
            while not B["DOF"].done(t & 1):
                yield
            pipe.append(("mma", "dP"))
            pipe.append(("commit", "DPF"))
        while not B["KV"].done(0):
            yield
        if n > 0:
            yield from issue_s(0)
            yield from issue_dp(0)
        for t in range(n):
            while not B["PF"].done(t & 1):
                yield
            pipe.append(("mma", "S", "dV"))
            pipe.append(("commit", "DOE"))
            if t + 1 < n:
                yield from issue_s(t + 1)
            while not B["DSF"].done(t & 1):
                yield
            pipe.append(("mma", "dS", "dP", ("dQ", t)))   # dQ^T(t) into the dP columns
            pipe.append(("commit", "DQF"))
            pipe.append(("mma", "dS", "dK"))
            pipe.append(("commit", f"QE{t % qs}"))
            pipe.append(("commit", "DSE"))
            if t + 1 < n:
                while not B["DQE"].done(t & 1):
                    yield
                yield from issue_dp(t + 1)
        pipe.append(("commit", "Final"))

    def pwarp():
        for t in range(n):
            while not B["SF"].done(t & 1):
                yield
            assert not touches(pipe, "S")
            yield
            B["PF"].arrive()
            while not B["DPF"].done(t & 1):
                yield
            if t > 0:
                while not B["DSE"].done((t - 1) & 1):
                    yield
            assert not touches(pipe, "dS") and not touches(pipe, "dP")
            yield
            B["DSF"].arrive()
        while not B["Final"].done(0):
            yield
        assert not touches(pipe, "dV") and not touches(pipe, "dK")

    def dqwarp():
        for t in range(n):
            if readout_wait:
                while not B["DQF"].done(t & 1):
                    yield
            assert not touches(pipe, "dP"), "dQ^T read while a product writes the dP columns"
            assert content.get("dP") == ("dQ", t), "dQ^T read before the product that forms it"
            yield
            B["DQE"].arrive()

    content = {}
    return simulate([producer(), mma()] + [pwarp() for _ in range(8)] +
                    [dqwarp() for _ in range(4)], loads, pipe, B, rnd, content)


@pytest.mark.parametrize("seed", range(40))
def test_fused_protocol(seed):
    rnd = random.Random(seed)
    assert run_fused(rnd.choice([0, 1, 2, 3, 4, 7, 12]), seed)


def test_fused_model_catches_a_missing_readout_wait():
    caught = 0
    for seed in range(40):
        try:
            run_fused(6, seed, readout_wait=False)
        except AssertionError as e:
            assert "dQ^T read" in str(e), e
            caught += 1
    assert caught > 0
