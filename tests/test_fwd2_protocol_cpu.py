"""A model of the persistent two-query-tile forward's barrier protocol,
checked on random unit sequences and interleavings (no GPU).

It follows the kernel's roles step by step: the TMA producer (Q per unit,
K / V through two-stage rings), the MMA warp (P V(j) then S(j+1) per tile,
commits), and the eight softmax warps (S_FULL wait, P_FULL arrival per warp,
the rescale of O, the epilogue and O_FREE).  Tensor-core products and their
commits go through one in-order queue, as on the hardware: a commit arrives
on its barrier only once every product issued before it has completed.
mbarriers are modelled with their phase/parity semantics.

Checked: every run ends (no wait that can never complete: a protocol
deadlock or a parity wait aliased by a skipped phase), and whenever a
softmax warpgroup reads or rescales O (tile u), no P V product on that tile
is still queued or running -- the property the kernel gets from S_FULL of
tile j + 1 implying P V(j) has completed, instead of waiting for O_DONE on
every tile."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


def unit_tiles(blk, nq, nk, causal):
    out = []
    for u in range(2):
        first = blk * 256 + 128 * u
        n = (nk + 127) // 128
        if first >= nq:
            n = 0
        elif causal:
            last_key = min(first + 128, nq) - 1 + nk - nq
            n = 0 if last_key < 0 else min(n, last_key // 128 + 1)
        out.append(n)
    return out


def run(units, seed):
    rnd = random.Random(seed)
    B = {n: Bar(1) for n in ("QFull", "QEmpty", "K0F", "K1F", "K0E", "K1E", "V0F", "V1F",
                              "V0E", "V1E", "S0", "S1", "O0", "O1")}
    for u in range(2):
        B[f"P{u}"] = Bar(4)        # one arrival per softmax warp
        B[f"OF{u}"] = Bar(4)
    loads = []                     # TMA completions, any order
    pipe = []                      # tensor-core queue: ("mma", tile) or ("commit", barrier)

    def producer():
        it = kt = 0
        for w in units:
            n_max = max(w)

            def load_kv(j):
                g = kt + j
                s = g & 1
                if g >= 2:
                    while not B[f"K{s}E"].done(((g >> 1) + 1) & 1):
                        yield
                loads.append(f"K{s}F")
                if g >= 2:
                    while not B[f"V{s}E"].done(((g >> 1) + 1) & 1):
                        yield
                loads.append(f"V{s}F")
            if n_max > 0:
                yield from load_kv(0)
            if it >= 1:
                while not B["QEmpty"].done((it - 1) & 1):
                    yield
            loads.append("QFull")
            for j in range(1, n_max):
                yield from load_kv(j)
            kt += n_max
            it += 1

    def mma():
        it = kt = 0
        cp = [0, 0]
        of = [0, 0]
        for w in units:
            n_max = max(w)
            while not B["QFull"].done(it & 1):
                yield
            if n_max > 0:
                while not B[f"K{kt & 1}F"].done((kt >> 1) & 1):
                    yield
                for u in range(2):
                    if w[u] > 0:
                        pipe.append(("mma", None))
                        pipe.append(("commit", f"S{u}"))
                pipe.append(("commit", f"K{kt & 1}E"))
            if n_max <= 1:
                pipe.append(("commit", "QEmpty"))
            for u in range(2):
                if w[u] > 0 and of[u] > 0:
                    while not B[f"OF{u}"].done((of[u] - 1) & 1):
                        yield
                of[u] += 1 if w[u] > 0 else 0
            for j in range(n_max):
                g = kt + j
                s = g & 1
                while not B[f"V{s}F"].done((g >> 1) & 1):
                    yield
                if j + 1 < n_max:
                    while not B[f"K{(g + 1) & 1}F"].done(((g + 1) >> 1) & 1):
                        yield
                for u in range(2):
                    if j >= w[u]:
                        continue
                    while not B[f"P{u}"].done(cp[u] & 1):
                        yield
                    cp[u] += 1
                    pipe.append(("mma", u))            # P V_u(j) writes O_u
                    pipe.append(("commit", f"O{u}"))
                    if j + 1 < w[u]:
                        pipe.append(("mma", None))     # S_u(j + 1)
                        pipe.append(("commit", f"S{u}"))
                pipe.append(("commit", f"V{s}E"))
                if j + 1 < n_max:
                    pipe.append(("commit", f"K{(g + 1) & 1}E"))
                if j + 2 == n_max:
                    pipe.append(("commit", "QEmpty"))
            kt += n_max
            it += 1

    def o_busy(u):
        return any(op == ("mma", u) for op in pipe)

    def softmax(u):
        cs = co = 0
        for w in units:
            nk = w[u]
            for j in range(nk):
                while not B[f"S{u}"].done(cs & 1):
                    yield
                cs += 1
                yield
                if j > 0 and rnd.random() < 0.3:           # a rescale of O
                    assert not o_busy(u), "O rescaled while a P V on it is in flight"
                B[f"P{u}"].arrive()
            if nk > 0:
                co += nk
                while not B[f"O{u}"].done((co - 1) & 1):
                    yield
                assert not o_busy(u), "O read out while a P V on it is in flight"
                yield
                B[f"OF{u}"].arrive()

    roles = [producer(), mma()] + [softmax(u) for u in range(2) for _ in range(4)]
    alive = list(range(len(roles)))
    for _ in range(2_000_000):
        if not alive and not loads and not pipe:
            return True
        r = rnd.random()
        if loads and (r < 0.2 or not alive):
            B[loads.pop(rnd.randrange(len(loads)))].arrive()
        elif pipe and (r < 0.45 or not alive):
            op, arg = pipe.pop(0)                          # in-order completion
            if op == "commit":
                B[arg].arrive()
        elif alive:
            k = rnd.choice(alive)
            try:
                next(roles[k])
            except StopIteration:
                alive.remove(k)
    return False


@pytest.mark.parametrize("seed", range(40))
def test_persistent_forward_protocol(seed):
    rnd = random.Random(seed)
    nq = rnd.choice([129, 300, 700, 1100, 1500])
    nk = rnd.choice([nq, 64, 300, 1300])
    causal = rnd.random() < 0.5
    nqt = (nq + 255) // 256
    units = [unit_tiles(rnd.randrange(nqt), nq, nk, causal) for _ in range(rnd.randint(1, 6))]
    assert run(units, seed), f"protocol stalled: units {units}"


def run_one_tile(units, kst, vst, seed, kp=1, vp=1, plant=None, records=False):
    """The one-tile forward (d = 64 / 256, short, split and block-sparse
    paths), persistent: one CTA walks the units of `units` (their key-tile
    counts, 0 allowed) one after another.  Per key tile: S(g+1) is issued
    before P V(g), into the other of two score buffers, and the softmax waits
    for O_DONE only before a rescale of O and on the last tile of a unit.  Per
    unit: Q is loaded once the previous unit's last S has completed (Q_EMPTY,
    committed after that S is issued); its first P V overwrites O with no
    wait of its own, since every softmax warp reads the previous unit's O out
    before it arrives on P_FULL for this unit's first tile (the model checks
    that the read-out finds the unit's last product).  kp, vp: pieces per K and V tile (d = 256: four 64-column
    chunks of K, two halves of V); the rings then hold kst and vst pieces.
    Q and K are loaded by one producer lane, V by another, each with its own
    waits.
    Global indices (tiles over all units) give the parities.  Every product
    checks, when it runs, that Q and the ring slots it reads hold its own
    unit's and tile's pieces and that it reads the P of its own tile; the
    epilogue that O holds the unit's last product.  plant: None or a mistake
    ("no_qempty_wait", "early_qempty", "early_p_full": a softmax warp arrives
    on P_FULL of a unit's first tile before its read-out of the previous
    unit's O; "early_release": a softmax warp releases a unit record before
    it has walked the unit's tiles).  records: the block-sparse form, in which
    the Q / K lane publishes each unit's record (its kept tiles) in one of two
    slots (UNIT_FULL) once the six readers — the V lane, the MMA warp and the
    four softmax warps — have released the slot's previous unit (UNIT_EMPTY);
    each reader checks that the slot still holds its unit while it uses it."""
    rnd = random.Random(seed)
    B = {"QFull": Bar(1), "QEmpty": Bar(1), "ODone": Bar(1)}
    for s in range(kst):
        B[f"KF{s}"], B[f"KE{s}"] = Bar(1), Bar(1)
    for s in range(vst):
        B[f"VF{s}"], B[f"VE{s}"] = Bar(1), Bar(1)
    for s in range(2):
        B[f"SF{s}"] = Bar(1)
        B[f"PF{s}"] = Bar(4)           # the model's four softmax warps
        B[f"UF{s}"] = Bar(1)
        B[f"UE{s}"] = Bar(6)
    loads, pipe, content = [], [], {}

    def take_record(k):
        if records:
            yield from wait(f"UF{k & 1}", (k >> 1) & 1)
            assert content.get(("rec", k & 1)) == k, "a unit record of another unit"

    def release_record(k):
        if records:
            assert content.get(("rec", k & 1)) == k, "a unit record overwritten while in use"
            B[f"UE{k & 1}"].arrive()

    def wait(name, parity):
        while not B[name].done(parity):
            yield

    def producer_ring(tag, slots, pieces):
        # tag K: this lane also loads each unit's Q before the unit's K pieces
        i = 0
        for k, n in enumerate(units):
            if tag == "K" and records:
                if k >= 2:
                    yield from wait(f"UE{k & 1}", ((k >> 1) - 1) & 1)
                content[("rec", k & 1)] = k
                yield
                B[f"UF{k & 1}"].arrive()
            if tag == "V":
                yield from take_record(k)
            if tag == "K":
                if k >= 1 and plant != "no_qempty_wait":
                    yield from wait("QEmpty", (k - 1) & 1)
                loads.append(("QFull", "Q", k))
            for j in range(n):
                for c in range(pieces):
                    s = i % slots
                    if i >= slots:
                        yield from wait(f"{tag}E{s}", ((i // slots) + 1) & 1)
                    loads.append((f"{tag}F{s}", f"{tag}{s}", (k, j, c)))
                    i += 1
            if tag == "V":
                release_record(k)

    def mma():
        def issue_s(g, k, j):
            for c in range(kp):
                i = g * kp + c
                yield from wait(f"KF{i % kst}", (i // kst) & 1)
                pipe.append(("mma", f"S{g & 1}", ("S", g)))
                pipe.append(("check", "Q", k))
                pipe.append(("check", f"K{i % kst}", (k, j, c)))
                pipe.append(("commit", f"KE{i % kst}"))
            pipe.append(("commit", f"SF{g & 1}"))

        def issue_pv(g, k, j):
            for h in range(vp):
                i = g * vp + h
                yield from wait(f"VF{i % vst}", (i // vst) & 1)
                pipe.append(("check", f"S{g & 1}", ("P", g)))
                pipe.append(("mma", f"S{g & 1}", "O", ("O", k, j)))
                pipe.append(("check", f"V{i % vst}", (k, j, h)))
                pipe.append(("commit", f"VE{i % vst}"))
            pipe.append(("commit", "ODone"))
        g = 0
        for k, n in enumerate(units):
            yield from take_record(k)
            release_record(k)                  # (only the count is needed)
            yield from wait("QFull", k & 1)
            if n > 0:
                if plant == "early_qempty" and n == 1:
                    pipe.append(("commit", "QEmpty"))
                yield from issue_s(g, k, 0)
            for j in range(n):
                if j + 1 < n:
                    yield from issue_s(g + j + 1, k, j + 1)
                elif not (plant == "early_qempty" and n == 1):
                    pipe.append(("commit", "QEmpty"))
                yield from wait(f"PF{(g + j) & 1}", ((g + j) >> 1) & 1)
                yield from issue_pv(g + j, k, j)
            if n == 0:
                pipe.append(("commit", "QEmpty"))
            g += n

    def busy(region):
        return any(op[0] == "mma" and region in op[1:] for op in pipe)

    def softmax():
        g = 0
        pending = None                 # (unit, last tile) whose O is still to be read out
        for k, n in enumerate(units):
            yield from take_record(k)
            if plant == "early_release":
                release_record(k)
            for j in range(n):
                gj = g + j
                yield from wait(f"SF{gj & 1}", (gj >> 1) & 1)
                if records:
                    # (the kernel reads the tile's index from the record here,
                    # for its mask, after the scores have arrived)
                    assert content.get(("rec", k & 1)) == k, "a unit record overwritten while in use"
                assert not busy(f"S{gj & 1}"), "score buffer read while a product uses it"
                assert content.get(f"S{gj & 1}") in (("S", gj), ("P", gj)), "scores of another tile"
                yield
                content[f"S{gj & 1}"] = ("P", gj)
                rescale = j > 0 and rnd.random() < 0.3
                if j > 0 and (rescale or j == n - 1):
                    yield from wait("ODone", (gj - 1) & 1)
                if rescale:
                    assert not busy("O"), "O rescaled while a P V is in flight"
                    assert content.get("O") == ("O", k, j - 1), "O rescaled holding another tile's sum"
                B[f"PF{gj & 1}"].arrive()
                if pending is not None:
                    yield from read_out(*pending)
                    pending = None
            if plant != "early_release":
                release_record(k)
            if n > 0:
                yield from wait("ODone", (g + n - 1) & 1)
                if plant == "early_p_full":
                    pending = (k, n - 1)       # read out after the next arrival
                else:
                    yield from read_out(k, n - 1)
            g += n
        if pending is not None:
            yield from read_out(*pending)

    def read_out(k, last):
        yield
        assert not busy("O"), "O read out while a P V is in flight"
        assert content.get("O") == ("O", k, last), "O read out without the unit's last product"
        yield

    roles = [producer_ring("K", kst, kp), producer_ring("V", vst, vp), mma()] + \
        [softmax() for _ in range(4)]
    alive = list(range(len(roles)))
    for _ in range(300_000):
        if not alive and not loads and not pipe:
            return True
        r = rnd.random()
        if loads and (r < 0.2 or not alive):
            bar, key, val = loads.pop(rnd.randrange(len(loads)))
            content[key] = val
            B[bar].arrive()
        elif pipe and (r < 0.45 or not alive):
            op = pipe.pop(0)
            if op[0] == "commit":
                B[op[1]].arrive()
            elif op[0] == "check":
                assert content.get(op[1]) == op[2], f"a product read {op[1]} holding another piece"
            elif len(op) == 4:
                content[op[2]] = op[3]
            elif len(op) == 3:
                content[op[1]] = op[2]
        elif alive:
            k = rnd.choice(alive)
            try:
                next(roles[k])
            except StopIteration:
                alive.remove(k)
    return False


def random_units(rnd):
    return [rnd.choice([0, 1, 1, 2, 3, 5]) for _ in range(rnd.randint(1, 5))]


@pytest.mark.parametrize("seed", range(30))
def test_one_tile_forward_protocol(seed):
    rnd = random.Random(seed)
    assert run_one_tile(random_units(rnd), rnd.choice([2, 3]), rnd.choice([2, 3]), seed)


@pytest.mark.parametrize("seed", range(30))
def test_one_tile_forward_protocol_in_pieces(seed):
    """d = 256: K in four chunks through a ring of four to six, V in two
    halves through a ring of two or three, each ring loaded by its own lane."""
    rnd = random.Random(seed)
    assert run_one_tile(random_units(rnd), rnd.choice([4, 5, 6]), rnd.choice([2, 3]), seed, kp=4, vp=2)


@pytest.mark.parametrize("seed", range(30))
def test_one_tile_forward_protocol_block_sparse(seed):
    """Block mask: the unit records between the Q / K lane and the readers."""
    rnd = random.Random(seed)
    pieces = rnd.random() < 0.5
    assert run_one_tile(random_units(rnd) + random_units(rnd), rnd.choice([4, 5]) if pieces else 2,
                        2, seed, kp=4 if pieces else 1, vp=2 if pieces else 1, records=True)


def test_one_tile_model_catches_an_early_record_release():
    caught = False
    for seed in range(80):
        rnd = random.Random(900 + seed)
        units = [rnd.choice([0, 1, 1, 2]) for _ in range(rnd.randint(4, 8))]
        try:
            if not run_one_tile(units, 6, 3, seed, plant="early_release", records=True):
                caught = True
        except AssertionError:
            caught = True
        if caught:
            break
    assert caught


@pytest.mark.parametrize("plant", ["no_qempty_wait", "early_qempty", "early_p_full"])
def test_one_tile_model_catches_a_planted_mistake(plant):
    caught = 0
    for seed in range(60):
        rnd = random.Random(500 + seed)
        units = [rnd.choice([1, 1, 2, 3]) for _ in range(rnd.randint(2, 5))]
        try:
            finished = run_one_tile(units, 2, 2, seed, plant=plant)
        except AssertionError:
            caught += 1
            continue
        if not finished:      # a hang: a barrier phase completed twice unseen
            caught += 1
    assert caught > 0
