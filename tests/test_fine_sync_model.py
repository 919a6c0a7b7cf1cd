"""A discrete-event model of the fine kernel's synchronisation (csrc/fine.cu),
checked on the CPU.

Each warp role of one CTA is a generator that yields its waits in program
order: mbarrier parity waits (with the phase the code means to wait for),
named-barrier syncs, and arrivals; MMA commits arrive after random delays;
the scheduler picks warps in random order.  Over random unit sequences
(including units with an empty union) the test checks that every run ends
(no deadlock) and that no parity wait ever passes before the phase it stands
for has completed: a parity wait cannot tell phase p from phase p + 2, so a
barrier more than one phase away from a waiter would let the wait pass early
(or never), and the kernel relies on every barrier staying within one phase.

The model follows the kernel's roles: warp 0 builds the unit lists and loads
K into a 3-slot ring, warp 1 issues Q.K^T into two S buffers, warp 2 loads V
into a 3-slot ring, warp 3 issues P.V, and eight softmax warps (two per TMEM
lane quarter, one per key cube of a step) exchange row maxima through a named
barrier, hand P to the P.V warp and stage the next unit's Q.  A planted
protocol -- the same softmax split into warps that take alternate steps but
still wait for the previous step's P.V on one barrier -- must be caught.
"""
import random

import pytest


class MBar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1

    def passes(self, parity):  # mbarrier.try_wait.parity
        return (self.done & 1) != parity


class Cta:
    def __init__(self, softmax_counts):
        self.mb = {}
        for i in range(3):
            for n in ("k_full", "k_empty", "v_full", "v_empty"):
                self.mb[f"{n}{i}"] = MBar(1)
        for i in range(2):
            self.mb[f"s_full{i}"] = MBar(1)
            self.mb[f"s_free{i}"] = MBar(softmax_counts)
            self.mb[f"list_full{i}"] = MBar(1)
            self.mb[f"list_empty{i}"] = MBar(10)  # V producer, P.V warp, 8 softmax warps
        self.mb["p_full"] = MBar(softmax_counts)
        for n in ("pv_done", "pv_done0", "pv_done1", "q_empty"):
            self.mb[n] = MBar(1)
        self.mb["q_full"] = MBar(8)
        self.count = [0, 0]
        self.commits = []

    def commit(self, name, rng):
        self.commits.append([name, rng.randint(0, 6)])


def wait(name, phase):
    """A parity wait for `phase` of barrier `name`."""
    return ("wait", name, phase & 1, phase)


def producer_k(c, units):
    g = 0
    for ul, nst in enumerate(units):
        lb = ul & 1
        if ul >= 2:
            yield wait(f"list_empty{lb}", (ul >> 1) - 1)
        c.count[lb] = nst
        c.mb[f"list_full{lb}"].arrive()
        for _ in range(nst):
            if g >= 3:
                yield wait(f"k_empty{g % 3}", g // 3 - 1)
            c.mb[f"k_full{g % 3}"].arrive()  # the TMA copy lands
            g += 1
            yield ("step",)


def producer_v(c, units):
    g = 0
    for ul, nst in enumerate(units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        assert c.count[lb] == nst
        for _ in range(nst):
            if g >= 3:
                yield wait(f"v_empty{g % 3}", g // 3 - 1)
            c.mb[f"v_full{g % 3}"].arrive()
            g += 1
            yield ("step",)
        c.mb[f"list_empty{lb}"].arrive()


def mma_qk(c, units, rng):
    g = 0
    for ul, nst in enumerate(units):
        yield wait(f"list_full{ul & 1}", ul >> 1)
        yield wait("q_full", ul)
        for _ in range(nst):
            if g >= 2:
                yield wait(f"s_free{g & 1}", (g >> 1) - 1)
            yield wait(f"k_full{g % 3}", g // 3)
            c.commit(f"s_full{g & 1}", rng)
            c.commit(f"k_empty{g % 3}", rng)
            g += 1
        c.commit("q_empty", rng)


def mma_pv(c, units, rng, per_parity):
    g = 0
    for ul, nst in enumerate(units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        for _ in range(nst):
            yield wait("p_full", g)
            yield wait(f"v_full{g % 3}", g // 3)
            c.commit(f"pv_done{g & 1}" if per_parity else "pv_done", rng)
            c.commit(f"v_empty{g % 3}", rng)
            g += 1
        c.mb[f"list_empty{lb}"].arrive()


def softmax_kernel(c, units, warp):
    """The softmax warps as the kernel runs them: both warps of a quarter on every step."""
    quarter = warp & 3
    bar = ("nbar", 1 + quarter)
    g = 0
    c.mb["q_full"].arrive()  # the first unit's Q
    for ul, nst in enumerate(units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        more = ul + 1 < len(units)
        if nst == 0 and more:
            yield wait("q_empty", ul)
            c.mb["q_full"].arrive()
        for t in range(nst):
            yield wait(f"s_full{g & 1}", g >> 1)
            if t + 1 == nst and more:
                yield wait("q_empty", ul)
                c.mb["q_full"].arrive()
            c.mb[f"s_free{g & 1}"].arrive()
            yield bar  # row-max exchange with the other key cube's thread
            if g > 0:
                yield wait("pv_done", g - 1)
            c.mb["p_full"].arrive()
            g += 1
        c.mb[f"list_empty{lb}"].arrive()
        yield bar  # partial sums
        if nst > 0:
            yield wait("pv_done", g - 1)
        yield bar


def softmax_alternating(c, units, warp):
    """Planted protocol: warp parity p takes the steps g with g % 2 == p and
    waits for P.V(g - 1) on the single pv_done barrier."""
    par = (warp - 4) >> 2
    g = 0
    c.mb["q_full"].arrive()
    for ul, nst in enumerate(units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        more = ul + 1 < len(units)
        last_owner = (g + nst - 1) & 1 if nst else -1
        for t in range((g + par) & 1, nst, 2):
            gs = g + t
            yield wait(f"s_full{gs & 1}", gs >> 1)
            if t + 1 == nst and more:
                yield wait("q_empty", ul)
                c.mb["q_full"].arrive()
            c.mb[f"s_free{gs & 1}"].arrive()
            if gs > 0:
                yield wait("pv_done", gs - 1)
            c.mb["p_full"].arrive()
        if (nst == 0 or last_owner != par) and more:
            yield wait("q_empty", ul)
            c.mb["q_full"].arrive()
        c.mb[f"list_empty{lb}"].arrive()
        if nst > 0:
            yield wait("pv_done", g + nst - 1)
        g += nst


def run(units, seed, softmax=softmax_kernel, softmax_counts=8, per_parity=False):
    rng = random.Random(seed)
    c = Cta(softmax_counts)
    warps = {0: producer_k(c, units), 1: mma_qk(c, units, rng), 2: producer_v(c, units),
             3: mma_pv(c, units, rng, per_parity)}
    for w in range(4, 12):
        warps[w] = softmax(c, units, w)
    blocked, finished = {}, set()
    nbar_count, nbar_gen = {}, {}
    while len(finished) < len(warps):
        for item in list(c.commits):
            item[1] -= 1
            if item[1] < 0:
                c.commits.remove(item)
                c.mb[item[0]].arrive()
        order = [w for w in warps if w not in finished]
        rng.shuffle(order)
        moved = False
        for w in order:
            op = blocked.get(w)
            if op is not None:
                if op[0] == "wait":
                    if not c.mb[op[1]].passes(op[2]):
                        continue
                    if c.mb[op[1]].done <= op[3]:
                        return f"early pass: warp {w} waited for phase {op[3]} of {op[1]}"
                elif nbar_gen.get(op[1], 0) <= op[2]:
                    continue
                del blocked[w]
            try:
                op = next(warps[w])
            except StopIteration:
                finished.add(w)
                moved = True
                break
            moved = True
            if op[0] == "wait":
                if not c.mb[op[1]].passes(op[2]):
                    blocked[w] = op
                elif c.mb[op[1]].done <= op[3]:
                    return f"early pass: warp {w} waited for phase {op[3]} of {op[1]}"
            elif op[0] == "nbar":  # bar.sync id, 64: the two warps of a quarter
                bid = op[1]
                g0 = nbar_gen.get(bid, 0)
                nbar_count[bid] = nbar_count.get(bid, 0) + 1
                if nbar_count[bid] == 2:
                    nbar_count[bid], nbar_gen[bid] = 0, g0 + 1
                else:
                    blocked[w] = ("nbar", bid, g0)
            break
        if not moved and not c.commits:
            return "deadlock: " + ", ".join(f"warp {w} at {blocked.get(w)}" for w in sorted(warps)
                                            if w not in finished)
    return "ok"


def unit_sequences(n, seed):
    rng = random.Random(seed)
    return [[rng.choice([0, 1, 2, 3, 5, 39, 40]) for _ in range(rng.randint(1, 6))] for _ in range(n)]


def test_kernel_protocol_never_deadlocks_or_passes_early():
    for i, units in enumerate(unit_sequences(400, 1)):
        assert run(units, seed=i) == "ok", units


@pytest.mark.parametrize("units", [[0], [0, 0, 3], [1], [1, 0, 1], [2, 40, 0, 41]])
def test_kernel_protocol_edge_units(units):
    for seed in range(50):
        assert run(units, seed) == "ok"


def test_model_catches_a_wait_that_can_pass_early():
    bad = [run(units, seed=i, softmax=softmax_alternating, softmax_counts=4)
           for i, units in enumerate(unit_sequences(200, 2))]
    assert any(r.startswith("early pass") for r in bad)
