"""A discrete-event model of the fine kernel's synchronisation (csrc/fine.cu),
checked on the CPU.

Each warp role of one CTA is a generator that yields its waits in program
order: mbarrier parity waits (with the phase the code means to wait for),
named-barrier syncs, arrivals and data-hazard checks.  Each MMA-issuing warp
commits into its own queue whose arrivals land in issue order after random
delays (a tcgen05.commit completes once every earlier MMA of its thread has),
and the scheduler picks warps in random order.  Over random unit sequences
(including units with an empty union) the test checks that every run ends (no
deadlock), that no parity wait ever passes before the phase it stands for has
completed (a parity wait cannot tell phase p from phase p + 2, so the kernel
relies on every barrier staying within one phase of each waiter), and that
the TMEM hazards hold: P is rewritten only after the P.V that read it, a
group's O is rescaled only after the last P.V into it, and the epilogue
reads O only after the unit's last P.V.

The model follows the kernel's roles: warp 0 builds the unit lists and loads
K into a 3-slot ring, warp 1 issues Q.K^T into the one S buffer, warp 2 loads
V into a 3-slot ring, warp 3 issues P.V into the O of the step's group, and
two softmax groups of four warps (one per TMEM lane quarter) take the even
and the odd steps, stage the next unit's Q, and merge their results in a
per-unit epilogue through a named barrier per lane quarter.  Both unit
schedules are modelled: static (every role knows the CTA's unit count) and
dynamic (units are claimed one ahead at run time, so each list says whether
another unit follows, and a final list, the end marker, stops every role).
Planted protocol mistakes must be caught.
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
    def __init__(self, shared_s_full=False, dynamic=True):
        self.dynamic = dynamic
        self.mb = {}
        for i in range(3):
            for n in ("k_full", "k_empty", "v_full", "v_empty"):
                self.mb[f"{n}{i}"] = MBar(1)
        for i in range(2):
            self.mb[f"list_full{i}"] = MBar(1)
            self.mb[f"list_empty{i}"] = MBar(11)  # V producer, both MMA warps, 8 softmax warps
            self.mb[f"pv_grp{i}"] = MBar(1)
        self.shared_s_full = shared_s_full
        self.mb["s_full0"] = MBar(1)
        self.mb["s_full1"] = MBar(1)
        for n in ("s_free", "p_full", "q_full"):
            self.mb[n] = MBar(4)
        for n in ("q_empty", "unit_done"):
            self.mb[n] = MBar(1)
        self.mb["o_free"] = MBar(8)
        self.count = [0, 0]
        self.info = [None, None]  # per list buffer: (steps, another unit follows) or END
        self.queues = {}

    def commit(self, issuer, name, rng):
        self.queues.setdefault(issuer, []).append([name, rng.randint(0, 6)])


def wait(name, phase):
    """A parity wait for `phase` of barrier `name`."""
    return ("wait", name, phase & 1, phase)


def check(cond, what):
    return ("check", cond, what)


END = "end"


def producer_k(c, units):
    g = 0
    for ul in range(len(units) + (1 if c.dynamic else 0)):
        lb = ul & 1
        if ul >= 2:
            yield wait(f"list_empty{lb}", (ul >> 1) - 1)
        if ul == len(units):  # dynamic: no unit left, the end marker
            c.info[lb] = END
            c.mb[f"list_full{lb}"].arrive()
            return
        nst = units[ul]
        c.count[lb] = nst
        c.info[lb] = (nst, ul + 1 < len(units))
        c.mb[f"list_full{lb}"].arrive()
        for _ in range(nst):
            if g >= 3:
                yield wait(f"k_empty{g % 3}", g // 3 - 1)
            c.mb[f"k_full{g % 3}"].arrive()  # the TMA copy lands
            g += 1
            yield ("step",)


def unit_range(c, units):
    return range(len(units) + 1) if c.dynamic else range(len(units))


def producer_v(c, units):
    g = 0
    for ul in unit_range(c, units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        if c.info[lb] == END:
            return
        nst = c.info[lb][0]
        assert c.count[lb] == nst == units[ul]
        for _ in range(nst):
            if g >= 3:
                yield wait(f"v_empty{g % 3}", g // 3 - 1)
            c.mb[f"v_full{g % 3}"].arrive()
            g += 1
            yield ("step",)
        c.mb[f"list_empty{lb}"].arrive()


def mma_qk(c, units, rng):
    g = 0
    for ul in unit_range(c, units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        if c.info[lb] == END:
            return
        nst = c.info[lb][0]
        yield wait("q_full", ul)
        for t in range(nst):
            gs = g + t
            if gs >= 1:
                yield wait("s_free", gs - 1)
            yield wait(f"k_full{gs % 3}", gs // 3)
            c.commit("qk", "s_full0" if c.shared_s_full else f"s_full{gs & 1}", rng)
            c.commit("qk", f"k_empty{gs % 3}", rng)
        c.commit("qk", "q_empty", rng)
        c.mb[f"list_empty{lb}"].arrive()
        g += nst


def mma_pv(c, units, rng, gate_empty=True):
    g = 0
    for ul in unit_range(c, units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        if c.info[lb] == END:
            return
        nst = c.info[lb][0]
        if ul >= 1 and (nst > 0 or gate_empty):
            yield wait("o_free", ul - 1)
        for t in range(nst):
            gs = g + t
            yield wait("p_full", gs)
            yield wait(f"v_full{gs % 3}", gs // 3)
            c.commit("pv", f"pv_grp{gs & 1}", rng)
            c.commit("pv", f"v_empty{gs % 3}", rng)
        c.commit("pv", "unit_done", rng)
        c.mb[f"list_empty{lb}"].arrive()
        g += nst


def softmax(c, units, warp, rng, p_waits_own=False):
    quarter = warp & 3
    G = (warp - 4) >> 2
    bar = ("nbar", 1 + quarter)
    g = jg = 0
    if G == 0:
        c.mb["q_full"].arrive()  # the first unit's Q (every CTA has a first unit)
    for ul in unit_range(c, units):
        lb = ul & 1
        yield wait(f"list_full{lb}", ul >> 1)
        if c.info[lb] == END:
            return
        nst, has_next = c.info[lb]
        if not c.dynamic:
            has_next = ul + 1 < len(units)  # the static schedule knows its unit count
        first = True
        for t in range((g + G) & 1, nst, 2):
            gs = g + t
            yield wait("s_full0" if c.shared_s_full else f"s_full{G}", jg if not c.shared_s_full else gs)
            jg += 1
            c.mb["s_free"].arrive()
            if gs > 0 and not p_waits_own:  # P: P.V(gs - 1), the other group's, has read it
                yield wait(f"pv_grp{G ^ 1}", (gs - 1) >> 1)
            elif gs > 1:  # planted: waits for this group's own previous P.V instead
                yield wait(f"pv_grp{G}", (gs - 2) >> 1)
            yield check(lambda gs=gs: gs == 0 or c.mb[f"pv_grp{(gs - 1) & 1}"].done > (gs - 1) >> 1,
                        f"P({gs}) written before P.V({gs - 1}) completed")
            if not first and rng.random() < 0.5:  # a row's max grew: rescale this group's O
                yield wait(f"pv_grp{G}", (gs - 2) >> 1)
                yield check(lambda gs=gs: c.mb[f"pv_grp{gs & 1}"].done > (gs - 2) >> 1,
                            f"O rescaled before P.V({gs - 2}) completed")
            c.mb["p_full"].arrive()
            first = False
        if ((g + nst) & 1) == G and has_next:  # stage the next unit's Q
            yield wait("q_empty", ul)
            c.mb["q_full"].arrive()
        c.mb[f"list_empty{lb}"].arrive()
        yield bar  # (m, l) exchange with the other group's warp of this quarter
        yield wait("unit_done", ul)
        yield check(lambda e0=(g + nst + 1) >> 1, e1=(g + nst) >> 1:
                    c.mb["pv_grp0"].done >= e0 and c.mb["pv_grp1"].done >= e1,
                    "epilogue before the unit's last P.V")
        c.mb["o_free"].arrive()
        g += nst


def run(units, seed, gate_empty=True, shared_s_full=False, p_waits_own=False, dynamic=True):
    rng = random.Random(seed)
    c = Cta(shared_s_full, dynamic)
    warps = {0: producer_k(c, units), 1: mma_qk(c, units, rng), 2: producer_v(c, units),
             3: mma_pv(c, units, rng, gate_empty)}
    for w in range(4, 12):
        warps[w] = softmax(c, units, w, random.Random(seed * 31 + (w & 3)), p_waits_own)
    blocked, finished = {}, set()
    nbar_count, nbar_gen = {}, {}
    while len(finished) < len(warps):
        for q in c.queues.values():  # each issuer's commits arrive in issue order
            if q:
                q[0][1] -= 1
                if q[0][1] < 0:
                    c.mb[q.pop(0)[0]].arrive()
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
            elif op[0] == "check":
                if not op[1]():
                    return f"hazard: warp {w}: {op[2]}"
            elif op[0] == "nbar":  # bar.sync id, 64: one warp of each group, same quarter
                bid = op[1]
                g0 = nbar_gen.get(bid, 0)
                nbar_count[bid] = nbar_count.get(bid, 0) + 1
                if nbar_count[bid] == 2:
                    nbar_count[bid], nbar_gen[bid] = 0, g0 + 1
                else:
                    blocked[w] = ("nbar", bid, g0)
            break
        if not moved and not any(c.queues.values()):
            return "deadlock: " + ", ".join(f"warp {w} at {blocked.get(w)}" for w in sorted(warps)
                                            if w not in finished)
    return "ok"


def unit_sequences(n, seed):
    rng = random.Random(seed)
    return [[rng.choice([0, 1, 2, 3, 4, 5, 39, 40]) for _ in range(rng.randint(1, 7))] for _ in range(n)]


@pytest.mark.parametrize("dynamic", [False, True])
def test_kernel_protocol_never_deadlocks_or_passes_early(dynamic):
    for i, units in enumerate(unit_sequences(400, 1)):
        assert run(units, seed=i, dynamic=dynamic) == "ok", units


@pytest.mark.parametrize("units", [[0], [0, 0, 3], [1], [1, 0, 1], [2, 40, 0, 41], [0, 0, 0], [3, 0, 0, 2]])
def test_kernel_protocol_edge_units(units):
    for seed in range(50):
        assert run(units, seed, dynamic=False) == "ok"
        assert run(units, seed, dynamic=True) == "ok"


@pytest.mark.parametrize("mistake", ["gate_empty", "shared_s_full", "p_waits_own"])
def test_model_catches_planted_mistakes(mistake):
    """An empty unit that does not wait for the previous epilogue (unit_done
    then runs two phases ahead), one S-ready barrier for both groups (the odd
    group's first wait passes before the even step completes), and a P
    write that waits for the group's own previous P.V instead of the other
    group's (P is single-buffered) must each be caught."""
    kw = {"gate_empty": False} if mistake == "gate_empty" else {mistake: True}
    for dynamic in (False, True):
        bad = [run(units, seed=i, dynamic=dynamic, **kw) for i, units in enumerate(unit_sequences(200, 2))]
        assert any(r != "ok" for r in bad)
