"""The mbarrier protocol of grouped_gemm_kernel, checked on the CPU.

A model of one block's roles runs random interleavings of the kernel's
barrier operations:
  code producer  wait c_empty (reuse), then the copy lands on c_full;
  act. producer  wait a_empty (reuse), then the copy lands on x_full;
  expand warps   (phase j = step mod 4, quarter q) wait c_full, arrive
                 c_empty, wait a_empty (reuse), quarter 0 waits x_full,
                 arrive a_full; gate/up: the previous item's epilogue (wait
                 acc_full, arrive acc_empty) after the warp's first step of
                 the next item, or at once when the warp owns no step of it;
  issuing warps  gate/up: both take every item (wait acc_empty before an
                 item, a_full per step, commit a_empty per step and
                 acc_full per item); down: the items alternate, each warp
                 first waits the other's handoff arrival for the item
                 before, then its accumulator's acc_empty;
  down epilogue  wait acc_full[li % 2], arrive acc_empty[li % 2];
  async units    TMA completions and MMA commits, in issue order per issuer,
                 after any delay.
An mbarrier wait on parity P succeeds when the number of completed phases c
has c % 2 != P; a role waiting for completion t is only correct while
c is t or t + 1 (t - 1 or t + 2 alias the parity). Every wait attempt checks
that, and every run must end with all roles done (no deadlock). A negative
control drops the down kernel's handoff barrier and must fail the check."""
import random

import pytest

SC = {2: 12, 1: 16}   # code stages (grouped_gemm_kernel Geo::SC)
SA = 4                # expanded-operand / activation stages (Geo::SA == Geo::SX)


class Bar:
    def __init__(self, count):
        self.count, self.arrived, self.completed = count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count
        if self.arrived == self.count:
            self.arrived, self.completed = 0, self.completed + 1


class PhaseError(AssertionError):
    pass


def run(nproj, n_items, KT, seed, handoff=True):
    rnd = random.Random(seed)
    sc = SC[nproj]
    bars = {}

    def bar(name, count):
        if name not in bars:
            bars[name] = Bar(count)
        return bars[name]

    for s in range(sc):
        bar(("c_full", s), 1), bar(("c_empty", s), 4)
    for s in range(SA):
        bar(("x_full", s), 1), bar(("a_full", s), 4), bar(("a_empty", s), 2 if nproj == 2 else 1)
    if nproj == 2:
        bar(("acc_full", 0), 2), bar(("acc_empty", 0), 16)
    else:
        for p in range(2):
            bar(("acc_full", p), 1), bar(("acc_empty", p), 4), bar(("handoff", p), 1)

    asyncq = []  # pending completions: (issuer, barrier name); per issuer FIFO

    def wait(name, t):
        """Generator step: block until completion t of barrier `name`."""
        while True:
            c = bars[name].completed
            if not (t <= c <= t + 1):
                raise PhaseError(f"wait {name} for completion {t} with {c} completed")
            if c % 2 != t % 2:
                return
            yield False

    def code_producer():
        for g in range(n_items * KT):
            s = g % sc
            if g >= sc:
                yield from wait(("c_empty", s), g // sc - 1)
            asyncq.append(("tma_c", ("c_full", s)))
            yield True

    def act_producer():
        for g in range(n_items * KT):
            s = g % SA
            if g >= SA:
                yield from wait(("a_empty", s), g // SA - 1)
            asyncq.append(("tma_x", ("x_full", s)))
            yield True

    def epilogue_gu(li):
        yield from wait(("acc_full", 0), li)
        bars[("acc_empty", 0)].arrive()
        yield True

    def expand(j, q):
        prev = -1
        for li in range(n_items):
            g0 = li * KT
            for g in range(g0 + (j - g0) % 4, g0 + KT, 4):
                yield from wait(("c_full", g % sc), g // sc)
                bars[("c_empty", g % sc)].arrive()
                if g >= SA:
                    yield from wait(("a_empty", g % SA), g // SA - 1)
                if q == 0:
                    yield from wait(("x_full", g % SA), g // SA)
                bars[("a_full", g % SA)].arrive()
                yield True
                if nproj == 2 and prev >= 0:
                    yield from epilogue_gu(prev)
                    prev = -1
            if nproj == 2:
                if prev >= 0:
                    yield from epilogue_gu(prev)
                prev = li
        if nproj == 2 and prev >= 0:
            yield from epilogue_gu(prev)

    def issuer(p):
        for li in range(n_items):
            if nproj == 1 and li % 2 != p:
                continue
            use = li if nproj == 2 else li // 2
            acc = 0 if nproj == 2 else p
            if nproj == 1 and handoff and li > 0:
                yield from wait(("handoff", p ^ 1), (li - 1) // 2)
            if use > 0:
                yield from wait(("acc_empty", acc), use - 1)
            for kt in range(KT):
                g = li * KT + kt
                yield from wait(("a_full", g % SA), g // SA)
                asyncq.append((("mma", p), ("a_empty", g % SA)))
                yield True
            asyncq.append((("mma", p), ("acc_full", acc)))
            if nproj == 1:
                bars[("handoff", p)].arrive()
            yield True

    def epilogue_dn(q):
        for li in range(n_items):
            yield from wait(("acc_full", li % 2), li // 2)
            bars[("acc_empty", li % 2)].arrive()
            yield True

    roles = [code_producer(), act_producer()]
    roles += [expand(j, q) for j in range(4) for q in range(4)]
    roles += [issuer(0), issuer(1)]
    if nproj == 1:
        roles += [epilogue_dn(q) for q in range(4)]
    live = list(roles)
    stalls = 0
    while live or asyncq:
        moved = False
        # complete one pending async operation (the oldest of a random issuer)
        if asyncq and rnd.random() < 0.5:
            issuers = sorted({a for a, _ in asyncq}, key=str)
            who = rnd.choice(issuers)
            i = next(k for k, (a, _) in enumerate(asyncq) if a == who)
            bars[asyncq.pop(i)[1]].arrive()
            moved = True
        order = list(live)
        rnd.shuffle(order)
        for r in order:
            try:
                if next(r):
                    moved = True
                    break
            except StopIteration:
                live.remove(r)
                moved = True
                break
        if moved:
            stalls = 0
        else:
            if asyncq:
                continue
            stalls += 1
            assert stalls < 3, "deadlock: no role can move and nothing is in flight"
    for name, b in bars.items():
        assert b.arrived == 0, f"{name}: {b.arrived} arrivals left in an open phase"


@pytest.mark.parametrize("nproj", [2, 1])
def test_grouped_barrier_protocol(nproj):
    rnd = random.Random(1234 + nproj)
    for trial in range(150):
        n_items = rnd.randint(1, 7)
        KT = rnd.choice([1, 2, 3, 4, 5, 8, 16, 32])
        run(nproj, n_items, KT, seed=trial)


def test_down_issuers_without_handoff_alias_a_phase():
    # Negative control: without the handoff barrier the second issuing warp
    # waits on step barriers whole items ahead of the first one.
    with pytest.raises(PhaseError):
        for trial in range(50):
            run(1, 4, 16, seed=trial, handoff=False)
