"""The streamed decode kernel's hand-off protocols, checked on the CPU.

decode_stream_kernel (csrc/decode_fused.cu) meets in two places where an
interleaving, not a value, decides correctness; models of both run random
interleavings and check the waits.

1. The batched ring (several tokens, one block): the producer fills stage
   q % S in fill order (gate/up fills of the units, then the down fills of
   dpack units each) once the stage's previous fill is consumed, and stores
   the fill number lap + 1 after issuing; the 16 compute warps take items
   round-robin (gate/up items, a barrier, down items), and for an item of
   fill q first wait until that fill number is reached, then wait the
   stage's full barrier for completion lap; the warp finishing a fill's last
   item frees the stage. An mbarrier wait for completion t is correct only
   while the completed count is t or t + 1 (the parity aliases otherwise).
   Negative control: without the fill-number wait a warp waits on a later
   lap's parity.
2. The one-token exchange between blocks (G blocks, consecutive calls
   chained so that a call's blocks start after the previous call's blocks
   exit): each block releases unit u once its h rows are out (counter
   cnt[u] += 1), each block's exchange warp polls cnt[u] >= G before copying
   unit u's h, and the last block to count out resets the counters. A poll
   must never pass before every block of the same call released the unit.
   Negative control: without the reset the second call's polls pass on the
   first call's counts."""
import random

import pytest


class PhaseError(AssertionError):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.arrived, self.completed = count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count
        if self.arrived == self.count:
            self.arrived, self.completed = 0, self.completed + 1


def schedule(roles, asyncq, bars, rnd):
    live = list(roles)
    stalls = 0
    while live or asyncq:
        moved = False
        if asyncq and rnd.random() < 0.5:
            bars[asyncq.pop(0)].arrive()  # copies land in issue order (one issuing warp)
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
        elif not asyncq:
            stalls += 1
            assert stalls < 3, "deadlock: no role can move and nothing is in flight"


def run_ring(S, units, ng, dpack, seed, wait_fill=True):
    rnd = random.Random(seed)
    W = 16
    U = len(units)
    uoff = [0]
    for c in units:
        uoff.append(uoff[-1] + c)
    Qd = (U + dpack - 1) // dpack
    Q = U + Qd
    bars = {}
    for s in range(S):
        bars[("full", s)] = Bar(1)
        bars[("empty", s)] = Bar(1)
    fillno = [0] * S
    fdone = [0] * Q
    need = [units[u] * ng for u in range(U)] + [uoff[min(U, (j + 1) * dpack)] - uoff[j * dpack] for j in range(Qd)]
    asyncq = []
    gate_done = [0]

    def wait(name, t):
        while True:
            c = bars[name].completed
            if not (t <= c <= t + 1):
                raise PhaseError(f"wait {name} for completion {t} with {c} completed")
            if c % 2 != t % 2:
                return
            yield False

    def producer():
        for q in range(Q):
            s, lap = q % S, q // S
            if lap > 0:
                yield from wait(("empty", s), lap - 1)
            asyncq.append(("full", s))
            fillno[s] = lap + 1
            yield True

    def consume(q):
        s, lap = q % S, q // S
        if wait_fill:
            while fillno[s] <= lap:
                yield False
        yield from wait(("full", s), lap)
        fdone[q] += 1
        if fdone[q] == need[q]:
            bars[("empty", s)].arrive()
        yield True

    def compute(w):
        NG = uoff[U] * ng
        for j in range(w, NG, W):
            c = j // ng
            u = next(i for i in range(U) if uoff[i + 1] > c)
            yield from consume(u)
        gate_done[0] += 1
        while gate_done[0] < W:  # the grid barrier between gate/up and down items
            yield False
        for j in range(w, uoff[U], W):
            u = next(i for i in range(U) if uoff[i + 1] > j)
            yield from consume(U + u // dpack)

    schedule([producer()] + [compute(w) for w in range(W)], asyncq, bars, rnd)
    assert all(fdone[q] == need[q] for q in range(Q))


def run_exchange(G, calls, seed, reset=True):
    rnd = random.Random(seed)
    cnt = {}
    released = {}  # (call, u) -> blocks that released
    out = [0]
    exited = [0]
    bad = []

    def block(call, b, U):
        # compute warps release each unit after their gate/up items (any order)
        order = list(range(U))
        rnd.shuffle(order)
        pending_polls = set(range(U))

        def release():
            u = order.pop()
            cnt[u] = cnt.get(u, 0) + 1
            released[(call, u)] = released.get((call, u), 0) + 1

        while order or pending_polls:
            if order and rnd.random() < 0.5:
                release()
                yield True
                continue
            polled = False
            for u in rnd.sample(sorted(pending_polls), len(pending_polls)):
                if cnt.get(u, 0) >= G:
                    if released.get((call, u), 0) < G:
                        bad.append((call, b, u, released.get((call, u), 0)))
                    pending_polls.discard(u)
                    polled = True
                    break
            if polled:
                yield True
            elif order:
                release()
                yield True
            else:
                yield False
        # count out after the last poll; the last block out resets the counters
        out[0] += 1
        if out[0] == G:
            if reset:
                for u in list(cnt):
                    cnt[u] = 0
            out[0] = 0
        exited[0] += 1
        yield True

    for call in range(calls):
        U = rnd.randint(1, 16)
        exited[0] = 0
        schedule([block(call, b, U) for b in range(G)], [], {}, rnd)
        assert exited[0] == G
        assert not reset or all(v == 0 for v in cnt.values())
    return bad


def test_batched_ring_protocol():
    rnd = random.Random(99)
    for trial in range(200):
        S = rnd.randint(1, 12)
        units = [rnd.randint(1, 6) for _ in range(rnd.randint(1, 20))]
        run_ring(S, units, ng=rnd.choice([1, 2, 4]), dpack=rnd.choice([1, 2, 3]), seed=trial)


def test_batched_ring_without_fill_numbers_aliases_a_phase():
    with pytest.raises(PhaseError):
        for trial in range(100):
            run_ring(2, [3, 1, 4, 1, 5, 2, 6], ng=2, dpack=2, seed=trial, wait_fill=False)


def test_one_token_exchange_protocol():
    for trial in range(100):
        assert run_exchange(G=random.Random(trial).randint(1, 6), calls=3, seed=trial) == []


def test_one_token_exchange_without_reset_reads_stale_counts():
    assert any(run_exchange(G=4, calls=2, seed=t, reset=False) for t in range(20))
