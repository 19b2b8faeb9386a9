"""Stream ordering of the residency manager, checked without a GPU.

The manager logs every stream operation it enqueues (event records, waits,
host-to-device copies, slot-table publishes); a dry run logs the same
operations without enqueuing them. This test interleaves the caller's expert
reads (on the compute stream, after each prepare, one per needed expert's
published slot) and replays the whole host-ordered sequence with vector
clocks over the two streams. It checks the "03 / Arquitetura" (ADR 0009)
rules: a slot is overwritten only after every earlier reader of it has
finished (reuse only after readers retire), and a reader sees the copy of the
expert the published table names for that slot (readers see a valid
generation)."""
import numpy as np
import pytest

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding

moe = binding()
COMPUTE, COPY = 0, 1
READ = 99  # the caller's expert read, a compute-stream operation of this test


class Replay:
    """Host-ordered operations with vector clocks (one component per stream)."""

    def __init__(self):
        self.vc = {COMPUTE: [0, 0], COPY: [0, 0]}
        self.ev = {}
        self.ops = []  # (kind, stream, layer, slot, expert, vc)

    def add(self, kind, stream, event=-1, layer=-1, slot=-1, expert=-1):
        v = self.vc[stream]
        if kind == moe.MOE_OP_WAIT:
            if event in self.ev:  # a wait on a never-recorded event waits for nothing
                self.vc[stream] = [max(a, b) for a, b in zip(v, self.ev[event])]
            return
        v[stream] += 1
        if kind == moe.MOE_OP_RECORD:
            self.ev[event] = list(v)
        self.ops.append((kind, stream, layer, slot, expert, list(v)))

    @staticmethod
    def before(a, b):
        """Operation a happens before operation b on the device."""
        return a[5][a[1]] <= b[5][a[1]]

    def violations(self, initial):
        """initial[(layer, slot)] = expert placed at creation (complete before any op)."""
        bad = []
        for i, b in enumerate(self.ops):
            if b[0] == moe.MOE_OP_COPY:
                # Every earlier reader of the slot must have finished.
                for a in self.ops[:i]:
                    if a[0] == READ and (a[2], a[3]) == (b[2], b[3]) and not self.before(a, b):
                        bad.append(("copy overtakes a reader", i, b[2], b[3]))
            elif b[0] == READ:
                # The slot's latest copy (host order) holds the expected expert and lands first.
                last = None
                for a in self.ops[:i]:
                    if a[0] == moe.MOE_OP_COPY and (a[2], a[3]) == (b[2], b[3]):
                        last = a
                holder = initial.get((b[2], b[3])) if last is None else last[4]
                if holder != b[4]:
                    bad.append(("reader sees another expert", i, b[2], b[3], holder, b[4]))
                elif last is not None and not self.before(last, b):
                    bad.append(("reader overtakes its copy", i, b[2], b[3]))
        return bad


def run_scenario(E=12, C=4, S=0, L=2, k=2, T=2, steps=60, policy="decay", prefetch=False, inject_at=None,
                 drop=None):
    """Drive a dry-run manager like a decode loop; returns (replay, initial placement)."""
    ranks = synth.zipf_ranks(3, 0, E)
    profile = np.tile(1.0 / ranks.astype(np.float64), (L, 1))
    pinned = max(0, C - T * k) if policy == "pinned" else 0
    cfg = dict(layers=L, experts=E, slots=C, spares=S, max_ids_per_step=T * k, dry_run=1, log_ops=1,
               block_bytes=4096, decay=0.9, policy=policy, pinned=pinned,
               profile=profile if policy == "pinned" else None)
    h = moe.moe_residency_create(cfg, None, None, None)
    rp = Replay()
    initial = {}
    seen = [0]

    def pull():
        ops = moe.moe_residency_ops(h)
        for (kind, stream, event, layer, slot, expert) in ops[seen[0]:]:
            if drop is not None and drop(kind, stream, event):
                continue
            rp.add(kind, stream, event, layer, slot, expert)
        seen[0] = len(ops)

    try:
        for l in range(L):
            for e, s in enumerate(moe.moe_residency_slot_table(h, l, E)):
                if s >= 0:
                    initial[(l, int(s))] = e
        n_prepare = 0
        injected = False
        for step in range(steps):
            for l in range(L):
                lg = synth.logits_zipf(3, l, step, T, E, 1.0)
                ids, _ = moe_oracle.route(lg, k, False)
                if inject_at is not None and n_prepare >= inject_at and not injected:
                    # The step's first copy fails; a step with no copy leaves the hook armed.
                    moe.moe_residency_inject_copy_failure(h, 0)
                    try:
                        moe.moe_residency_prepare(h, l, ids)
                        moe.moe_residency_inject_copy_failure(h, -1)
                    except moe.MoeError:
                        injected = True
                    pull()
                    if injected:
                        moe.moe_residency_prepare(h, l, ids)  # the retried step
                else:
                    moe.moe_residency_prepare(h, l, ids)
                n_prepare += 1
                pull()
                table = moe.moe_residency_slot_table(h, l, E)
                for e in sorted(set(ids.reshape(-1).tolist())):
                    rp.add(READ, COMPUTE, layer=l, slot=int(table[e]), expert=e)
                if prefetch:
                    nl = (l + 1) % L
                    counts = moe.moe_residency_counts(h, nl, E)
                    tab = moe.moe_residency_slot_table(h, nl, E)
                    cand = [e for e in np.lexsort((np.arange(E), -counts)) if tab[e] < 0][:S]
                    moe.moe_residency_prefetch(h, nl, cand)
                    pull()
        st = moe.moe_residency_get_stats(h)
        assert inject_at is None or injected
    finally:
        moe.moe_residency_destroy(h)
    return rp, initial, st


@pytest.mark.parametrize("kw", [
    dict(S=0),
    dict(S=2),
    dict(S=3, prefetch=True),
    dict(S=3, prefetch=True, policy="lru"),
    dict(S=2, prefetch=True, policy="pinned", C=6),
    dict(S=0, inject_at=17),
    dict(S=2, prefetch=True, inject_at=23),
])
def test_ordering_has_no_race(kw):
    rp, initial, st = run_scenario(**kw)
    assert st["misses"] > 20  # the scenario exercises evictions and copies
    if kw.get("prefetch"):
        assert st["prefetched"] > 0
    assert rp.violations(initial) == []


def test_checker_sees_a_missing_reader_wait():
    # Without the copy stream's wait on "readers done", in-place reuse of a
    # victim's slot overtakes that slot's earlier readers.
    rp, initial, _ = run_scenario(S=0, drop=lambda kind, stream, event: kind == moe.MOE_OP_WAIT and
                                  stream == COPY and event == 0)
    assert any(v[0] == "copy overtakes a reader" for v in rp.violations(initial))


def test_prefetch_copies_need_no_wait_of_their_own():
    # A prefetch adds no wait: the slots it fills were freed by a prepare()
    # whose copy-stream wait follows their readers, and the copy stream runs
    # in order. Dropping every wait except that one keeps the log race-free.
    rp, initial, st = run_scenario(S=3, prefetch=True,
                                   drop=lambda kind, stream, event: kind == moe.MOE_OP_WAIT and
                                   not (stream == COPY and event == 0) and not (stream == COMPUTE and event == 1))
    assert st["prefetch_copies"] > 0 and rp.violations(initial) == []


def test_checker_sees_a_missing_publish_wait():
    # Without the compute stream's wait on "copies done", readers overtake
    # the copies of the experts they read.
    rp, initial, _ = run_scenario(S=2, drop=lambda kind, stream, event: kind == moe.MOE_OP_WAIT and
                                  stream == COMPUTE and event == 1)
    assert any(v[0] == "reader overtakes its copy" for v in rp.violations(initial))
