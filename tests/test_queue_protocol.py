"""The one-kernel layer's queue-mode work distribution as a protocol model, run
on CPU under random interleavings of the CTAs' steps.

Protocol (as in the kernel, batch 1, no ordered list requested):
  publisher of CTA c   keeps the first K active neurons of its range for its
                       own producer, reserves count - K queue slots with one
                       atomic add on the tail, writes one tagged entry per
                       reserved slot (in any order), then counts itself done;
  producer of CTA c    runs its own rows, then takes T slots per atomic add on
                       the head, reads them in slot order, takes each entry
                       whose tag is this launch's, and stops once every CTA is
                       done and its next slot is at or past the final tail.
Checked: every active neuron is run exactly once, by its own CTA or through
the queue; every producer stops; a stale entry from an earlier launch (other
tag) is never taken."""
import random

import pytest

K_OWN, Q_TAKE = 4, 4


def run_protocol(counts, seed, F=None, stale=0):
    rng = random.Random(seed)
    G = len(counts)
    ranges, base = [], 0
    for c, n in enumerate(counts):
        ranges.append(list(range(base, base + n)))
        base += n + rng.randrange(0, 5)         # inactive neurons between ranges
    F = F or base + 1
    qent = [("old", -1)] * stale + [None] * (F - stale)   # entries of an earlier launch
    tail, head, done = 0, 0, 0
    ran = []

    def publisher(c):
        nonlocal tail, done
        act = ranges[c]
        own = min(len(act), K_OWN)
        own_rows[c] = act[:own]
        ready[c] = True
        yield
        qbase = tail
        tail += len(act) - own                  # the atomic add returns the old tail
        yield
        order = list(range(own, len(act)))
        rng.shuffle(order)
        for k in order:                         # entries land in any order
            qent[qbase + (k - own)] = ("now", act[k])
            yield
        done += 1                               # release: after every entry

    def producer(c):
        nonlocal head
        while not ready[c]:
            yield
        for j in own_rows[c]:
            ran.append(j)
            yield
        pend, pk = -1, 0
        spins = 0
        while True:
            if pend < 0:
                pend, pk = head, 0
                head += Q_TAKE                  # one atomic add per batch
                yield
            took = 0
            while pk < Q_TAKE:
                slot = pend + pk
                e = qent[slot] if slot < F else None
                if e is None or e[0] != "now":
                    break
                ran.append(e[1])
                pk += 1
                took += 1
                yield
            if pk == Q_TAKE:
                pend = -1
                continue
            if took:
                spins = 0
                continue
            if done == G and pend + pk >= tail:
                return                          # the tail is final and reached
            spins += 1
            assert spins < 100000, "producer never finished"
            yield

    own_rows = [[] for _ in range(G)]
    ready = [False] * G
    agents = [publisher(c) for c in range(G)] + [producer(c) for c in range(G)]
    live = list(range(len(agents)))
    while live:
        i = rng.choice(live)
        try:
            next(agents[i])
        except StopIteration:
            live.remove(i)
    return ran, [j for r in ranges for j in r]


@pytest.mark.parametrize("seed", range(12))
def test_queue_protocol_runs_every_active_neuron_once(seed):
    rng = random.Random(1000 + seed)
    G = rng.choice([3, 8, 152])
    # range counts from empty to far above the own share, some all-zero ranges
    counts = [rng.choice([0, 0, 1, 3, 4, 5, 7, 12, 30]) for _ in range(G)]
    ran, active = run_protocol(counts, seed)
    assert sorted(ran) == sorted(active)


def test_queue_protocol_edge_cases():
    for counts in ([0, 0, 0], [4, 4, 4], [0, 0, 50], [1], [K_OWN + 1] * 5):
        ran, active = run_protocol(counts, 5)
        assert sorted(ran) == sorted(active), counts


def test_stale_entries_of_an_earlier_launch_are_never_taken():
    # slots beyond this launch's tail still hold an earlier launch's entries
    ran, active = run_protocol([6, 9, 0, 12], 3, F=80, stale=80)
    assert sorted(ran) == sorted(active)
    assert -1 not in ran
