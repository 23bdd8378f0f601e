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
                       A producer claims a batch only while its share table
                       (own rows included) has room for the whole batch.
Checked: every active neuron is run exactly once, by its own CTA or through
the queue; every producer stops; a stale entry from an earlier launch (other
tag) is never taken; with share tables of S rows, no row is lost as long as
the layer has at most (S - T + 1) neurons per CTA (the bound under which the
host picks this mode), even when one CTA's range is all active.  A model of
the earlier claim rule (claim while the table is not full, stop reading a
claimed batch when it fills) loses rows in the same setting."""
import random

import pytest

K_OWN, Q_TAKE = 4, 4


def run_protocol(counts, seed, F=None, stale=0, cap=None, old_rule=False):
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
        held = 0
        for j in own_rows[c]:
            ran.append(j)
            held += 1
            yield
        pend, pk = -1, 0
        spins = 0
        while True:
            if pend < 0:
                if cap is not None and (held >= cap if old_rule else held + Q_TAKE > cap):
                    return                      # table full: this CTA takes no more rows
                pend, pk = head, 0
                head += Q_TAKE                  # one atomic add per batch
                yield
            took = 0
            while pk < Q_TAKE:
                if cap is not None and old_rule and held >= cap:
                    break                       # earlier rule: the rest of the batch is never read
                slot = pend + pk
                e = qent[slot] if slot < F else None
                if e is None or e[0] != "now":
                    break
                ran.append(e[1])
                held += 1
                pk += 1
                took += 1
                yield
            if pk == Q_TAKE or (cap is not None and old_rule and held >= cap):
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


@pytest.mark.parametrize("seed", range(6))
def test_share_table_capacity_keeps_every_row(seed):
    """Near-dense tokens: every neuron of the widest queue-mode layer active
    (S - T + 1 neurons per CTA on average, one CTA's range entirely active).
    With the claim rule of the kernel no row is lost."""
    S = 16
    G = 5
    rng = random.Random(seed)
    total = (S - Q_TAKE + 1) * G
    counts = [0] * G
    for _ in range(total):                      # uneven ranges, one of them large
        counts[rng.randrange(G) if rng.random() < 0.6 else 0] += 1
    ran, active = run_protocol(counts, seed, cap=S)
    assert sorted(ran) == sorted(active)


def test_earlier_claim_rule_loses_rows():
    """The earlier rule, on layers it admitted (up to S neurons per CTA): some
    interleaving loses a claimed row."""
    S, G = 16, 5
    lost = 0
    for seed in range(40):
        rng = random.Random(seed)
        counts = [0] * G
        for _ in range(S * G - 3):
            counts[rng.randrange(G) if rng.random() < 0.6 else 0] += 1
        ran, active = run_protocol(counts, seed, cap=S, old_rule=True)
        lost += len(active) - len(ran)
    assert lost > 0
