"""Bounded waits that run out, as a protocol model on the CPU.

The cross-CTA count scan of the predictor kernel: CTA c owns a contiguous
range of neurons, publishes its active count in a status word tagged with the
launch's epoch, then sums the counts of all CTAs before it, polling each
predecessor's word until it carries this launch's tag; a poll that reaches its
limit sets the error bit, counts that predecessor as 0 and goes on.  Each CTA
then writes its active neurons at (prefix + local position), only where that
position is below the list's capacity.  The last CTA to finish moves the epoch
on.  Here one CTA never publishes (a flag that nothing sets): every other CTA
must still finish, report the timeout, and write nothing outside the list.
After the workspace is zero-filled again, a launch gives the exact list."""
import random

import numpy as np

ERR_TIMEOUT = 1


def run_scan(masks, ws, cap, silent=(), limit=50, seed=0):
    rng = random.Random(seed)
    G = len(masks)
    sizes = [len(m) for m in masks]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    idx = [None] * cap
    writes = []
    epoch = ws["epoch"]
    want = (epoch << 1) | 1

    def cta(c):
        count = int(np.count_nonzero(masks[c]))
        if c in silent:
            return                              # never publishes, never finishes
        ws["status"][c] = (want, count)
        yield
        total = 0
        for i in range(c):
            spins = 0
            while ws["status"][i][0] != want:
                spins += 1
                if spins > limit:
                    ws["err"] |= ERR_TIMEOUT
                    break
                yield
            else:
                total += ws["status"][i][1]
        local = np.flatnonzero(masks[c])
        for k, j in enumerate(local):
            pos = total + k
            writes.append(pos)
            if pos < cap:
                idx[pos] = int(offs[c] + j)
            yield
        ws["done"] += 1
        if ws["done"] == G:
            ws["done"] = 0
            ws["epoch"] += 1

    agents = [cta(c) for c in range(G)]
    live = list(range(G))
    steps = 0
    while live:
        i = rng.choice(live)
        try:
            next(agents[i])
        except StopIteration:
            live.remove(i)
        steps += 1
        assert steps < 10 ** 6, "a CTA never finished"
    return idx, writes


def fresh_ws(G):
    return {"err": 0, "epoch": 0, "done": 0, "status": [(0, 0)] * G}


def test_scan_gives_up_on_a_silent_predecessor_and_stays_in_bounds():
    rng = np.random.default_rng(3)
    G, cap = 7, 40
    masks = [(rng.random(12) < 0.5).astype(np.uint8) for _ in range(G)]
    ws = fresh_ws(G)
    idx, writes = run_scan(masks, ws, cap, silent={2}, seed=1)
    assert ws["err"] & ERR_TIMEOUT
    assert all(0 <= p for p in writes)
    assert all(v is None or 0 <= v < 12 * G for v in idx)
    # the recovery the library documents: zero-fill, then a clean launch
    ws = fresh_ws(G)
    idx, _ = run_scan(masks, ws, 12 * G, seed=2)
    ref = np.flatnonzero(np.concatenate(masks))
    assert ws["err"] == 0
    assert idx[: ref.size] == ref.tolist()


def test_scan_without_a_silent_cta_never_times_out():
    rng = np.random.default_rng(4)
    for seed in range(10):
        G = 1 + seed
        masks = [(rng.random(9) < 0.3).astype(np.uint8) for _ in range(G)]
        ws = fresh_ws(G)
        for launch in range(3):                 # the epoch moves on; stale words are ignored
            idx, _ = run_scan(masks, ws, 9 * G, limit=10 ** 5, seed=seed * 10 + launch)
            ref = np.flatnonzero(np.concatenate(masks))
            assert ws["err"] == 0
            assert idx[: ref.size] == ref.tolist()
            assert ws["epoch"] == launch + 1
