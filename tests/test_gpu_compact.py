"""Active-index compaction on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _run(mask_np, cap=None, ws=None):
    n = mask_np.size
    mask = torch.from_numpy(mask_np).cuda()
    cap = n if cap is None else cap
    idx = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = B.pi_compact(mask, idx, cnt, cap=cap, ws=ws)
    st = B.pi_sync_status(ws)
    return idx.cpu().numpy(), int(cnt.item()), st, ws


@pytest.mark.parametrize("n", [1, 31, 32, 33, 1000, 2049, 11008, 28672, 32768, 49152, 100003, 1 << 20])
def test_compact_bit_exact(n):
    rng = np.random.default_rng(n)
    masks = [np.zeros(n, np.uint8), np.ones(n, np.uint8), (rng.random(n) < 0.05).astype(np.uint8),
             (rng.random(n) < 0.5).astype(np.uint8), rng.integers(0, 256, n).astype(np.uint8)]
    for pos in {0, n - 1, min(31, n - 1), min(32, n - 1), n // 2}:
        m = np.zeros(n, np.uint8)
        m[pos] = 1
        masks.append(m)
    ws = None
    for m in masks:                      # one workspace reused across launches
        idx, cnt, st, ws = _run(m, ws=ws)
        ref = oracle.compact(m)
        assert st == B.PI_OK
        assert cnt == ref.size
        assert np.array_equal(idx[:cnt], ref)
        assert np.all(idx[cnt:] == -7)


def test_compact_capacity_overflow():
    n = 5000
    m = (np.random.default_rng(3).random(n) < 0.3).astype(np.uint8)
    ref = oracle.compact(m)
    cap = ref.size // 2
    idx, cnt, st, _ = _run(m, cap=cap)
    assert st == 5                       # PI_ERR_CAPACITY
    assert cnt == cap
    assert np.array_equal(idx, ref[:cap])


@pytest.mark.parametrize("n", [1000, 8192, 8193, 65537])
@pytest.mark.parametrize("offset", [0, 4, 3])
def test_compact_both_paths(n, offset):
    """Masks of at most 8 Ki entries at a 4-byte-aligned address take the
    one-CTA scan; a misaligned mask or a longer one takes the multi-CTA scan.
    Both give the oracle's list."""
    rng = np.random.default_rng(n + offset)
    m = (rng.random(n) < 0.3).astype(np.uint8)
    buf = torch.zeros(n + 16, dtype=torch.uint8, device="cuda")
    buf[offset:offset + n] = torch.from_numpy(m).cuda()
    mask = buf[offset:offset + n]
    idx = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = B.pi_compact(mask, idx, cnt, cap=n)
    assert B.pi_sync_status(ws) == B.PI_OK
    ref = oracle.compact(m)
    assert int(cnt.item()) == ref.size
    assert np.array_equal(idx.cpu().numpy()[: ref.size], ref)
