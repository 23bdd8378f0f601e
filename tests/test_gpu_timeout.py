"""A bounded device wait that runs out, and recovery from it.

The one-kernel layer step synchronises its CTAs with a grid barrier on a
counter in the workspace.  The test makes that barrier's target unreachable
(the workspace's launch sequence number is set far ahead of the arrival
counter, so nothing ever meets it) and shortens the poll limit, a field of
the workspace's control block, so the wait gives up within milliseconds.  The
call must report PI_ERR_TIMEOUT through pi_sync_status and leave the context
usable; after the workspace is zero-filled again, as the library's contract
asks, the next call must match the oracle.  No kernel is made to fault, trap
or spin without a bound."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu

PI_ERR_TIMEOUT = 7
# control block words (uint32 index): error word, poll limit, ..., launch sequence
W_ERR, W_POLL_LIMIT, W_BAR_SEQ = 0, 1, 6


def _check_against_oracle(lay, olay, H, x_np, y):
    """y against the oracle on the predicted list, with the decisions at
    borderline logits taken from an ordered run on a fresh workspace."""
    F = olay.d_ff
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_tmp = torch.empty_like(y)
    ws = B.pi_ffn_layer(lay, torch.from_numpy(x_np).cuda(), y_tmp, idx=idx, n_active=n)
    assert B.pi_sync_status(ws) == 0
    h, logit_ref, M = oracle.predict(olay, x_np)
    amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
    got = set(idx.cpu().numpy()[: int(n.item())].tolist())
    ref = set(np.flatnonzero(M).tolist())
    assert all(amb[j] for j in got ^ ref)
    res = np.array(sorted(got), np.int32)
    assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olay, x_np, res), what="after recovery")


@pytest.mark.parametrize("ordered", [False, True])
def test_grid_barrier_timeout_is_reported_and_recovered(ordered):
    d, F, r = 1024, 4100, 128
    L = synth.make_layer(d, F, r, gated=True, wtype="f16", sparsity=0.85, seed=501, device="cuda")
    lay, olay, H = make_pair(L)
    x_np = synth.tokens(1, d, 502).numpy()[0]
    x = torch.from_numpy(x_np).cuda()
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    idx = torch.zeros(F, dtype=torch.int32, device="cuda") if ordered else None
    n = torch.zeros(1, dtype=torch.int32, device="cuda") if ordered else None
    ws = B.workspace(B.pi_workspace_bytes(lay, 1))
    words = ws.view(torch.int32)

    # a healthy call first, on the same workspace
    B.pi_ffn_layer(lay, x, y, idx=idx, n_active=n, ws=ws)
    assert B.pi_sync_status(ws) == 0

    words[W_POLL_LIMIT] = 2000
    words[W_BAR_SEQ] = 1 << 20          # barrier targets far beyond any arrival count
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    B.pi_ffn_layer(lay, x, y, idx=idx, n_active=n, ws=ws)
    t1.record()
    assert B.pi_sync_status(ws) == PI_ERR_TIMEOUT
    assert t0.elapsed_time(t1) < 2000.0   # ms: the waits gave up promptly
    assert B.pi_sync_status(ws) == 0      # the error word was cleared by the read

    # the context is still usable: the documented recovery is a zero-filled workspace
    ws.zero_()
    for _ in range(2):
        B.pi_ffn_layer(lay, x, y, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        _check_against_oracle(lay, olay, H, x_np, y)
