"""GPU parity of the batched (2..8 tokens) union path against the oracle.

Every token of the batch is computed on every row of the union list, so the
oracle reference for token b is its sparse FFN over that same list.  Sizes span
several row tiles, ragged tiles (n % 16 != 0), ragged d_model chunks, both
operand-group layouts (batch <= 4 and > 4), fp16 and Q4_0, gated and not."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu

SHAPES = [  # d_model, d_ff, rank
    (256, 1000, 64),
    (520, 2049, 32),     # d_model not a multiple of 32 (fp16 only): ragged last step
    (1024, 4100, 128),
]


def _layer(d, F, r, gated, wtype, seed, sparsity=0.8, act=0):
    L = synth.make_layer(d, F, r, gated=gated, wtype="f16", sparsity=sparsity, predictor="projection", seed=seed,
                         device="cuda")
    L["wtype"] = wtype
    return make_pair(L, act=act)


def _union_true(olay, X):
    m = np.zeros(olay.d_ff, dtype=np.uint8)
    for x in X:
        m |= oracle.true_mask(olay, x)[0]
    return oracle.compact(m)


@pytest.mark.parametrize("batch", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("wtype", ["f16", "q4_0"])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_union_sparse_ffn(batch, wtype, gated, shape):
    d, F, r = shape
    if wtype == "q4_0" and d % 256:
        pytest.skip("Q4_0 needs d_model % 256")
    lay, olay, H = _layer(d, F, r, gated, wtype, seed=d + F + batch)
    X = synth.tokens(batch, d, 21 + batch).numpy()
    idx_np = _union_true(olay, X)
    x = torch.from_numpy(X).cuda()
    idx = torch.from_numpy(idx_np).cuda()
    n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    ws = B.pi_sparse_ffn(lay, x, idx, n, y)
    assert B.pi_sync_status(ws) == 0
    yg = y.cpu().numpy()
    for b in range(batch):
        assert_ffn_close(yg[b], oracle.sparse_ffn(olay, X[b], idx_np),
                         what=f"{wtype} gated={gated} {shape} B={batch} token {b}")
    # the same workspace again (its per-tile buffers must have been left zero)
    y.fill_(float("nan"))
    B.pi_sparse_ffn(lay, x, idx, n, y, ws=ws)
    assert B.pi_sync_status(ws) == 0
    assert np.array_equal(np.isnan(y.cpu().numpy()), np.zeros_like(yg, dtype=bool))
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], idx_np), what=f"repeat token {b}")


@pytest.mark.parametrize("act", [0, 1])
def test_union_relu2_residual_in_place(act):
    d, F, r, batch = 512, 3000, 64, 6
    lay, olay, H = _layer(d, F, r, True, "f16", seed=91, act=act)
    X = synth.tokens(batch, d, 4).numpy()
    idx_np = _union_true(olay, X)
    R = synth.tokens(batch, d, 5).numpy()
    y = torch.from_numpy(R.copy()).cuda()  # residual == y
    n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
    ws = B.pi_sparse_ffn(lay, torch.from_numpy(X).cuda(), torch.from_numpy(idx_np).cuda(), n, y, residual=y)
    assert B.pi_sync_status(ws) == 0
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], idx_np) + R[b], what=f"act={act} b={b}")


def test_union_edge_cases():
    d, F, r, batch = 256, 700, 32, 4
    lay, olay, H = _layer(d, F, r, False, "f16", seed=7)
    X = synth.tokens(batch, d, 3).numpy()
    x = torch.from_numpy(X).cuda()
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    ws = None
    for idx_np in (np.zeros(0, np.int32), np.array([5], np.int32), np.arange(17, dtype=np.int32),
                   np.arange(F, dtype=np.int32)):
        idx = torch.from_numpy(idx_np if idx_np.size else np.zeros(1, np.int32)).cuda()
        n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
        ws = B.pi_sparse_ffn(lay, x, idx, n, y, ws=ws)
        assert B.pi_sync_status(ws) == 0
        for b in range(batch):
            assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], idx_np), what=f"n={idx_np.size} b={b}")
    # the dense FFN at batch 4 runs the same kernels over all rows
    B.pi_dense_ffn(lay, x, y, ws=ws)
    assert B.pi_sync_status(ws) == 0
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.dense_ffn(olay, X[b]), what=f"dense b={b}")


def test_union_large_magnitudes():
    """Tokens far outside fp16 range: the per-token power-of-two scaling keeps
    the fp16 operand terms finite and the result relative-accurate."""
    d, F, r, batch = 512, 1500, 32, 3
    lay, olay, H = _layer(d, F, r, False, "f16", seed=13)
    X = synth.tokens(batch, d, 6).numpy() * np.array([[1e6], [1e-5], [3.0]], dtype=np.float32)
    idx_np = np.arange(0, F, 3, dtype=np.int32)
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
    ws = B.pi_sparse_ffn(lay, torch.from_numpy(X).cuda(), torch.from_numpy(idx_np).cuda(), n, y)
    assert B.pi_sync_status(ws) == 0
    for b in range(batch):
        ref = oracle.sparse_ffn(olay, X[b], idx_np)
        err = np.linalg.norm(y.cpu().numpy()[b] - ref) / np.linalg.norm(ref)
        assert err <= 1e-3, (b, err)


def test_union_bad_index_flagged_and_skipped():
    d, F, r, batch = 256, 600, 32, 2
    lay, olay, H = _layer(d, F, r, False, "f16", seed=8)
    X = synth.tokens(batch, d, 2).numpy()
    idx_np = np.array([1, 2, F + 5, 9], dtype=np.int32)
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
    ws = B.pi_sparse_ffn(lay, torch.from_numpy(X).cuda(), torch.from_numpy(idx_np).cuda(), n, y)
    assert B.pi_sync_status(ws) == 10    # PI_ERR_INDEX
    good = np.array([1, 2, 9], dtype=np.int32)
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], good), what=f"bad index skipped b={b}")
    assert B.pi_sync_status(ws) == 0     # cleared


@pytest.mark.parametrize("batch", [3, 8])
@pytest.mark.parametrize("wtype", ["f16", "q4_0"])
def test_union_ffn_layer(batch, wtype):
    """Predictor union + compaction + union FFN through pi_ffn_layer."""
    d, F, r = 1024, 4100, 128
    lay, olay, H = _layer(d, F, r, False, wtype, seed=5 + batch)
    X = synth.tokens(batch, d, 30 + batch).numpy()
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = B.pi_ffn_layer(lay, torch.from_numpy(X).cuda(), y, idx=idx, n_active=n)
    assert B.pi_sync_status(ws) == 0
    got_list = idx.cpu().numpy()[: int(n.item())]
    assert np.all(np.diff(got_list) > 0)
    ref, amb = set(), np.zeros(F, dtype=bool)
    for b in range(batch):
        h, logit, M = oracle.predict(olay, X[b])
        ref |= set(np.flatnonzero(M).tolist())
        amb |= ambiguous(logit, logit_scale(H, h), olay.threshold)
    got = set(got_list.tolist())
    assert all(amb[j] for j in got ^ ref)
    idx_res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), dtype=np.int32)
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], idx_res), what=f"{wtype} B={batch} b={b}")


@pytest.mark.parametrize("batch", [4, 8])
@pytest.mark.parametrize("name", ["falcon40b-relu-fp16", "falcon40b-relu-q4_0"])
def test_union_workload_full_size(name, batch):
    """The Falcon-40B-shaped layer at batch 4 and 8 (union of ~90%-sparse
    per-token sets), every token compared in full."""
    w = synth.WORKLOADS[name]
    L = synth.workload_layer(w, 0, device="cuda")
    lay, olay, H = make_pair(L)
    X = synth.workload_tokens(w, n=batch, device="cpu").numpy()
    m = np.zeros(w.d_ff, dtype=np.uint8)
    for b in range(batch):
        m |= oracle.predict(olay, X[b])[2]
    idx_np = oracle.compact(m)
    y = torch.empty(batch, w.d_model, dtype=torch.float32, device="cuda")
    n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
    ws = B.pi_sparse_ffn(lay, torch.from_numpy(X).cuda(), torch.from_numpy(idx_np).cuda(), n, y)
    assert B.pi_sync_status(ws) == 0
    for b in range(batch):
        assert_ffn_close(y.cpu().numpy()[b], oracle.sparse_ffn(olay, X[b], idx_np), what=f"{name} B={batch} b={b}")
