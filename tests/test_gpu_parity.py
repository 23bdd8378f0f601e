"""GPU parity against the oracle on seeded inputs at sizes the oracle finishes
in seconds: several CTAs / scan tiles, ragged d_ff, every weight format,
gated and non-gated, ReLU and squared ReLU, the edge cases.  Calls go through
the C ABI (the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair, q4_blob_random

pytestmark = pytest.mark.gpu

SHAPES = [  # d_model, d_ff, rank
    (256, 1000, 64),
    (512, 2049, 32),
    (1024, 4100, 128),
]


def _layer(d, F, r, gated, wtype, seed, sparsity=0.8, predictor="projection", act=0):
    L = synth.make_layer(d, F, r, gated=gated, wtype="f32" if wtype == "f32" else "f16", sparsity=sparsity,
                         predictor=predictor, seed=seed, device="cuda")
    L["wtype"] = wtype
    return make_pair(L, act=act)


def _cuda(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


# ---------------------------------------------------------------- sparse FFN, given idx
@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_sparse_ffn_true_mask(wtype, gated, shape):
    d, F, r = shape
    if wtype == "q4_0" and d % 256:
        pytest.skip("Q4_0 needs d_model % 256")
    lay, olay, H = _layer(d, F, r, gated, wtype, seed=d + F)
    X = synth.tokens(3, d, 5).numpy()
    ws = None
    for t in range(3):
        T, _ = oracle.true_mask(olay, X[t])
        idx_np = oracle.compact(T)
        y_ref = oracle.sparse_ffn(olay, X[t], idx_np)
        x = _cuda(X[t])
        idx = _cuda(idx_np)
        n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_sparse_ffn(lay, x, idx, n, y, ws=ws)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"{wtype} gated={gated} {shape} t={t}")


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("gated", [False, True])
def test_sparse_ffn_predicted_mask_and_relu2(act, gated):
    d, F, r = 512, 3000, 64
    lay, olay, H = _layer(d, F, r, gated, "f16", seed=77, act=act)
    X = synth.tokens(2, d, 8).numpy()
    for t in range(2):
        _, _, M = oracle.predict(olay, X[t])
        idx_np = oracle.compact(M)
        y_ref = oracle.sparse_ffn(olay, X[t], idx_np)
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
        ws = B.pi_sparse_ffn(lay, _cuda(X[t]), _cuda(idx_np), n, y)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"act={act} gated={gated}")


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
def test_integer_layers_bit_exact(gated, wtype):
    """Small-integer weights and tokens: every fp32 partial sum is an exact
    integer, so GPU and oracle agree bit for bit whatever the order."""
    d, F, r = 512, 1500, 16
    L = synth.integer_layer(d, F, r, gated=gated, wtype="f32" if wtype == "f32" else "f16", seed=5, device="cuda")
    if wtype == "q4_0":
        for i, k in enumerate(("w_up", "w_gate", "w_down")):
            if L[k] is not None:
                L[k] = torch.from_numpy(q4_blob_random(F, d, 100 + i)).cuda()
    L["wtype"] = wtype
    lay, olay, H = make_pair(L)
    X = synth.integer_tokens(3, d, 9).numpy()
    for t in range(3):
        # down rows on the oracle side are exact too: compare bitwise
        _, logit_ref, M = oracle.predict(olay, X[t])
        idx_ref = oracle.compact(M)
        y_ref = oracle.sparse_ffn(olay, X[t], idx_ref)
        x = _cuda(X[t])
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros(F, dtype=torch.float32, device="cuda")
        ws = B.pi_predict(lay, x, idx, n, logits=logits)
        assert B.pi_sync_status(ws) == 0
        assert np.array_equal(logits.cpu().numpy().astype(np.float64), logit_ref)
        assert int(n.item()) == idx_ref.size
        assert np.array_equal(idx.cpu().numpy()[:idx_ref.size], idx_ref)
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_sparse_ffn(lay, x, idx, n, y, ws=ws)
        assert B.pi_sync_status(ws) == 0
        assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


# ---------------------------------------------------------------- predictor
@pytest.mark.parametrize("ptype", ["f32", "f16"])
@pytest.mark.parametrize("batch", [1, 3, 8])
@pytest.mark.parametrize("shape", SHAPES)
def test_predict_parity(ptype, batch, shape):
    d, F, r = shape
    lay, olay, H = _layer(d, F, r, False, ptype, seed=3 * d + batch)
    X = synth.tokens(batch, d, 11).numpy()
    logit_ref, union_ref = oracle.predict_union(olay, X)
    amb = np.zeros(F, bool)
    for b in range(batch):
        h_b, _, _ = oracle.predict(olay, X[b])
        amb |= ambiguous(logit_ref[b], logit_scale(H, h_b), olay.threshold)
    x = _cuda(X)
    idx = torch.full((F,), -1, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.zeros(batch, F, dtype=torch.float32, device="cuda")
    mask = torch.zeros(F, dtype=torch.uint8, device="cuda")
    ws = B.pi_predict(lay, x, idx, n, logits=logits, mask=mask)
    assert B.pi_sync_status(ws) == 0
    lg = logits.cpu().numpy().astype(np.float64)
    for b in range(batch):
        h_b, _, _ = oracle.predict(olay, X[b])
        tol = 2e-5 * (logit_scale(H, h_b) + 1.0)
        assert np.all(np.abs(lg[b] - logit_ref[b]) <= tol)
    m = mask.cpu().numpy()
    # the GPU mask is its own logits thresholded (union over tokens)
    assert np.array_equal(m.astype(bool), (lg > olay.threshold).any(0))
    # ... and equals the oracle's except where either decision is correct
    assert np.all((m.astype(bool) == union_ref.astype(bool)) | amb)
    got = idx.cpu().numpy()[: int(n.item())]
    assert np.array_equal(got, np.flatnonzero(m))


# ---------------------------------------------------------------- whole layer
@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
@pytest.mark.parametrize("gated", [False, True])
def test_ffn_layer_parity(wtype, gated):
    d, F, r = (512, 2500, 64) if wtype != "q4_0" else (512, 2500, 64)
    lay, olay, H = _layer(d, F, r, gated, wtype, seed=41)
    X = synth.tokens(4, d, 12).numpy()
    ws = None
    for t in range(4):
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        x = _cuda(X[t])
        res = _cuda(synth.tokens(1, d, 50 + t).numpy()[0])
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y, residual=res, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got = set(idx.cpu().numpy()[: int(n.item())].tolist())
        ref = set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)           # disagreement only where either is correct
        idx_res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))),
                           dtype=np.int32)
        y_ref = oracle.sparse_ffn(olay, X[t], idx_res) + res.cpu().numpy().astype(np.float64)
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"layer {wtype} gated={gated} t={t}")


@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
def test_dense_ffn_equals_oracle_dense(wtype):
    d, F, r = 512, 1111, 32
    lay, olay, H = _layer(d, F, r, True, wtype, seed=9)
    X = synth.tokens(2, d, 13).numpy()
    for t in range(2):
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_dense_ffn(lay, _cuda(X[t]), y)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y.cpu().numpy(), oracle.dense_ffn(olay, X[t]), what=f"dense {wtype}")


# ---------------------------------------------------------------- edge cases
def test_edge_empty_single_last_and_inplace_residual():
    d, F, r = 256, 999, 16
    lay, olay, H = _layer(d, F, r, False, "f16", seed=19)
    H_bdown = np.random.default_rng(0).standard_normal(d).astype(np.float32)
    bd = _cuda(H_bdown)
    lay2 = B.Layer(d, F, r, lay.tensors["w_up"], lay.tensors["w_down"], b_act=lay.tensors["b_act"], b_down=bd,
                   p1=lay.tensors["p1"], p2=lay.tensors["p2"], p_bias=lay.tensors["p_bias"])
    olay2 = oracle.Layer(d, F, r, H["w_up"], H["w_down"], b_act=H["b_act"], b_down=H_bdown, p1=H["p1"], p2=H["p2"],
                         p_bias=H["p_bias"])
    x_np = synth.tokens(1, d, 21).numpy()[0]
    x = _cuda(x_np)
    # a neuron that fires, placed at the last position, alone
    z = H["w_up"].astype(np.float64) @ x_np + H["b_act"]
    j_last = F - 1
    cases = [np.zeros(0, np.int32), np.array([j_last], np.int32), np.arange(F, dtype=np.int32),
             np.flatnonzero(z > 0).astype(np.int32)]
    for idx_np in cases:
        y_ref = oracle.sparse_ffn(olay2, x_np, idx_np)
        idx = _cuda(idx_np if idx_np.size else np.zeros(1, np.int32))
        n = torch.tensor([idx_np.size], dtype=torch.int32, device="cuda")
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_sparse_ffn(lay2, x, idx, n, y)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"n={idx_np.size}")
        # residual accumulated in place: y <- y + FFN(x)
        y2 = y.clone()
        B.pi_sparse_ffn(lay2, x, idx, n, y2, residual=y2, ws=ws)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y2.cpu().numpy(), y_ref + y.cpu().numpy().astype(np.float64), what="in place residual")


def test_threshold_above_all_logits_gives_empty_list():
    d, F, r = 256, 700, 16
    lay, olay, H = _layer(d, F, r, False, "f16", seed=23)
    lay_hi = B.Layer(d, F, r, lay.tensors["w_up"], lay.tensors["w_down"], b_act=lay.tensors["b_act"],
                     p1=lay.tensors["p1"], p2=lay.tensors["p2"], p_bias=lay.tensors["p_bias"], threshold=1e30)
    x = _cuda(synth.tokens(1, d, 2).numpy()[0])
    y = torch.full((d,), 5.0, device="cuda")
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = B.pi_ffn_layer(lay_hi, x, y, idx=idx, n_active=n)
    assert B.pi_sync_status(ws) == 0
    assert int(n.item()) == 0
    assert torch.all(y == 0)


def test_out_of_range_index_is_flagged_and_skipped():
    d, F, r = 256, 500, 16
    lay, olay, H = _layer(d, F, r, False, "f16", seed=29)
    x_np = synth.tokens(1, d, 3).numpy()[0]
    good = np.array([1, 5, 9], np.int32)
    idx = _cuda(np.array([1, 5, F + 3, 9], np.int32))
    n = torch.tensor([4], dtype=torch.int32, device="cuda")
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    ws = B.pi_sparse_ffn(lay, _cuda(x_np), idx, n, y)
    assert B.pi_sync_status(ws) == 10    # PI_ERR_INDEX
    assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olay, x_np, good), what="bad index skipped")
    assert B.pi_sync_status(ws) == 0     # cleared


def test_quantizer_matches_oracle_bit_exact():
    rng = np.random.default_rng(31)
    for rows, cols in [(7, 64), (300, 512), (1024, 8192)]:
        w = (rng.standard_normal((rows, cols)) * 10.0 ** rng.integers(-3, 3, (rows, 1))).astype(np.float32)
        w[0, :32] = 0.0                                   # all-zero block
        w[1, :32] = np.linspace(-1, 1, 32)                # ties in magnitude
        for src in (torch.from_numpy(w).cuda(), torch.from_numpy(w).half().cuda()):
            blob = B.pi_quantize_q4_0(src)
            torch.cuda.synchronize()
            ref = oracle.q4_0_quantize(src.float().cpu().numpy())
            assert np.array_equal(blob.cpu().numpy(), ref)


def test_permute_rows_and_rms_residual():
    rng = np.random.default_rng(41)
    F, d = 777, 64
    w = rng.standard_normal((F, d)).astype(np.float16)
    b = rng.standard_normal(F).astype(np.float32)
    perm = rng.permutation(F).astype(np.int32)
    pw = B.pi_permute_rows(_cuda(w), _cuda(perm))
    pb = B.pi_permute_rows(_cuda(b).view(F, 1), _cuda(perm))
    torch.cuda.synchronize()
    assert np.array_equal(pw.cpu().numpy(), w[perm])
    assert np.array_equal(pb.cpu().numpy().ravel(), b[perm])
    x = rng.standard_normal((3, 1024)).astype(np.float32)
    y = rng.standard_normal((3, 1024)).astype(np.float32)
    out = torch.empty(3, 1024, device="cuda")
    B.pi_rms_residual(_cuda(x), _cuda(y), out)
    torch.cuda.synchronize()
    for t in range(3):
        ref = oracle.rms_residual(x[t], y[t].astype(np.float64))
        np.testing.assert_allclose(out[t].cpu().numpy(), ref, rtol=1e-5, atol=1e-6)


def test_fire_counts_and_hot_first_permutation():
    d, F, r = 256, 1000, 16
    lay, olay, H = _layer(d, F, r, False, "f16", seed=43)
    X = synth.tokens(100, d, 44).numpy()
    counts = torch.zeros(F, dtype=torch.int32, device="cuda")
    B.pi_fire_counts(lay, _cuda(X), counts)
    torch.cuda.synchronize()
    got = counts.cpu().numpy()
    ref = oracle.fire_counts(olay, X)
    # a pre-activation within rounding of 0 may be counted either way
    z = X.astype(np.float64) @ H["w_up"].astype(np.float64).T + H["b_act"]
    slack = (np.abs(z) <= 1e-4).sum(0)
    assert np.all(np.abs(got - ref) <= slack)
    assert np.array_equal(B.pi_hot_first_perm(ref), oracle.hot_first_perm(ref))


@pytest.mark.parametrize("shape", [(256, 100, 8), (256, 151, 16), (512, 153, 2048 // 8), (1024, 80000, 64)])
def test_ffn_layer_degenerate_ranges(shape):
    """Layers with fewer neurons or predictor rows than SMs (empty per-CTA
    ranges), and one too wide for the one-kernel path (the three-kernel
    fallback): same parity criteria as test_ffn_layer_parity."""
    d, F, r = shape
    lay, olay, H = _layer(d, F, r, False, "f16", seed=F + r)
    X = synth.tokens(2, d, 14).numpy()
    ws = None
    for t in range(2):
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(lay, _cuda(X[t]), y, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got = set(idx.cpu().numpy()[: int(n.item())].tolist())
        ref = set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)
        idx_res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))),
                           dtype=np.int32)
        assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olay, X[t], idx_res), what=f"{shape} t={t}")


def test_layer_and_predict_share_a_workspace():
    """pi_ffn_layer (one kernel) and pi_predict (separate kernels) called in
    turn on one workspace: neither may read the other's leftovers."""
    d, F, r = 512, 6000, 64
    lay, olay, H = _layer(d, F, r, True, "f16", seed=71)
    X = synth.tokens(4, d, 72).numpy()
    ws = B.workspace(B.pi_workspace_bytes(lay, 1))
    for t in range(4):
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        ref = set(np.flatnonzero(M).tolist())
        x = _cuda(X[t])
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y, ws=ws)
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.pi_predict(lay, x, idx, n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got = set(idx.cpu().numpy()[: int(n.item())].tolist())
        assert all(amb[j] for j in got ^ ref)


def test_next_layer_hint_changes_nothing():
    """Naming the next layer is a scheduling hint the kernels do not use:
    outputs and active lists stay those of the oracle with another, a
    self-referencing or no next layer."""
    d, F, r = 512, 3000, 64
    lay, olay, H = _layer(d, F, r, True, "f16", seed=97)
    lay2, _, _ = _layer(d, F, r, False, "f16", seed=98)
    X = synth.tokens(3, d, 99).numpy()
    for nxt in (lay2, lay, None):
        lay.set_next(nxt)
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = None
        for t in range(X.shape[0]):
            ws = B.pi_ffn_layer(lay, _cuda(X[t]), y, idx=idx, n_active=n, ws=ws)
            assert B.pi_sync_status(ws) == 0
            h, logit_ref, M = oracle.predict(olay, X[t])
            amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
            got, ref = set(idx.cpu().numpy()[: int(n.item())].tolist()), set(np.flatnonzero(M).tolist())
            assert all(amb[j] for j in got ^ ref)
            res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), np.int32)
            assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olay, X[t], res), what=f"next={nxt is not None} t={t}")
    lay.set_next(None)


@pytest.mark.parametrize("d", [8, 1030, 12288, 16384, 20000])
def test_rms_residual_both_paths_and_in_place(d):
    """16-byte aligned rows with d % 4 == 0 and d <= 16384 take the one-pass
    vector kernel, the rest the strided one; out may alias x."""
    rng = np.random.default_rng(d)
    x = rng.standard_normal((3, d)).astype(np.float32)
    y = rng.standard_normal((3, d)).astype(np.float32)
    xd = _cuda(x)
    B.pi_rms_residual(xd, _cuda(y), xd)          # in place
    torch.cuda.synchronize()
    for t in range(3):
        np.testing.assert_allclose(xd[t].cpu().numpy(), oracle.rms_residual(x[t], y[t].astype(np.float64)),
                                   rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("ptype,rank", [("f16", 2048), ("f32", 768)])
def test_wide_rank_layer(ptype, rank):
    """Predictor ranks wider than the per-lane register slices of h (fp16 above
    1024, fp32 above 512): the one-kernel layer reads the rest of h from
    shared memory.  Ordered and queue mode against the oracle."""
    d, F = 1024, 4100
    lay, olay, H = _layer(d, F, rank, True, ptype, seed=171 + rank, sparsity=0.85)
    X = synth.tokens(2, d, 172).numpy()
    ws = None
    for t in range(X.shape[0]):
        x = _cuda(X[t])
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        y1 = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y1, idx=idx, n_active=n, ws=ws)
        y2 = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y2, ws=ws)
        assert B.pi_sync_status(ws) == 0
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        got, ref = set(idx.cpu().numpy()[: int(n.item())].tolist()), set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)
        res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), np.int32)
        y_ref = oracle.sparse_ffn(olay, X[t], res)
        assert_ffn_close(y1.cpu().numpy(), y_ref, what=f"ordered {ptype} r={rank} t={t}")
        assert_ffn_close(y2.cpu().numpy(), y_ref, what=f"queue {ptype} r={rank} t={t}")


@pytest.mark.parametrize("wtype,gated,sparsity", [("f32", False, 0.8), ("f32", True, 0.8), ("f16", False, 0.8),
                                                  ("f16", True, 0.8), ("q4_0", False, 0.8), ("q4_0", True, 0.8),
                                                  ("f16", True, 0.4), ("f16", False, 0.995)])
def test_queue_mode_matches_ordered_mode(wtype, gated, sparsity):
    """Without idx / n_active, the one-kernel layer keeps the first active
    neurons of each CTA's range and takes the rest from a shared work queue
    instead of an ordered list.  The predicted set is the same (the logits path
    is deterministic), so its output must match the oracle on the ordered run's
    resolved list.  Densities span ranges with fewer active neurons than a CTA
    keeps (a nearly empty queue) and far more.  Modes alternate on one
    workspace."""
    d, F, r = 1024, 4100, 128
    lay, olay, H = _layer(d, F, r, gated, wtype, seed=131 + gated, sparsity=sparsity)
    X = synth.tokens(4, d, 132).numpy()
    ws = None
    for t in range(X.shape[0]):
        x = _cuda(X[t])
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        y1 = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y1, idx=idx, n_active=n, ws=ws)
        y2 = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y2, ws=ws)                       # queue mode
        B.pi_ffn_layer(lay, x, y2, ws=ws)                       # twice: the counters alternate
        assert B.pi_sync_status(ws) == 0
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        got, ref = set(idx.cpu().numpy()[: int(n.item())].tolist()), set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)
        res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), np.int32)
        y_ref = oracle.sparse_ffn(olay, X[t], res)
        assert_ffn_close(y1.cpu().numpy(), y_ref, what=f"ordered {wtype} gated={gated} t={t}")
        assert_ffn_close(y2.cpu().numpy(), y_ref, what=f"queue {wtype} gated={gated} t={t}")


def _sm_count():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


@pytest.mark.parametrize("which,gated,density", [("queue_max", False, 1.0), ("queue_max", True, 0.85),
                                                 ("queue_mid", False, 1.0), ("ordered_only", False, 1.0),
                                                 ("ordered_only", True, 0.9)])
def test_near_dense_wide_layer_runs_every_neuron(which, gated, density):
    """Near-dense tokens on the widest layers the one-kernel step accepts, where
    one CTA must run about 500 rows.  Without a list asked for, the rows go
    through the shared work queue up to 509 rows per SM (every CTA's share table
    then holds all of them); above that the step uses the ordered list.  Every
    predicted neuron must be run in both cases, and the ordered list must be
    exact.  The mask is fixed by the predictor's output bias (+-1e4 against
    logits of order 1), so it is known without any rounding question."""
    G = _sm_count()
    F = {"queue_max": 509 * G, "queue_mid": 470 * G + 13, "ordered_only": 512 * G - 21}[which]
    d, r = 256, 64
    L = synth.make_layer(d, F, r, gated=gated, wtype="f16", sparsity=0.5, predictor="random", seed=F + gated,
                         device="cuda")
    on = np.random.default_rng(F + 1).random(F) < density
    L["p_bias"] = torch.from_numpy(np.where(on, 1e4, -1e4).astype(np.float32)).cuda()
    lay, olay, H = make_pair(L)
    X = synth.tokens(2, d, 91).numpy()
    ws = None
    for t in range(2):
        _, _, M = oracle.predict(olay, X[t])
        assert np.array_equal(M.astype(bool), on)
        ref_idx = oracle.compact(M)
        y_ref = oracle.sparse_ffn(olay, X[t], ref_idx)
        x = _cuda(X[t])
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        y1 = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y1, idx=idx, n_active=n, ws=ws)
        y2 = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y2, ws=ws)
        y3 = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y3, ws=ws)                      # the queue counters alternate by launch
        assert B.pi_sync_status(ws) == 0
        assert int(n.item()) == ref_idx.size
        assert np.array_equal(idx.cpu().numpy()[: ref_idx.size], ref_idx)
        for y, mode in ((y1, "ordered"), (y2, "no list"), (y3, "no list, again")):
            assert_ffn_close(y.cpu().numpy(), y_ref, what=f"{which} F={F} gated={gated} {mode} t={t}")
