"""The always-on prefix (neurons [0, dense_prefix) computed at every step, the
predictor deciding only the tail): every path against the oracle's mask
(prefix | logit > threshold) and sparse FFN -- the one-kernel step in both of
its modes, the predictor + scan + sparse chain, the batched union path and
pi_predict alone.  Prefixes from none to the whole layer."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu


def _pair(d, F, r, gated, wtype, seed, prefix, ptype=None, sparsity=0.85):
    L = synth.make_layer(d, F, r, gated=gated, wtype="f32" if wtype == "f32" else "f16", sparsity=sparsity,
                         seed=seed, device="cuda")
    L["wtype"] = wtype
    if ptype == "f16":
        L["p1"], L["p2"] = L["p1"].half(), L["p2"].half()
    lay, olay, H = make_pair(L)
    lay.desc.dense_prefix = prefix
    olay_p = oracle.Layer(d, F, r, H["w_up"], H["w_down"], w_gate=H["w_gate"], b_act=H["b_act"],
                          b_down=H["b_down"], p1=H["p1"], p2=H["p2"], p_bias=H["p_bias"],
                          threshold=H["threshold"], dense_prefix=prefix)
    return lay, olay_p, H


def _resolve(olay, H, X, got):
    """Oracle union mask of the tokens X; decisions at borderline logits of the
    tail are taken from the GPU's list `got` (either side is correct there)."""
    union = np.zeros(olay.d_ff, bool)
    amb = np.zeros(olay.d_ff, bool)
    for x in X:
        h, logit, m = oracle.predict(olay, x)
        union |= m.astype(bool)
        a = ambiguous(logit, logit_scale(H, h), olay.threshold)
        a[: olay.dense_prefix] = False      # the prefix is decided exactly
        amb |= a
    ref = set(np.flatnonzero(union).tolist())
    assert all(amb[j] for j in got ^ ref), "decisions differ away from the threshold"
    assert set(range(olay.dense_prefix)) <= got
    return np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), np.int32)


@pytest.mark.parametrize("prefix", [0, 7, 1000, 4100])
@pytest.mark.parametrize("wtype,ptype,gated", [("f16", None, True), ("f16", None, False), ("q4_0", None, False),
                                              ("f32", "f16", False)])
def test_prefix_batch1_both_modes(prefix, wtype, ptype, gated):
    d, F, r = (1024 if wtype != "q4_0" else 1024), 4100, 128
    lay, olay, H = _pair(d, F, r, gated, wtype, seed=301 + prefix, prefix=prefix, ptype=ptype)
    X = synth.tokens(3, d, 302).numpy()
    ws = None
    for t in range(3):
        x = torch.from_numpy(X[t]).cuda()
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        y1 = torch.empty(d, dtype=torch.float32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y1, idx=idx, n_active=n, ws=ws)
        y2 = torch.empty(d, dtype=torch.float32, device="cuda")
        B.pi_ffn_layer(lay, x, y2, ws=ws)                          # no list asked for
        assert B.pi_sync_status(ws) == 0
        lst = idx.cpu().numpy()[: int(n.item())]
        assert np.all(np.diff(lst) > 0)
        res = _resolve(olay, H, X[t:t + 1], set(lst.tolist()))
        y_ref = oracle.sparse_ffn(olay, X[t], res)
        assert_ffn_close(y1.cpu().numpy(), y_ref, what=f"list prefix={prefix} {wtype} t={t}")
        assert_ffn_close(y2.cpu().numpy(), y_ref, what=f"no list prefix={prefix} {wtype} t={t}")


@pytest.mark.parametrize("prefix", [0, 300, 4100])
@pytest.mark.parametrize("batch", [3, 8])
def test_prefix_union_path(prefix, batch):
    d, F, r = 1024, 4100, 128
    lay, olay, H = _pair(d, F, r, False, "f16", seed=311, prefix=prefix)
    X = synth.tokens(batch, d, 312).numpy()
    x = torch.from_numpy(X).cuda()
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    ws = B.pi_ffn_layer(lay, x, y, idx=idx, n_active=n)
    assert B.pi_sync_status(ws) == 0
    res = _resolve(olay, H, X, set(idx.cpu().numpy()[: int(n.item())].tolist()))
    for b in range(batch):
        assert_ffn_close(y[b].cpu().numpy(), oracle.sparse_ffn(olay, X[b], res), what=f"union b={b}")


@pytest.mark.parametrize("batch", [1, 4])
def test_prefix_in_pi_predict_mask(batch):
    d, F, r = 512, 3000, 64
    prefix = 500
    lay, olay, H = _pair(d, F, r, False, "f16", seed=321, prefix=prefix)
    X = synth.tokens(batch, d, 322).numpy()
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.zeros(F, dtype=torch.uint8, device="cuda")
    ws = B.pi_predict(lay, torch.from_numpy(X if batch > 1 else X[0]).cuda(), idx, n, mask=mask)
    assert B.pi_sync_status(ws) == 0
    m = mask.cpu().numpy().astype(bool)
    assert m[:prefix].all()
    got = set(idx.cpu().numpy()[: int(n.item())].tolist())
    assert got == set(np.flatnonzero(m).tolist())
    _resolve(olay, H, X, got)


def test_prefix_of_profiled_hot_neurons_raises_recall():
    """Hot-first order from a profiling pass, prefix = the neurons that fired
    on more than half of the profiling tokens: the predicted set then contains
    every such neuron, and recall against the true activity does not drop."""
    d, F, r = 1024, 8192, 128
    L = synth.make_layer(d, F, r, gated=False, wtype="f16", sparsity=0.9, seed=331, device="cuda")
    lay, olay, H = make_pair(L)
    Xp = synth.tokens(256, d, 332).numpy()
    counts = oracle.fire_counts(olay, Xp)
    perm = oracle.hot_first_perm(counts)
    hot = int(np.sum(counts > Xp.shape[0] // 2))
    assert hot > 0
    Hp = dict(H)
    for k in ("w_up", "w_down", "p2", "b_act", "p_bias"):
        Hp[k] = np.ascontiguousarray(H[k][perm])
    dev = {k: torch.from_numpy(Hp[k]).cuda() for k in ("w_up", "w_down", "p2", "b_act", "p_bias")}
    rec = {}
    for prefix in (0, hot):
        layp = B.Layer(d, F, r, dev["w_up"], dev["w_down"], b_act=dev["b_act"], b_down=torch.from_numpy(Hp["b_down"]).cuda(),
                       p1=torch.from_numpy(Hp["p1"]).cuda(), p2=dev["p2"], p_bias=dev["p_bias"],
                       threshold=Hp["threshold"], dense_prefix=prefix)
        olayp = oracle.Layer(d, F, r, Hp["w_up"], Hp["w_down"], b_act=Hp["b_act"], b_down=Hp["b_down"],
                             p1=Hp["p1"], p2=Hp["p2"], p_bias=Hp["p_bias"], threshold=Hp["threshold"],
                             dense_prefix=prefix)
        X = synth.tokens(8, d, 333).numpy()
        recs = []
        ws = None
        for t in range(X.shape[0]):
            idx = torch.zeros(F, dtype=torch.int32, device="cuda")
            n = torch.zeros(1, dtype=torch.int32, device="cuda")
            y = torch.empty(d, dtype=torch.float32, device="cuda")
            ws = B.pi_ffn_layer(layp, torch.from_numpy(X[t]).cuda(), y, idx=idx, n_active=n, ws=ws)
            assert B.pi_sync_status(ws) == 0
            got = set(idx.cpu().numpy()[: int(n.item())].tolist())
            res = _resolve(olayp, Hp, X[t:t + 1], got)
            assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olayp, X[t], res), what=f"prefix={prefix} t={t}")
            T, _ = oracle.true_mask(olayp, X[t])
            recs.append(oracle.recall_precision(np.isin(np.arange(F), res), T)[0])
        rec[prefix] = float(np.mean(recs))
    assert rec[hot] >= rec[0]
