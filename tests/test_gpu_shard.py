"""Neuron-sharded layers on the GPU against the oracle: a layer's neurons are
dealt round-robin from the hot-first order (pi_shard_neurons), each shard's
rows gathered on the device (pi_gather_rows through Layer.shard), every shard
run through pi_ffn_layer with b_down and the residual on shard 0 only, and the
partial outputs summed (the all-reduce of a sharded deployment, done here on
one device).  The sum must equal the oracle's unsharded layer on the union of
the shards' active lists, mapped back to the layer's neuron ids."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("shards", [2, 3])
@pytest.mark.parametrize("gated,wtype", [(True, "f16"), (False, "f16"), (False, "q4_0")])
def test_sharded_layer_sums_to_the_layer(gated, wtype, shards, batch):
    d, F, r = 1024, 4100, 128
    L = synth.make_layer(d, F, r, gated=gated, wtype="f16", sparsity=0.9, seed=300 + shards, device="cuda")
    L["wtype"] = wtype
    L["b_down"] = torch.full((d,), 0.25, dtype=torch.float32, device="cuda")   # added by one shard only
    lay, olay, H = make_pair(L)
    Xp = synth.tokens(128, d, 301).numpy()
    order = oracle.hot_first_perm(oracle.fire_counts(olay, Xp))
    X = synth.tokens(batch, d, 302 + batch).numpy()
    Rs = synth.tokens(batch, d, 303).numpy()
    x = _cuda(X)
    y = torch.zeros(batch, d, dtype=torch.float32, device="cuda")
    got = set()
    for g in range(shards):
        S = B.pi_shard_neurons(order, shards, g)
        assert np.array_equal(S, order[g::shards])
        sh = lay.shard(_cuda(S), keep_b_down=(g == 0))
        osh = oracle.neuron_shard(olay, S, keep_b_down=(g == 0))
        torch.cuda.synchronize()
        for k in ("w_up", "w_gate", "w_down", "b_act", "p2", "p_bias"):
            if sh.tensors[k] is not None:
                ref = getattr(osh, k)
                assert np.array_equal(sh.tensors[k].cpu().numpy().view(ref.dtype).reshape(ref.shape), ref), k
        yg = torch.empty(batch, d, dtype=torch.float32, device="cuda")
        idx = torch.zeros(S.size, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        res = _cuda(Rs) if g == 0 else None
        if batch == 1:
            ws = B.pi_ffn_layer(sh, x[0], yg[0], residual=None if res is None else res[0], idx=idx, n_active=n)
        else:
            ws = B.pi_ffn_layer(sh, x, yg, residual=res, idx=idx, n_active=n)
        assert B.pi_sync_status(ws) == 0
        got |= set(S[idx.cpu().numpy()[: int(n.item())]].tolist())
        y += yg
    torch.cuda.synchronize()

    ref, amb = set(), np.zeros(F, dtype=bool)
    for b in range(batch):
        h, logit, m = oracle.predict(olay, X[b])
        ref |= set(np.flatnonzero(m).tolist())
        amb |= ambiguous(logit, logit_scale(H, h), olay.threshold)
    assert all(amb[j] for j in got ^ ref)
    idx_res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), dtype=np.int32)
    for b in range(batch):
        y_ref = oracle.sparse_ffn(olay, X[b], idx_res) + Rs[b]
        assert_ffn_close(y.cpu().numpy()[b], y_ref, what=f"{wtype} gated={gated} shards={shards} B={batch} b={b}")
