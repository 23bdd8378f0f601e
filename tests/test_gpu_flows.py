"""End-to-end flows through the C ABI against the oracle:

* hot-first order: firing counts over profiling tokens -> stable descending
  order -> rows of every per-neuron array permuted -> the layer run on the
  permuted weights (the OPT-30B workload's offline step, at a reduced shape);
* a stack of 12 layers, each output plus residual rescaled into the next
  layer's input (the OPT-175B workload's glue, at a reduced shape), at batch 1
  and through the batched union path.

Oracle chains start from the same inputs and never consume a GPU result."""
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


def _predicted_union(olay, H, X):
    """Oracle union mask of a group of tokens and the neurons whose decision is
    borderline for at least one token."""
    union = np.zeros(olay.d_ff, dtype=bool)
    amb = np.zeros(olay.d_ff, dtype=bool)
    for x in X:
        h, logit, m = oracle.predict(olay, x)
        union |= m.astype(bool)
        amb |= ambiguous(logit, logit_scale(H, h), olay.threshold)
    return union, amb


def test_hot_first_permuted_layer():
    d, F, r = 512, 3000, 64
    L = synth.make_layer(d, F, r, gated=False, wtype="f16", sparsity=0.95, seed=71, device="cuda")
    lay, olay, H = make_pair(L)
    Xp = synth.tokens(512, d, 72).numpy()                  # profiling pass
    counts_ref = oracle.fire_counts(olay, Xp)
    perm = oracle.hot_first_perm(counts_ref)
    assert np.all(np.diff(counts_ref[perm]) <= 0)          # hot neurons first
    counts = torch.zeros(F, dtype=torch.int32, device="cuda")
    B.pi_fire_counts(lay, _cuda(Xp), counts)
    torch.cuda.synchronize()
    z = Xp.astype(np.float64) @ H["w_up"].astype(np.float64).T + H["b_act"]
    assert np.all(np.abs(counts.cpu().numpy() - counts_ref) <= (np.abs(z) <= 1e-4).sum(0))
    assert np.array_equal(B.pi_hot_first_perm(counts_ref), perm)

    # permute every per-neuron array on the device; the oracle permutes its own copies
    dev_perm = _cuda(perm)
    Lp = dict(L)
    for k in ("w_up", "w_down", "p2"):
        Lp[k] = B.pi_permute_rows(L[k], dev_perm)
    for k in ("b_act", "p_bias"):
        Lp[k] = B.pi_permute_rows(L[k].view(F, 1), dev_perm).view(F)
    torch.cuda.synchronize()
    Hp = dict(H)
    for k in ("w_up", "w_down", "p2", "b_act", "p_bias"):
        Hp[k] = np.ascontiguousarray(H[k][perm])
        assert np.array_equal(Lp[k].cpu().numpy(), Hp[k])
    layp = B.Layer.from_dict(Lp)
    olayp = oracle.Layer(d, F, r, Hp["w_up"], Hp["w_down"], b_act=Hp["b_act"], b_down=Hp["b_down"], p1=Hp["p1"],
                         p2=Hp["p2"], p_bias=Hp["p_bias"], threshold=Hp["threshold"])

    X = synth.tokens(6, d, 73).numpy()
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    ws = None
    low = []
    for t in range(X.shape[0]):
        ws = B.pi_ffn_layer(layp, _cuda(X[t]), y, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got = set(idx.cpu().numpy()[: int(n.item())].tolist())
        ref_mask, amb = _predicted_union(olayp, Hp, X[t:t + 1])
        ref = set(np.flatnonzero(ref_mask).tolist())
        assert all(amb[j] for j in got ^ ref)
        res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), dtype=np.int32)
        y_ref = oracle.sparse_ffn(olayp, X[t], res)
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"permuted layer t={t}")
        # the permutation changes neither the set of neurons nor the output
        assert_ffn_close(y_ref, oracle.sparse_ffn(olay, X[t], np.sort(perm[res])), what=f"permutation invariance t={t}")
        low.append(np.mean(np.array(sorted(got)) < F // 4) if got else 1.0)
    # hot-first: most active neurons now sit in the first quarter of the rows
    assert np.mean(low) > 0.5


@pytest.mark.parametrize("batch", [1, 4])
def test_stack_of_twelve_layers(batch):
    d, F, r, depth = 512, 2048, 64, 12
    layers = []
    for l in range(depth):
        L = synth.make_layer(d, F, r, gated=False, wtype="f16", sparsity=0.95, seed=900 + l, device="cuda")
        layers.append(make_pair(L))
    X0 = synth.tokens(batch, d, 901).numpy()

    # GPU chain: pi_ffn_layer then pi_rms_residual, all on the device
    xg = _cuda(X0)
    y = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    xn = torch.empty(batch, d, dtype=torch.float32, device="cuda")
    idx = torch.zeros(F, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    gpu_x, gpu_sets = [], []
    for lay, _, _ in layers:
        ws = B.pi_ffn_layer(lay, xg if batch > 1 else xg[0], y if batch > 1 else y[0], idx=idx, n_active=n, ws=ws)
        B.pi_rms_residual(xg, y, xn)
        assert B.pi_sync_status(ws) == 0
        gpu_sets.append(set(idx.cpu().numpy()[: int(n.item())].tolist()))
        xg, xn = xn, xg
        gpu_x.append(xg.cpu().numpy().copy())

    # oracle chain from the same input
    xo = X0.astype(np.float32)
    for l, (_, olay, H) in enumerate(layers):
        union, amb = _predicted_union(olay, H, xo)
        ref = set(np.flatnonzero(union).tolist())
        diff = gpu_sets[l] ^ ref
        assert all(amb[j] for j in diff), f"layer {l}: decisions differ away from the threshold"
        if diff:
            # a borderline neuron went the other way: both chains are valid from here on
            break
        idx_np = np.flatnonzero(union).astype(np.int32)
        xnext = np.empty((batch, d), dtype=np.float64)
        for b in range(batch):
            xnext[b] = oracle.rms_residual(xo[b], oracle.sparse_ffn(olay, xo[b], idx_np))
        for b in range(batch):
            assert_ffn_close(gpu_x[l][b], xnext[b], what=f"layer {l} token {b}")
        xo = xnext.astype(np.float32)
    else:
        return
    pytest.skip(f"chain compared through layer {l - 1}; a borderline decision at layer {l} split the chains")
