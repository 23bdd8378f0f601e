"""GPU parity at the workloads' full sizes (one layer, a few tokens each):
the ReLU-LLaMA-7B gated fp16 layer, the OPT-30B fp16 layer, the Falcon-40B
layer in fp16 and Q4_0, and one OPT-175B layer.  These shapes make every
shared-memory ring of the kernels wrap around several times.  Outputs are
compared in full (the oracle's sparse path costs well under a second per
token here); active lists are compared where the oracle and the GPU must
agree, i.e. away from borderline logits."""
import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu

NAMES = ["llama7b-reglu-fp16", "opt30b-relu-fp16-perm", "falcon40b-relu-fp16", "falcon40b-relu-q4_0",
         "opt175b-relu-fp16-stack12"]


@pytest.mark.parametrize("name", NAMES)
def test_workload_layer_parity(name):
    w = synth.WORKLOADS[name]
    L = synth.workload_layer(w, 0, device="cuda")
    lay, olay, H = make_pair(L)
    X = synth.workload_tokens(w, n=2, device="cpu").numpy()
    F, d = w.d_ff, w.d_model
    ws = None
    for t in range(2):
        h, logit_ref, M = oracle.predict(olay, X[t])
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        x = torch.from_numpy(X[t]).cuda()
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, y, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got_list = idx.cpu().numpy()[: int(n.item())]
        assert np.all(np.diff(got_list) > 0)
        got, ref = set(got_list.tolist()), set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)
        idx_res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))),
                           dtype=np.int32)
        assert_ffn_close(y.cpu().numpy(), oracle.sparse_ffn(olay, X[t], idx_res), what=f"{name} layer t={t}")
        # the sparse operator alone on the oracle's own list, and the predictor's list
        y2 = torch.empty(d, dtype=torch.float32, device="cuda")
        idx_o = torch.from_numpy(np.flatnonzero(M).astype(np.int32)).cuda()
        n_o = torch.tensor([idx_o.numel()], dtype=torch.int32, device="cuda")
        B.pi_sparse_ffn(lay, x, idx_o, n_o, y2, ws=ws)
        assert B.pi_sync_status(ws) == 0
        assert_ffn_close(y2.cpu().numpy(), oracle.sparse_ffn(olay, X[t], np.flatnonzero(M).astype(np.int32)),
                         what=f"{name} sparse t={t}")
        idx3 = torch.zeros(F, dtype=torch.int32, device="cuda")
        n3 = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.pi_predict(lay, x, idx3, n3, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got3 = set(idx3.cpu().numpy()[: int(n3.item())].tolist())
        assert all(amb[j] for j in got3 ^ ref)      # each path may resolve borderline logits its own way


def test_opt30b_hot_first_permuted_layer_full_size():
    """The OPT-30B-shaped layer in hot-first order at full size: firing counts
    of a profiling pass (its own token stream; 32 tokens here, so the oracle's
    count finishes in seconds) by the oracle and by pi_fire_counts, the oracle's
    stable hot-first order applied to every per-neuron array on the device by
    pi_permute_rows and on the host by indexing, then the permuted layer
    against the oracle on the permuted host arrays."""
    w = synth.WORKLOADS["opt30b-relu-fp16-perm"]
    F, d = w.d_ff, w.d_model
    L = synth.workload_layer(w, 0, device="cuda")
    lay, olay, H = make_pair(L)
    Xp = synth.workload_tokens(w, n=32, device="cpu", stream=1).numpy()
    counts_ref = oracle.fire_counts(olay, Xp)
    counts = torch.zeros(F, dtype=torch.int32, device="cuda")
    B.pi_fire_counts(lay, torch.from_numpy(Xp).cuda(), counts)
    torch.cuda.synchronize()
    z = Xp.astype(np.float64) @ H["w_up"].astype(np.float64).T + H["b_act"]
    assert np.all(np.abs(counts.cpu().numpy() - counts_ref) <= (np.abs(z) <= 1e-4).sum(0))
    perm = oracle.hot_first_perm(counts_ref)
    dev_perm = torch.from_numpy(perm).cuda()
    Lp = dict(L)
    for k in ("w_up", "w_down", "p2"):
        Lp[k] = B.pi_permute_rows(L[k], dev_perm)
    for k in ("b_act", "p_bias"):
        Lp[k] = B.pi_permute_rows(L[k].view(F, 1), dev_perm).view(F)
    torch.cuda.synchronize()
    Hp = dict(H)
    for k in ("w_up", "w_down", "p2", "b_act", "p_bias"):
        Hp[k] = np.ascontiguousarray(H[k][perm])
    assert np.array_equal(Lp["w_up"][:64].cpu().numpy(), Hp["w_up"][:64])
    layp = B.Layer.from_dict(Lp)
    olayp = oracle.Layer(d, F, w.rank, Hp["w_up"], Hp["w_down"], b_act=Hp["b_act"], b_down=Hp["b_down"],
                         p1=Hp["p1"], p2=Hp["p2"], p_bias=Hp["p_bias"], threshold=Hp["threshold"])
    X = synth.workload_tokens(w, n=2, device="cpu").numpy()
    ws = None
    for t in range(2):
        h, logit_ref, M = oracle.predict(olayp, X[t])
        amb = ambiguous(logit_ref, logit_scale(Hp, h), olayp.threshold)
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(layp, torch.from_numpy(X[t]).cuda(), y, idx=idx, n_active=n, ws=ws)
        assert B.pi_sync_status(ws) == 0
        got, ref = set(idx.cpu().numpy()[: int(n.item())].tolist()), set(np.flatnonzero(M).tolist())
        assert all(amb[j] for j in got ^ ref)
        res = np.array(sorted((ref - set(np.flatnonzero(amb))) | (got & set(np.flatnonzero(amb)))), np.int32)
        y_ref = oracle.sparse_ffn(olayp, X[t], res)
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"permuted OPT-30B t={t}")
        # same neurons and output as the layer in its original order
        assert_ffn_close(y_ref, oracle.sparse_ffn(olay, X[t], np.sort(perm[res])), what=f"invariance t={t}")
        # hot-first: most predicted neurons sit in the first quarter of the rows
        assert np.mean(np.array(sorted(got)) < F // 4) > 0.5
