"""Neuron-sharded layer on CPU ranks (gloo, world size 2): each rank takes its
shard of the hot-first order from the library's host dealer, computes its
partial output with the oracle on its own rows, and one all-reduce (sum) of the
batch x d_model partials yields the layer output.  The exchange and the host
logic are what is tested here; the GPU runs of shard layers are in
test_gpu_shard.py."""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

D, F, R, BATCH = 128, 1000, 32, 3


def _layer():
    import oracle
    from activation_sparse_decode_predictor_gb300 import synth
    L = synth.make_layer(D, F, R, gated=True, wtype="f16", sparsity=0.8, predictor="random", seed=5)
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    return oracle.Layer(D, F, R, w["w_up"], w["w_down"], w_gate=w["w_gate"], b_act=w["b_act"],
                        b_down=w["b_down"] + 0.5, p1=w["p1"], p2=w["p2"], p_bias=w["p_bias"], threshold=0.0)


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import oracle
    from activation_sparse_decode_predictor_gb300 import binding as B
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lay = _layer()
        X = np.random.default_rng(11).standard_normal((BATCH, D)).astype(np.float32)
        Xp = np.random.default_rng(12).standard_normal((64, D)).astype(np.float32)
        order = B.pi_hot_first_perm(oracle.fire_counts(lay, Xp))
        S = B.pi_shard_neurons(order, world, rank)
        sh = oracle.neuron_shard(lay, S, keep_b_down=(rank == 0))
        part = np.zeros((BATCH, D), dtype=np.float64)
        active = torch.zeros(F, dtype=torch.int32)
        for b in range(BATCH):
            _, _, m = oracle.predict(sh, X[b])
            idx = oracle.compact(m)
            part[b] = oracle.sparse_ffn(sh, X[b], idx)
            active[torch.from_numpy(S[idx].astype(np.int64))] += 1
        y = torch.from_numpy(part)
        dist.all_reduce(y)               # the one exchange step of a sharded layer
        dist.all_reduce(active)
        ref = np.stack([oracle.sparse_ffn(lay, X[b], oracle.compact(oracle.predict(lay, X[b])[2]))
                        for b in range(BATCH)])
        ref_active = sum(oracle.predict(lay, X[b])[2].astype(np.int32) for b in range(BATCH))
        out[rank] = (float(np.max(np.abs(y.numpy() - ref))), float(np.max(np.abs(ref))), S.size,
                     bool(np.array_equal(active.numpy(), ref_active)))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharded_layer_equals_the_layer():
    from activation_sparse_decode_predictor_gb300 import build
    build.build()
    world = 2
    port = 29700 + (os.getpid() % 1000)
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    assert res[0][2] + res[1][2] == F and abs(res[0][2] - res[1][2]) <= 1
    for r in range(world):
        err, scale, _, same_active = res[r]
        assert scale > 0 and err <= 1e-12 * scale
        assert same_active
