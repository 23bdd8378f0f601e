"""The allocation-free layer step, pi_ffn_layer_static.

Some callers cannot allocate device memory: code in a host callback or an
allocator hook, plugins whose host application forbids cudaMalloc, threads
that must not risk the device-wide synchronisation cudaMalloc / cudaFree can
cause.  For them the library runs the batch-1 layer step on scratch space of
its own, a fixed device array shared by every call.  These tests call it
through the C ABI and check every call against the oracle, and its active list
bit for bit against the regular workspace path's.  Consecutive calls alternate
between layers of different shapes and between the one-kernel step and the
predictor + scan + sparse FFN chain (fp32 weights with an fp16 predictor), so
each call runs on scratch that a call of another shape left behind.  This file
is collected last: a failure here stops a run only after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import build, synth

from helpers import ambiguous, assert_ffn_close, logit_scale, make_pair

pytestmark = pytest.mark.gpu


def _layer(d, F, r, gated, wtype, seed, ptype=None, sparsity=0.9, dense=False):
    L = synth.make_layer(d, F, r, gated=gated, wtype="f32" if wtype == "f32" else "f16", sparsity=sparsity,
                         predictor="random" if dense else "projection", seed=seed, device="cuda")
    L["wtype"] = wtype
    if ptype == "f16":
        L["p1"], L["p2"] = L["p1"].half(), L["p2"].half()
    if dense:  # every neuron predicted active, without a borderline logit
        L["p_bias"] = torch.full((F,), 1e4, dtype=torch.float32, device="cuda")
    return make_pair(L)


def _static(lay, x, res, y, idx, n, status):
    stream = torch.cuda.current_stream()
    vp = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    return B.lib().pi_ffn_layer_static(ctypes.byref(lay.desc), vp(x), vp(res), vp(y), vp(idx), vp(n), vp(status),
                                       ctypes.c_void_p(stream.cuda_stream))


def test_static_scratch_matches_oracle_across_shapes():
    build.build()
    cases = {
        "fused": _layer(1024, 4096, 256, True, "f16", seed=61),
        "chain": _layer(512, 3000, 64, False, "f32", seed=62, ptype="f16"),   # no one-kernel step for this pair
        "dense": _layer(256, 65536, 64, False, "f16", seed=63, dense=True),   # the largest d_ff accepted
    }
    order = ["fused", "fused", "chain", "fused", "chain", "chain", "dense", "dense", "fused"]
    for call, name in enumerate(order):
        lay, olay, H = cases[name]
        d, F = olay.d_model, olay.d_ff
        x_np = synth.tokens(1, d, 70 + call).numpy()[0]
        r_np = synth.tokens(1, d, 90 + call).numpy()[0]
        x, res = torch.from_numpy(x_np).cuda(), torch.from_numpy(r_np).cuda()

        # the regular workspace path on the same inputs: the list must be the same bit for bit
        idx_ref = torch.zeros(F, dtype=torch.int32, device="cuda")
        n_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(lay, x, torch.empty(d, device="cuda"), residual=res, idx=idx_ref, n_active=n_ref)
        assert B.pi_sync_status(ws) == 0

        y = torch.empty(d, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert _static(lay, x, res, y, idx, n, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0, (call, name)
        k = int(n.item())
        assert k == int(n_ref.item()), (call, name)
        got = idx[:k].cpu().numpy()
        assert np.array_equal(got, idx_ref[:k].cpu().numpy()), (call, name)

        # the list against the oracle's prediction (either side of a borderline logit is correct)
        h, logit_ref, M = oracle.predict(olay, x_np)
        amb = ambiguous(logit_ref, logit_scale(H, h), olay.threshold)
        assert all(amb[j] for j in set(got.tolist()) ^ set(np.flatnonzero(M).tolist())), (call, name)
        y_ref = oracle.sparse_ffn(olay, x_np, got) + r_np.astype(np.float64)
        assert_ffn_close(y.cpu().numpy(), y_ref, what=f"static call {call} ({name})")

        if name == "dense":  # the same layer with no list asked for: work-queue distribution of the rows
            y2 = torch.empty(d, device="cuda")
            assert _static(lay, x, res, y2, None, None, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert_ffn_close(y2.cpu().numpy(), y_ref, what=f"static call {call} ({name}, no list)")


def test_static_rejects_oversized_layer():
    build.build()
    L = B.lib()
    big = B.FFNDesc(1024, 70000, 256, 0, 0, 1, 1, 0.0, 0x1000, None, 0x2000, None, None, 0x3000, 0x4000, None)
    assert L.pi_ffn_layer_static(ctypes.byref(big), None, None, None, None, None, None, None) == 2
    wide = B.FFNDesc(1024, 4096, 4096, 0, 0, 1, 1, 0.0, 0x1000, None, 0x2000, None, None, 0x3000, 0x4000, None)
    assert L.pi_ffn_layer_static(ctypes.byref(wide), None, None, None, None, None, None, None) == 2
