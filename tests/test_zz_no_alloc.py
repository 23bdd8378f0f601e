"""The allocation-free layer step (pi_ffn_layer_static), for callers that
cannot allocate device memory, must give the same results as the regular
workspace-based pi_ffn_layer.  Called through the C ABI, twice in a row, so
the second call runs on the scratch array the first call left behind."""
import ctypes

import numpy as np
import pytest
import torch

from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import build, synth

from helpers import assert_ffn_close

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_path():
    build.build()
    L = B.lib()
    d, F, r = 1024, 4096, 256
    lay = B.Layer.from_dict(synth.make_layer(d, F, r, gated=True, wtype="f16", sparsity=0.9, seed=61,
                                             device="cuda"))
    X = synth.tokens(2, d, 62, device="cuda")
    res = synth.tokens(2, d, 63, device="cuda")
    stream = torch.cuda.current_stream()
    for t in range(2):                                   # two calls in a row on the shared scratch
        y_ref = torch.empty(d, device="cuda")
        idx_ref = torch.zeros(F, dtype=torch.int32, device="cuda")
        n_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = B.pi_ffn_layer(lay, X[t], y_ref, residual=res[t], idx=idx_ref, n_active=n_ref)
        assert B.pi_sync_status(ws) == 0

        y = torch.empty(d, device="cuda")
        idx = torch.zeros(F, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        st = L.pi_ffn_layer_static(ctypes.byref(lay.desc), ctypes.c_void_p(X[t].data_ptr()),
                                   ctypes.c_void_p(res[t].data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                   ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(n.data_ptr()),
                                   ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert int(n.item()) == int(n_ref.item()) > 0
        k = int(n.item())
        assert np.array_equal(idx[:k].cpu().numpy(), idx_ref[:k].cpu().numpy())
        assert_ffn_close(y.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64), what=f"static call {t}")


def test_static_rejects_oversized_layer():
    build.build()
    L = B.lib()
    big = B.FFNDesc(1024, 70000, 256, 0, 0, 1, 1, 0.0, 0x1000, None, 0x2000, None, None, 0x3000, 0x4000, None)
    assert L.pi_ffn_layer_static(ctypes.byref(big), None, None, None, None, None, None, None) == 2
