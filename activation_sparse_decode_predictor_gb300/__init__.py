"""Predictor-guided, neuron-aware sparse FFN for single-token decode (GB300, sm_103a).

The compute lives in ``libpi_sparse_ffn.so`` (hand-written CUDA kernels behind a
C ABI, ``include/pi.h``); ``binding`` calls it through ctypes.  ``synth`` draws
the seeded synthetic workloads.  Build with ``build.build()``.
"""
from . import synth  # noqa: F401
from .binding import (  # noqa: F401
    EXPORTS, FFNDesc, Layer, PiError, PI_ACT_RELU, PI_ACT_RELU2, PI_F16, PI_F32, PI_Q4_0, lib,
    pi_compact, pi_compact_workspace_bytes, pi_dense_ffn, pi_ffn_layer, pi_fire_counts, pi_gather_rows,
    pi_hot_first_perm, pi_permute_rows, pi_predict, pi_q4_0_bytes, pi_quantize_q4_0, pi_quantize_q4_0_host, pi_rms_residual,
    pi_shard_neurons, pi_sparse_ffn, pi_status_str, pi_sync_status, pi_workspace_bytes, workspace,
)
