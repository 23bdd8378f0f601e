"""Test-side helpers: build the same seeded layer for the CUDA library (device
tensors) and for the oracle (host arrays), and the parity criteria.

Inputs flow generator -> both sides.  Q4_0 blobs fed to both sides are made
by the oracle's quantiser (the CUDA quantiser is tested against it
separately), so no oracle input ever comes from the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import synth
from activation_sparse_decode_predictor_gb300 import binding as B

# Output tolerance of the method's fp32-accumulating kernels against the oracle
# (relative L2 and max-abs error), from the workload specification.
REL_L2 = 1e-3
MAX_ABS = 1e-2


def to_host(L: dict) -> dict:
    return {k: (v.detach().cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}


def q4_blob_random(rows: int, cols: int, seed: int) -> np.ndarray:
    """A random Q4_0 blob with codes 6..10 and scales 0.5 or 1, so weights are
    multiples of 0.5 in [-2, 2]: with small integer tokens every fp32 partial
    sum of a layer of a few hundred neurons stays exactly representable."""
    rng = np.random.default_rng(seed)
    lo = rng.integers(6, 11, rows * cols // 2)
    hi = rng.integers(6, 11, rows * cols // 2)
    codes = (lo | (hi << 4)).astype(np.uint8)
    scales = (2.0 ** rng.integers(-1, 1, rows * (cols // 32))).astype(np.float16).view(np.uint8)
    return np.concatenate([codes, scales])


def make_pair(L: dict, device="cuda", act=0, quantize=True):
    """(library Layer, oracle Layer, host dict) for a synth layer dict.

    A "q4_0" layer's fp16 matrices are quantised by the oracle's quantiser and
    the same bytes are uploaded."""
    H = to_host(L)
    wtype = L["wtype"]
    if wtype == "q4_0" and quantize:
        for k in ("w_up", "w_gate", "w_down"):
            if H[k] is not None and H[k].dtype != np.uint8:
                H[k] = oracle.q4_0_quantize(H[k].astype(np.float32))
    dev = {}
    for k in ("w_up", "w_gate", "w_down", "b_act", "b_down", "p1", "p2", "p_bias"):
        v = H.get(k)
        dev[k] = None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(device)
    lay = B.Layer(L["d_model"], L["d_ff"], L["rank"], dev["w_up"], dev["w_down"], w_gate=dev["w_gate"],
                  b_act=dev["b_act"], b_down=dev["b_down"], p1=dev["p1"], p2=dev["p2"], p_bias=dev["p_bias"],
                  threshold=L["threshold"], act=act,
                  wtype=B.PI_Q4_0 if wtype == "q4_0" else None)
    olay = oracle.Layer(L["d_model"], L["d_ff"], L["rank"], H["w_up"], H["w_down"], w_gate=H["w_gate"],
                        b_act=H["b_act"], b_down=H["b_down"], p1=H["p1"], p2=H["p2"], p_bias=H["p_bias"],
                        threshold=L["threshold"], act=act)
    return lay, olay, H


def assert_ffn_close(y_gpu, y_ref, rel_l2=REL_L2, max_abs=MAX_ABS, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64).ravel()
    y_ref = np.asarray(y_ref, dtype=np.float64).ravel()
    err = y_gpu - y_ref
    nref = np.linalg.norm(y_ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else 0.0
    mx = float(np.max(np.abs(err))) if err.size else 0.0
    assert rel <= rel_l2 and mx <= max_abs, f"{what}: rel L2 {rel:.3e} (<= {rel_l2}), max abs {mx:.3e} (<= {max_abs})"
    return rel, mx


def logit_scale(H: dict, h: np.ndarray) -> np.ndarray:
    """Per-neuron magnitude sum_k |P2[j,k] h_k| + |p_bias_j|: scales the fp32
    rounding bound of a logit."""
    p2 = H["p2"].astype(np.float64)
    m = np.abs(p2) @ np.abs(h)
    if H.get("p_bias") is not None:
        m = m + np.abs(H["p_bias"].astype(np.float64))
    return m


def ambiguous(logit_ref: np.ndarray, scale: np.ndarray, tau: float) -> np.ndarray:
    """Neurons whose logit is so close to the threshold that an fp32 sum may
    land on either side: either decision is correct there."""
    return np.abs(logit_ref - tau) <= 2e-5 * (scale + 1.0)
