"""CPU oracle for the predictor-guided sparse FFN -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper around ``oracle.c`` (plain C, IEEE double accumulation,
ascending sums, no BLAS).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the CUDA library and
its Python binding never do, and the two share no code.

Every function states the definition it follows; the C file carries the page
citations.  Parity pins for each function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

F32, F16, Q4_0 = 0, 1, 2
ACT_RELU, ACT_RELU2 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Layer(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int64), ("d_ff", ctypes.c_int64), ("rank", ctypes.c_int64),
        ("gated", ctypes.c_int32), ("act", ctypes.c_int32),
        ("wtype", ctypes.c_int32), ("ptype", ctypes.c_int32),
        ("w_up", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
        ("b_act", ctypes.c_void_p), ("b_down", ctypes.c_void_p),
        ("p1", ctypes.c_void_p), ("p2", ctypes.c_void_p), ("p_bias", ctypes.c_void_p),
        ("threshold", ctypes.c_double), ("dense_prefix", ctypes.c_int64),
    ]


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_q4_0_quantize.argtypes = [P, i64, i64, P]
        lib.oracle_q4_0_quantize.restype = None
        lib.oracle_dequantize.argtypes = [P, ctypes.c_int32, i64, i64, P]
        lib.oracle_dequantize.restype = None
        lib.oracle_sparse_ffn.argtypes = [ctypes.POINTER(_Layer), P, P, i64, P, P, P]
        lib.oracle_sparse_ffn.restype = ctypes.c_int
        lib.oracle_dense_ffn.argtypes = [ctypes.POINTER(_Layer), P, P, P, P]
        lib.oracle_dense_ffn.restype = ctypes.c_int
        lib.oracle_true_mask.argtypes = [ctypes.POINTER(_Layer), P, P, P]
        lib.oracle_true_mask.restype = None
        lib.oracle_predict.argtypes = [ctypes.POINTER(_Layer), P, P, P, P]
        lib.oracle_predict.restype = None
        lib.oracle_compact.argtypes = [P, i64, P]
        lib.oracle_compact.restype = i64
        lib.oracle_fire_counts.argtypes = [ctypes.POINTER(_Layer), P, i64, P]
        lib.oracle_fire_counts.restype = None
        lib.oracle_hot_first_perm.argtypes = [P, i64, P]
        lib.oracle_hot_first_perm.restype = None
        lib.oracle_rms_residual.argtypes = [P, P, i64, P]
        lib.oracle_rms_residual.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _wtype_of(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype in (np.float16, np.uint16):
        return F16
    if a.dtype == np.uint8:
        return Q4_0
    raise TypeError(f"unsupported weight array dtype {a.dtype}")


def _as_bits(a):
    """fp16 arrays travel as their binary16 bit patterns."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    return a.view(np.uint16) if a.dtype == np.float16 else a


class Layer:
    """One FFN layer plus predictor, host arrays (neuron-major matrices).

    w_up / w_gate / w_down: [d_ff, d_model] as float32, float16 (or uint16 bit
    patterns), or uint8 Q4_0 blobs in the split layout of ``q4_0_quantize``.
    p1: [rank, d_model], p2: [d_ff, rank] (float32 or float16).
    """

    def __init__(self, d_model, d_ff, rank, w_up, w_down, w_gate=None, b_act=None, b_down=None,
                 p1=None, p2=None, p_bias=None, threshold=0.0, act=ACT_RELU, dense_prefix=0):
        self.d_model, self.d_ff, self.rank = int(d_model), int(d_ff), int(rank)
        self.gated = w_gate is not None
        self.wtype = _wtype_of(np.asarray(w_up))
        self.w_up = _as_bits(w_up)
        self.w_gate = _as_bits(w_gate)
        self.w_down = _as_bits(w_down)
        self.b_act = _c(b_act, np.float32)
        self.b_down = _c(b_down, np.float32)
        self.ptype = F32 if p1 is None else _wtype_of(np.asarray(p1))
        self.p1 = _as_bits(p1)
        self.p2 = _as_bits(p2)
        self.p_bias = _c(p_bias, np.float32)
        self.threshold = float(threshold)
        self.act = int(act)
        self.dense_prefix = int(dense_prefix)
        self._check()
        self._s = _Layer(self.d_model, self.d_ff, self.rank, int(self.gated), self.act,
                         self.wtype, self.ptype,
                         _ptr(self.w_up), _ptr(self.w_gate), _ptr(self.w_down),
                         _ptr(self.b_act), _ptr(self.b_down),
                         _ptr(self.p1), _ptr(self.p2), _ptr(self.p_bias), self.threshold, self.dense_prefix)

    def _check(self):
        d, F = self.d_model, self.d_ff
        for name in ("w_up", "w_gate", "w_down"):
            a = getattr(self, name)
            if a is None:
                continue
            if self.wtype == Q4_0:
                assert d % 32 == 0 and a.size == q4_0_bytes(F, d), name
            else:
                assert a.shape == (F, d), (name, a.shape)
        if self.p1 is not None:
            assert self.p1.shape == (self.rank, d) and self.p2.shape == (F, self.rank)
            assert self.ptype in (F32, F16)
        assert 0 <= self.dense_prefix <= F


def q4_0_bytes(rows: int, cols: int) -> int:
    return rows * (cols // 2) + rows * (cols // 32) * 2


def f16_to_f64(h) -> np.ndarray:
    lib = _L()
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f64(int(v)) for v in h], dtype=np.float64)


def f32_to_f16(f) -> np.ndarray:
    lib = _L()
    f = np.asarray(f, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_f16(float(v)) for v in f], dtype=np.uint16)


def q4_0_quantize(w: np.ndarray) -> np.ndarray:
    """Quantise a [rows, cols] float32 matrix (cols % 32 == 0) to a Q4_0 blob."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % 32 == 0
    out = np.zeros(q4_0_bytes(rows, cols), dtype=np.uint8)
    _L().oracle_q4_0_quantize(_ptr(w), rows, cols, _ptr(out))
    return out


def dequantize(m: np.ndarray, rows: int, cols: int) -> np.ndarray:
    m = _as_bits(m)
    out = np.empty((rows, cols), dtype=np.float64)
    _L().oracle_dequantize(_ptr(m), _wtype_of(m), rows, cols, _ptr(out))
    return out


def sparse_ffn(L: Layer, x: np.ndarray, idx: np.ndarray, want_a: bool = False):
    """y = sum over listed neurons (ascending) of a_j * W_down[j] + b_down, in fp64."""
    x = _c(x, np.float32)
    idx = _c(idx, np.int32)
    y = np.empty(L.d_model, dtype=np.float64)
    a = np.empty(max(1, idx.size), dtype=np.float64)
    z = np.empty(max(1, idx.size), dtype=np.float64)
    rc = _L().oracle_sparse_ffn(ctypes.byref(L._s), _ptr(x), _ptr(idx), idx.size, _ptr(y),
                                _ptr(a), _ptr(z))
    if rc != 0:
        raise ValueError("neuron index out of range")
    return (y, a[:idx.size], z[:idx.size]) if want_a else y


def dense_ffn(L: Layer, x: np.ndarray, want_a: bool = False):
    """The sparse FFN over every neuron 0..d_ff-1."""
    return sparse_ffn(L, x, np.arange(L.d_ff, dtype=np.int32), want_a)


def true_mask(L: Layer, x: np.ndarray):
    """(mask, z): mask_j = z_j > 0 with z the pre-activation feeding act()."""
    x = _c(x, np.float32)
    mask = np.empty(L.d_ff, dtype=np.uint8)
    z = np.empty(L.d_ff, dtype=np.float64)
    _L().oracle_true_mask(ctypes.byref(L._s), _ptr(x), _ptr(mask), _ptr(z))
    return mask, z


def predict(L: Layer, x: np.ndarray):
    """(h, logit, mask) of the low-rank predictor for one token; neurons below
    the layer's dense_prefix are always in the mask."""
    x = _c(x, np.float32)
    h = np.empty(L.rank, dtype=np.float64)
    logit = np.empty(L.d_ff, dtype=np.float64)
    mask = np.empty(L.d_ff, dtype=np.uint8)
    _L().oracle_predict(ctypes.byref(L._s), _ptr(x), _ptr(h), _ptr(logit), _ptr(mask))
    return h, logit, mask


def predict_union(L: Layer, X: np.ndarray):
    """Batched tokens share one active set: the union (OR) of per-token masks.
    Returns (logits [B, d_ff], union mask [d_ff])."""
    X = np.atleast_2d(X)
    logits = np.empty((X.shape[0], L.d_ff), dtype=np.float64)
    union = np.zeros(L.d_ff, dtype=np.uint8)
    for b in range(X.shape[0]):
        _, logits[b], m = predict(L, X[b])
        union |= m
    return logits, union


def compact(mask: np.ndarray) -> np.ndarray:
    """Ascending positions of the non-zero entries of mask."""
    mask = _c(mask, np.uint8)
    idx = np.empty(max(1, mask.size), dtype=np.int32)
    n = _L().oracle_compact(_ptr(mask), mask.size, _ptr(idx))
    return idx[:n].copy()


def fire_counts(L: Layer, X: np.ndarray) -> np.ndarray:
    X = _c(np.atleast_2d(X), np.float32)
    counts = np.zeros(L.d_ff, dtype=np.int32)
    _L().oracle_fire_counts(ctypes.byref(L._s), _ptr(X), X.shape[0], _ptr(counts))
    return counts


def hot_first_perm(counts: np.ndarray) -> np.ndarray:
    counts = _c(counts, np.int32)
    perm = np.empty(max(1, counts.size), dtype=np.int32)
    _L().oracle_hot_first_perm(_ptr(counts), counts.size, _ptr(perm))
    return perm[:counts.size].copy()


def rms_residual(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    y = _c(y, np.float64)
    out = np.empty(x.size, dtype=np.float64)
    _L().oracle_rms_residual(_ptr(x), _ptr(y), x.size, _ptr(out))
    return out


def neuron_shard(L: Layer, neurons: np.ndarray, keep_b_down: bool) -> Layer:
    """The layer restricted to the listed neurons: row neurons[i] of every
    per-neuron array (w_up, w_gate, w_down, b_act, p2, p_bias) becomes row i,
    p1 is shared, b_down is kept only when ``keep_b_down``.  Neurons are
    independent terms of the FFN sum, so the outputs of shards that partition
    0..d_ff-1 add up to the layer's output; the pages split one FFN between a
    GPU (hot neurons) and a CPU (cold neurons) that way (PowerInfer README
    translation, "摘要" abstract and "推理" inference)."""
    neurons = np.asarray(neurons, dtype=np.int64)
    d, F = L.d_model, L.d_ff

    def rows(a):
        if a is None:
            return None
        if L.wtype == Q4_0 and a.ndim == 1 and a.size == q4_0_bytes(F, d):
            codes = a[: F * (d // 2)].reshape(F, d // 2)[neurons]
            scales = a[F * (d // 2):].reshape(F, d // 16)[neurons]
            return np.concatenate([codes.ravel(), scales.ravel()])
        return np.ascontiguousarray(a[neurons])

    assert L.dense_prefix == 0, "a neuron shard of a layer with an always-on prefix is not defined"
    return Layer(d, neurons.size, L.rank, rows(L.w_up), rows(L.w_down), w_gate=rows(L.w_gate),
                 b_act=rows(L.b_act), b_down=L.b_down if keep_b_down else None, p1=L.p1, p2=rows(L.p2),
                 p_bias=rows(L.p_bias), threshold=L.threshold, act=L.act)


def recall_precision(pred_mask: np.ndarray, true_mask_: np.ndarray):
    """Predictor quality against the true activity: |M&T|/|T| and |M&T|/|M|."""
    m = np.asarray(pred_mask).astype(bool)
    t = np.asarray(true_mask_).astype(bool)
    inter = np.count_nonzero(m & t)
    rec = inter / max(1, np.count_nonzero(t))
    prec = inter / max(1, np.count_nonzero(m))
    return rec, prec
