"""Python binding of libpi_sparse_ffn.so (ctypes; argument marshalling only).

Every function below has the name of the C entry point it calls (include/pi.h)
and does nothing but turn torch tensors into pointers, pick the current CUDA
stream and raise on a non-OK status.  All compute runs in the library's CUDA
kernels; there is no Python or CPU path.  Importing works without a GPU;
calling needs the built library (``build.build()``) and a CUDA device, and
fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpi_sparse_ffn.so")

PI_OK = 0
PI_F32, PI_F16, PI_Q4_0 = 0, 1, 2
PI_ACT_RELU, PI_ACT_RELU2 = 0, 1
PI_MAX_BATCH = 8
STATUS_NAMES = {0: "PI_OK", 1: "PI_ERR_NULL", 2: "PI_ERR_SHAPE", 3: "PI_ERR_DTYPE", 4: "PI_ERR_ALIGN",
                5: "PI_ERR_CAPACITY", 6: "PI_ERR_CUDA", 7: "PI_ERR_TIMEOUT", 8: "PI_ERR_WORKSPACE",
                9: "PI_ERR_ALIAS", 10: "PI_ERR_INDEX"}

# every symbol include/pi.h declares
EXPORTS = ("pi_status_str", "pi_workspace_bytes", "pi_compact_workspace_bytes", "pi_compact", "pi_predict",
           "pi_sparse_ffn", "pi_ffn_layer", "pi_dense_ffn", "pi_q4_0_bytes", "pi_quantize_q4_0",
           "pi_quantize_q4_0_host", "pi_fire_counts", "pi_hot_first_perm", "pi_permute_rows", "pi_gather_rows",
           "pi_shard_neurons",
           "pi_rms_residual", "pi_sync_status", "pi_ffn_layer_static", "pi_ffn_layer_chain")


class PiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({_str(status)})")


class FFNDesc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("gated", ctypes.c_int32), ("act", ctypes.c_int32), ("wtype", ctypes.c_int32),
                ("ptype", ctypes.c_int32), ("threshold", ctypes.c_float),
                ("w_up", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("b_act", ctypes.c_void_p), ("b_down", ctypes.c_void_p),
                ("p1", ctypes.c_void_p), ("p2", ctypes.c_void_p), ("p_bias", ctypes.c_void_p),
                ("next", ctypes.c_void_p), ("dense_prefix", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library missing: {LIB_PATH}; run activation_sparse_decode_predictor_gb300"
                               ".build.build() (nvcc, sm_103a) first")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(FFNDesc)
        sig = {
            "pi_status_str": ([i32], ctypes.c_char_p),
            "pi_workspace_bytes": ([D, i32], sz),
            "pi_compact_workspace_bytes": ([i32], sz),
            "pi_compact": ([P, i32, P, P, i32, P, sz, P], i32),
            "pi_predict": ([D, P, i32, P, P, P, P, i32, P, sz, P], i32),
            "pi_sparse_ffn": ([D, P, i32, P, P, P, P, P, sz, P], i32),
            "pi_ffn_layer": ([D, P, i32, P, P, P, P, P, sz, P], i32),
            "pi_dense_ffn": ([D, P, i32, P, P, P, sz, P], i32),
            "pi_q4_0_bytes": ([i64, i64], sz),
            "pi_quantize_q4_0": ([P, i32, i64, i64, P, P], i32),
            "pi_quantize_q4_0_host": ([P, i64, i64, P], i32),
            "pi_fire_counts": ([D, P, i32, P, P], i32),
            "pi_hot_first_perm": ([P, i32, P], i32),
            "pi_permute_rows": ([P, P, i64, i64, P, P], i32),
            "pi_gather_rows": ([P, i64, P, i64, i64, P, P], i32),
            "pi_shard_neurons": ([P, i32, i32, i32, P, P], i32),
            "pi_rms_residual": ([P, P, i32, i32, P, P], i32),
            "pi_sync_status": ([P, sz, P], i32),
            "pi_ffn_layer_static": ([D, P, P, P, P, P, P, P], i32),
            "pi_ffn_layer_chain": ([D, P, P, i32, P, P, P, P, P, sz, P], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _str(status: int) -> str:
    try:
        return lib().pi_status_str(int(status)).decode()
    except Exception:  # noqa: BLE001 -- message only
        return "?"


def _check(st: int, where: str):
    if st != PI_OK:
        raise PiError(st, where)


def _p(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def q4_0_bytes(rows: int, cols: int) -> int:
    return rows * (cols // 2) + rows * (cols // 32) * 2


class Layer:
    """One FFN layer + predictor on the device, and its pi_ffn_desc.

    Keeps references to the tensors so the descriptor's pointers stay valid.
    Matrices: float32 / float16 [d_ff, d_model], or uint8 Q4_0 blobs
    (``wtype=PI_Q4_0``).  p1 [rank, d_model], p2 [d_ff, rank] float32 / float16.
    """

    def __init__(self, d_model, d_ff, rank, w_up, w_down, w_gate=None, b_act=None, b_down=None, p1=None, p2=None,
                 p_bias=None, threshold=0.0, act=PI_ACT_RELU, wtype=None, dense_prefix=0):
        self.tensors = dict(w_up=w_up, w_gate=w_gate, w_down=w_down, b_act=b_act, b_down=b_down, p1=p1, p2=p2,
                            p_bias=p_bias)
        for k, v in self.tensors.items():
            if v is not None:
                _dev(v, k)
        if wtype is None:
            wtype = {torch.float32: PI_F32, torch.float16: PI_F16, torch.uint8: PI_Q4_0}[w_up.dtype]
        ptype = PI_F16 if (p1 is not None and p1.dtype == torch.float16) else PI_F32
        self.d_model, self.d_ff, self.rank = int(d_model), int(d_ff), int(rank)
        self.gated = w_gate is not None
        self.wtype, self.ptype = wtype, ptype
        self.desc = FFNDesc(self.d_model, self.d_ff, self.rank, int(self.gated), int(act), int(wtype), int(ptype),
                            float(threshold), _p(w_up), _p(w_gate), _p(w_down), _p(b_act), _p(b_down), _p(p1),
                            _p(p2), _p(p_bias), None, int(dense_prefix))

    def set_next(self, other: "Layer | None"):
        """Name the layer run next on the same stream (a scheduling hint the
        current kernels do not use), or None."""
        self._next = other
        self.desc.next = ctypes.addressof(other.desc) if other is not None else None

    def shard(self, neurons, keep_b_down: bool, stream=None) -> "Layer":
        """The layer restricted to the neurons listed in `neurons` (device int32,
        e.g. one shard of pi_shard_neurons): their rows of every per-neuron array
        gathered in list order, p1 shared.  b_down is kept only when
        `keep_b_down` (the shard that adds it; the partial outputs of all shards
        sum to the layer output)."""
        _dev(neurons, "neurons")
        if self.desc.dense_prefix:
            raise ValueError("a neuron shard of a layer with an always-on prefix is not defined")
        n, F, d = int(neurons.numel()), self.d_ff, self.d_model
        T = self.tensors

        def rows(t):
            if t is None:
                return None
            if self.wtype == PI_Q4_0 and t.dtype == torch.uint8:
                t = t.reshape(-1)  # the blob: all code rows, then all scale rows
                codes, scales = F * (d // 2), F * (d // 32) * 2
                out = torch.empty(q4_0_bytes(n, d), dtype=torch.uint8, device=t.device)
                pi_gather_rows(t[:codes].view(F, d // 2), neurons, out[: n * (d // 2)].view(n, d // 2), stream)
                pi_gather_rows(t[codes:codes + scales].view(F, d // 16), neurons,
                               out[n * (d // 2):].view(n, d // 16), stream)
                return out
            return pi_gather_rows(t, neurons, stream=stream)

        return Layer(d, n, self.rank, rows(T["w_up"]), rows(T["w_down"]), w_gate=rows(T["w_gate"]),
                     b_act=rows(T["b_act"]), b_down=T["b_down"] if keep_b_down else None, p1=T["p1"],
                     p2=rows(T["p2"]), p_bias=rows(T["p_bias"]), threshold=self.desc.threshold, act=self.desc.act,
                     wtype=self.wtype)

    @classmethod
    def from_dict(cls, L: dict, act=PI_ACT_RELU, threshold=None):
        return cls(L["d_model"], L["d_ff"], L["rank"], L["w_up"], L["w_down"], w_gate=L.get("w_gate"),
                   b_act=L.get("b_act"), b_down=L.get("b_down"), p1=L.get("p1"), p2=L.get("p2"),
                   p_bias=L.get("p_bias"), threshold=L.get("threshold", 0.0) if threshold is None else threshold,
                   act=act, wtype=L.get("wtype_code"), dense_prefix=L.get("dense_prefix", 0))


def pi_status_str(status: int) -> str:
    return _str(status)


def pi_workspace_bytes(layer: Layer, batch: int = 1) -> int:
    return int(lib().pi_workspace_bytes(ctypes.byref(layer.desc), int(batch)))


def pi_compact_workspace_bytes(n: int) -> int:
    return int(lib().pi_compact_workspace_bytes(int(n)))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace of nbytes (torch allocations are 256-aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def pi_compact(mask, idx, count, cap=None, ws=None, stream=None):
    n = mask.numel()
    if ws is None:
        ws = workspace(pi_compact_workspace_bytes(n), mask.device)
    cap = idx.numel() if cap is None else cap
    _check(lib().pi_compact(_p(mask), n, _p(idx), _p(count), int(cap), _p(ws), ws.numel(), _stream(stream)),
           "pi_compact")
    return ws


def pi_predict(layer: Layer, x, idx, n_active, logits=None, mask=None, cap=None, ws=None, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    if ws is None:
        ws = workspace(pi_workspace_bytes(layer, B), x.device)
    cap = idx.numel() if cap is None else cap
    _check(lib().pi_predict(ctypes.byref(layer.desc), _p(x), B, _p(logits), _p(mask), _p(idx), _p(n_active),
                            int(cap), _p(ws), ws.numel(), _stream(stream)), "pi_predict")
    return ws


def pi_sparse_ffn(layer: Layer, x, idx, n_active, y, residual=None, ws=None, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    if ws is None:
        ws = workspace(pi_workspace_bytes(layer, B), x.device)
    _check(lib().pi_sparse_ffn(ctypes.byref(layer.desc), _p(x), B, _p(idx), _p(n_active), _p(residual), _p(y),
                               _p(ws), ws.numel(), _stream(stream)), "pi_sparse_ffn")
    return ws


def pi_ffn_layer(layer: Layer, x, y, residual=None, idx=None, n_active=None, ws=None, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    if ws is None:
        ws = workspace(pi_workspace_bytes(layer, B), x.device)
    _check(lib().pi_ffn_layer(ctypes.byref(layer.desc), _p(x), B, _p(residual), _p(y), _p(idx), _p(n_active),
                              _p(ws), ws.numel(), _stream(stream)), "pi_ffn_layer")
    return ws


def pi_ffn_layer_chain(layer: Layer, x_prev, y_prev, x, y, idx=None, n_active=None, ws=None, stream=None):
    """Layer of a stack fed by the previous one: x = rms rescale of x_prev +
    y_prev (written to x), then y = the layer at x."""
    B_ = x_prev.shape[0] if x_prev.dim() == 2 else 1
    if ws is None:
        ws = workspace(pi_workspace_bytes(layer, B_), x_prev.device)
    _check(lib().pi_ffn_layer_chain(ctypes.byref(layer.desc), _p(x_prev), _p(y_prev), B_, _p(x), _p(y), _p(idx),
                                    _p(n_active), _p(ws), ws.numel(), _stream(stream)), "pi_ffn_layer_chain")
    return ws


def pi_dense_ffn(layer: Layer, x, y, residual=None, ws=None, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    if ws is None:
        ws = workspace(pi_workspace_bytes(layer, B), x.device)
    _check(lib().pi_dense_ffn(ctypes.byref(layer.desc), _p(x), B, _p(residual), _p(y), _p(ws), ws.numel(),
                              _stream(stream)), "pi_dense_ffn")
    return ws


def pi_q4_0_bytes(rows: int, cols: int) -> int:
    return int(lib().pi_q4_0_bytes(int(rows), int(cols)))


def pi_quantize_q4_0(src, dst=None, stream=None):
    rows, cols = src.shape
    st = {torch.float32: PI_F32, torch.float16: PI_F16}[src.dtype]
    if dst is None:
        dst = torch.empty(q4_0_bytes(rows, cols), dtype=torch.uint8, device=src.device)
    _check(lib().pi_quantize_q4_0(_p(src), st, rows, cols, _p(dst), _stream(stream)), "pi_quantize_q4_0")
    return dst


def pi_quantize_q4_0_host(w) -> np.ndarray:
    """Q4_0 blob of a host fp32 [rows, cols] matrix, quantised on the CPU by the library."""
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float32))
    rows, cols = w.shape
    out = np.empty(max(1, q4_0_bytes(rows, cols)), dtype=np.uint8)
    _check(lib().pi_quantize_q4_0_host(w.ctypes.data_as(ctypes.c_void_p), rows, cols,
                                       out.ctypes.data_as(ctypes.c_void_p)), "pi_quantize_q4_0_host")
    return out


def pi_fire_counts(layer: Layer, X, counts, stream=None):
    _check(lib().pi_fire_counts(ctypes.byref(layer.desc), _p(X), int(X.shape[0]), _p(counts), _stream(stream)),
           "pi_fire_counts")


def pi_hot_first_perm(counts) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    perm = np.empty_like(c)
    _check(lib().pi_hot_first_perm(c.ctypes.data_as(ctypes.c_void_p), c.size, perm.ctypes.data_as(ctypes.c_void_p)),
           "pi_hot_first_perm")
    return perm


def pi_permute_rows(src, perm, dst=None, stream=None):
    rows = src.shape[0]
    row_bytes = src.numel() * src.element_size() // rows
    if dst is None:
        dst = torch.empty_like(src)
    _check(lib().pi_permute_rows(_p(src), _p(dst), rows, row_bytes, _p(perm), _stream(stream)), "pi_permute_rows")
    return dst


def pi_gather_rows(src, idx, dst=None, stream=None):
    """dst[i] = src[idx[i]] along the first dimension (device tensors)."""
    rows = src.shape[0]
    row_bytes = src.numel() * src.element_size() // rows
    if dst is None:
        dst = torch.empty((idx.numel(),) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    _check(lib().pi_gather_rows(_p(src), rows, _p(dst), int(dst.shape[0]), row_bytes, _p(idx), _stream(stream)),
           "pi_gather_rows")
    return dst


def pi_shard_neurons(order, shards: int, shard: int) -> np.ndarray:
    """Neurons of shard `shard` of `shards` when `order` is dealt round-robin."""
    o = np.ascontiguousarray(np.asarray(order, dtype=np.int32))
    out = np.empty(max(1, -(-o.size // max(1, shards))), dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int32)
    _check(lib().pi_shard_neurons(o.ctypes.data_as(ctypes.c_void_p), o.size, int(shards), int(shard),
                                  out.ctypes.data_as(ctypes.c_void_p), cnt.ctypes.data_as(ctypes.c_void_p)),
           "pi_shard_neurons")
    return out[: int(cnt[0])].copy()


def pi_rms_residual(x, y, out, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    _check(lib().pi_rms_residual(_p(x), _p(y), B, int(x.shape[-1]), _p(out), _stream(stream)), "pi_rms_residual")


def pi_sync_status(ws, stream=None) -> int:
    """Status code of the device error word (and clears it); does not raise."""
    return int(lib().pi_sync_status(_p(ws), ws.numel(), _stream(stream)))
