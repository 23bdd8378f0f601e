"""The C-ABI library loads, exports every symbol include/pi.h declares, and its
host-side logic (validation, workspace sizing, host-only entry points) behaves
as documented.  No GPU: nothing here enqueues device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from activation_sparse_decode_predictor_gb300 import binding as B
from activation_sparse_decode_predictor_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return B.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "pi.h")).read()
    return sorted(set(re.findall(r"^PI_API [^(]*?\b(pi_\w+)\(", txt, flags=re.M)))


def test_header_declares_binding_exports():
    assert declared_symbols() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = set(re.findall(r" T (pi_\w+)", out))
    assert set(declared_symbols()) <= exported


def test_status_strings(L):
    for code in range(11):
        s = B.pi_status_str(code)
        assert s and s != "unknown status"
    assert B.pi_status_str(99) == "unknown status"


def _desc(**kw):
    d = dict(d_model=512, d_ff=2048, rank=64, gated=0, act=0, wtype=B.PI_F16, ptype=B.PI_F16, threshold=0.0,
             w_up=0x1000, w_gate=None, w_down=0x2000, b_act=None, b_down=None, p1=0x3000, p2=0x4000, p_bias=None,
             next=None, dense_prefix=0)
    d.update(kw)
    return B.FFNDesc(*[d[f] for f, _ in B.FFNDesc._fields_])


def _call_layer(L, desc, x=0x10000, batch=1, y=0x20000, residual=None, ws=0x40000, ws_bytes=1 << 30):
    return L.pi_ffn_layer(ctypes.byref(desc) if desc is not None else None, x, batch, residual, y, None, None, ws,
                          ws_bytes, None)


def test_validation_before_launch(L):
    assert _call_layer(L, None) == 1                                   # NULL desc
    assert _call_layer(L, _desc(d_model=100)) == 2                     # d_model % 8
    assert _call_layer(L, _desc(d_model=1 << 15)) == 2                 # above the maximum
    assert _call_layer(L, _desc(rank=12)) == 2                         # rank % 8
    assert _call_layer(L, _desc(d_ff=0)) == 2
    assert _call_layer(L, _desc(wtype=7)) == 3
    assert _call_layer(L, _desc(wtype=B.PI_Q4_0, d_model=520)) == 2    # Q4_0 needs d_model % 256
    assert _call_layer(L, _desc(ptype=B.PI_Q4_0)) == 3
    assert _call_layer(L, _desc(gated=1)) == 1                         # gated without w_gate
    assert _call_layer(L, _desc(w_up=0x1004)) == 4                     # misaligned weights
    assert _call_layer(L, _desc(), x=0x10004) == 4                     # misaligned x
    assert _call_layer(L, _desc(), batch=9) == 2                       # batch above 8
    assert _call_layer(L, _desc(), batch=0) == 2
    assert _call_layer(L, _desc(), y=0x10000) == 9                     # y overlaps x
    assert _call_layer(L, _desc(), residual=0x20010) == 9              # residual partially overlaps y
    assert _call_layer(L, _desc(), ws=None) == 8
    assert _call_layer(L, _desc(), ws=0x40010) == 4                    # workspace alignment
    assert _call_layer(L, _desc(), ws_bytes=16) == 8
    assert _call_layer(L, _desc(wtype=B.PI_F32), batch=2) == 3         # union path is fp16 / Q4_0
    assert _call_layer(L, _desc(dense_prefix=-1)) == 2                 # always-on prefix out of range
    assert _call_layer(L, _desc(dense_prefix=2049)) == 2


def test_compact_validation(L):
    assert L.pi_compact(None, 10, 0x100, 0x200, 10, 0x1000, 4096, None) == 1
    assert L.pi_compact(0x10, 0, 0x100, 0x200, 10, 0x1000, 4096, None) == 2
    assert L.pi_compact(0x10, 10, 0x102, 0x200, 10, 0x1000, 4096, None) == 4
    assert L.pi_compact(0x10, 10, 0x100, 0x200, 10, 0x1000, 8, None) == 8


def test_workspace_sizes(L):
    d = _desc()
    w1 = L.pi_workspace_bytes(ctypes.byref(d), 1)
    w8 = L.pi_workspace_bytes(ctypes.byref(d), 8)
    assert w1 % 256 == 0 and w8 > w1
    assert w1 >= 256 + (2048 // 32) * 8 + 64 * 4 + 2048 * 4
    assert L.pi_workspace_bytes(ctypes.byref(d), 9) == 0
    assert L.pi_compact_workspace_bytes(0) == 0
    assert L.pi_compact_workspace_bytes(100) >= 256 + 4 * 8


def test_q4_0_bytes(L):
    assert B.pi_q4_0_bytes(3, 64) == oracle.q4_0_bytes(3, 64) == 3 * 32 + 3 * 2 * 2
    assert B.pi_q4_0_bytes(3, 48) == 0


@pytest.mark.parametrize("n", [1, 7, 1000, 49152])
def test_hot_first_perm_host_matches_oracle(L, n):
    rng = np.random.default_rng(n)
    counts = rng.integers(0, 40, n).astype(np.int32)
    got = B.pi_hot_first_perm(counts)
    assert np.array_equal(got, np.argsort(-counts, kind="stable"))
    if n <= 1000:
        assert np.array_equal(got, oracle.hot_first_perm(counts))


def test_hot_first_perm_errors(L):
    assert L.pi_hot_first_perm(None, 4, None) == 1
    c = np.zeros(1, np.int32)
    assert L.pi_hot_first_perm(c.ctypes.data_as(ctypes.c_void_p), 0, c.ctypes.data_as(ctypes.c_void_p)) == 2


@pytest.mark.parametrize("n,shards", [(1, 1), (10, 3), (11008, 4), (4100, 7)])
def test_shard_neurons_deal_round_robin(L, n, shards):
    order = np.random.default_rng(n).permutation(n).astype(np.int32)
    parts = [B.pi_shard_neurons(order, shards, g) for g in range(shards)]
    for g, S in enumerate(parts):
        assert np.array_equal(S, order[g::shards])
    assert np.array_equal(np.sort(np.concatenate(parts)), np.arange(n))
    # hot-first order dealt round-robin: every shard's firing total is within
    # one maximum count of every other's
    counts = np.random.default_rng(n + 1).integers(0, 50, n).astype(np.int32)
    hot = B.pi_hot_first_perm(counts)
    tot = [counts[B.pi_shard_neurons(hot, shards, g)].sum() for g in range(shards)]
    assert max(tot) - min(tot) <= counts.max()


def test_shard_neurons_errors(L):
    o = np.arange(8, dtype=np.int32)
    p = o.ctypes.data_as(ctypes.c_void_p)
    out = np.zeros(8, np.int32)
    cnt = np.zeros(1, np.int32)
    po, pc = out.ctypes.data_as(ctypes.c_void_p), cnt.ctypes.data_as(ctypes.c_void_p)
    assert L.pi_shard_neurons(None, 8, 2, 0, po, pc) == 1
    assert L.pi_shard_neurons(p, 8, 0, 0, po, pc) == 2
    assert L.pi_shard_neurons(p, 8, 2, 2, po, pc) == 2
    assert L.pi_shard_neurons(p, 8, 9, 0, po, pc) == 2
    bad = np.array([0, 1, 2, 3, 4, 5, 6, 6], np.int32)          # not a permutation
    assert L.pi_shard_neurons(bad.ctypes.data_as(ctypes.c_void_p), 8, 2, 0, po, pc) == 10
    bad[7] = 8                                                   # out of range
    assert L.pi_shard_neurons(bad.ctypes.data_as(ctypes.c_void_p), 8, 2, 0, po, pc) == 10


@pytest.mark.parametrize("scale", [1.0, 1e-3, 3e-6, 1e-7, 250.0])
def test_host_quantiser_matches_oracle(L, scale):
    """pi_quantize_q4_0_host against the oracle's quantiser, byte for byte, at
    magnitudes whose scales are normal, subnormal and flushed to zero in
    binary16, with zero blocks and exact rounding ties mixed in."""
    rng = np.random.default_rng(int(scale * 1e7) % 1000 + 5)
    rows, cols = 37, 256
    w = (rng.standard_normal((rows, cols)) * scale).astype(np.float32)
    w[3, 32:64] = 0.0                                       # a zero block
    w[5, :32] = np.float32(scale) * np.arange(-16, 16, dtype=np.float32) / 2   # steps and half steps
    w[6, 64:96] = -w[6, 64:96]
    got = B.pi_quantize_q4_0_host(w)
    assert np.array_equal(got, oracle.q4_0_quantize(w))


def test_host_quantiser_across_binary16_range(L):
    """Blocks whose scales sweep binary16 from below its smallest subnormal to
    near its largest normal, through the subnormal/normal boundary."""
    rng = np.random.default_rng(11)
    rows = 400
    mags = np.logspace(-9, 5.5, rows).astype(np.float32)
    w = (rng.standard_normal((rows, 64)) * mags[:, None]).astype(np.float32)
    assert np.array_equal(B.pi_quantize_q4_0_host(w), oracle.q4_0_quantize(w))


def test_host_quantiser_hand_worked_block(L):
    w = np.zeros((1, 32), np.float32)
    for e, v in {0: 1.0, 1: -4.0, 2: 3.5, 3: 0.3, 4: 0.25, 5: -0.25, 6: 4.0, 7: -3.9, 16: 2.0, 17: -1.75,
                 31: 0.74}.items():
        w[0, e] = v
    assert B.pi_quantize_q4_0_host(w).tobytes() == bytes.fromhex("CA508F8989888F8088888888888888980038")


def test_other_entry_validation(L):
    assert L.pi_quantize_q4_0(0x100, 0, 4, 48, 0x200, None) == 2          # cols % 32
    assert L.pi_quantize_q4_0(0x100, 2, 4, 64, 0x200, None) == 3          # source type
    assert L.pi_quantize_q4_0(0x100, 0, 4, 64, 0x108, None) == 4
    assert L.pi_quantize_q4_0(0x1000, 0, 4, 64, 0x1010, None) == 9       # overlap
    assert L.pi_quantize_q4_0_host(None, 4, 64, 0x100) == 1
    assert L.pi_quantize_q4_0_host(0x100, 4, 48, 0x100000) == 2           # cols % 32
    assert L.pi_quantize_q4_0_host(0x1000, 4, 64, 0x1010) == 9           # overlap
    assert L.pi_permute_rows(0x100, 0x1000, 4, 16, None, None) == 1
    assert L.pi_permute_rows(0x100, 0x110, 4, 16, 0x200, None) == 9
    assert L.pi_gather_rows(0x100, 4, 0x1000, 0, 16, 0x200, None) == 2      # no destination rows
    assert L.pi_gather_rows(0x100, 4, 0x1000, 2, 16, 0x202, None) == 4      # misaligned idx
    assert L.pi_gather_rows(0x100, 4, 0x120, 2, 16, 0x200, None) == 9       # dst inside src
    assert L.pi_gather_rows(None, 4, 0x1000, 2, 16, 0x200, None) == 1
    assert L.pi_rms_residual(0x100, 0x200, 0, 8, 0x300, None) == 2
    assert L.pi_sync_status(None, 0, None) == 8
