"""Pins for the CPU oracle, against things other than the oracle itself:
library routines (numpy's binary16, argsort, flatnonzero, float64 matmul),
closed forms, exact integer arithmetic, brute force on tiny shapes and the
invariants the method's definition fixes.  CPU only."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np_layer(d, F, r, gated, wtype, seed, act=oracle.ACT_RELU, sparsity=0.7):
    L = synth.make_layer(d, F, r, gated=gated, wtype="f32" if wtype == "f32" else "f16",
                         sparsity=sparsity, predictor="random", seed=seed)
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    if wtype == "q4_0":
        for k in ("w_up", "w_gate", "w_down"):
            if w[k] is not None:
                w[k] = oracle.q4_0_quantize(w[k].astype(np.float32))
    lay = oracle.Layer(d, F, r, w["w_up"], w["w_down"], w_gate=w["w_gate"], b_act=w["b_act"],
                       b_down=w["b_down"] + 0.25, p1=w["p1"], p2=w["p2"], p_bias=w["p_bias"],
                       threshold=0.0, act=act)
    return lay, w


def _dense_np(lay, w, x):
    """The FFN written with numpy float64 matmuls (a library routine)."""
    d, F = lay.d_model, lay.d_ff
    deq = lambda m: oracle.dequantize(m, F, d) if lay.wtype == oracle.Q4_0 else m.astype(np.float64)
    x = x.astype(np.float64)
    z = deq(w["w_gate"] if lay.gated else w["w_up"]) @ x + w["b_act"].astype(np.float64)
    a = np.maximum(z, 0.0)
    if lay.act == oracle.ACT_RELU2:
        a = a * a
    if lay.gated:
        a = a * (deq(w["w_up"]) @ x)
    return deq(w["w_down"]).T @ a + (w["b_down"] + 0.25).astype(np.float64), a, z


# --- binary16 conversions ------------------------------------------------------

def test_f16_to_f64_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f32_to_f16_round_to_nearest_even_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 5, 3000),
        np.array([0.0, -0.0, 65504, 65519.9, 65520, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2049, 2051],
                 dtype=np.float32)])
    ours = oracle.f32_to_f16(vals)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# --- compaction ----------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 5, 12])
def test_compact_brute_force_all_masks(n):
    for bits in itertools.product([0, 1], repeat=n):
        m = np.array(bits, dtype=np.uint8)
        assert np.array_equal(oracle.compact(m), np.flatnonzero(m).astype(np.int32))


@pytest.mark.parametrize("n", [31, 32, 33, 1000, 11008, 49152])
def test_compact_edges(n):
    rng = np.random.default_rng(n)
    masks = [np.zeros(n, np.uint8), np.ones(n, np.uint8),
             (rng.random(n) < 0.1).astype(np.uint8), (rng.integers(0, 255, n)).astype(np.uint8)]
    for pos in (0, n - 1, min(n - 1, 31), min(n - 1, 32)):
        m = np.zeros(n, np.uint8)
        m[pos] = 1
        masks.append(m)
    for m in masks:
        assert np.array_equal(oracle.compact(m), np.flatnonzero(m).astype(np.int32))


# --- FFN definition ------------------------------------------------------------

@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
@pytest.mark.parametrize("act", [oracle.ACT_RELU, oracle.ACT_RELU2])
def test_dense_matches_float64_matmul(gated, wtype, act):
    lay, w = _np_layer(64, 96, 16, gated, wtype, seed=3, act=act)
    x = synth.tokens(3, 64, 5).numpy()
    for t in range(3):
        y = oracle.dense_ffn(lay, x[t])
        y_ref, _, _ = _dense_np(lay, w, x[t])
        np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gated", [False, True])
def test_dense_is_exact_on_integer_layers(gated):
    L = synth.integer_layer(48, 80, 8, gated=gated, wtype="f16", seed=11)
    x = synth.integer_tokens(4, 48, 12).numpy()
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    lay = oracle.Layer(48, 80, 8, w["w_up"], w["w_down"], w_gate=w["w_gate"], b_act=w["b_act"],
                       b_down=w["b_down"], p1=w["p1"], p2=w["p2"], p_bias=w["p_bias"])
    I = lambda a: a.astype(np.float32).astype(np.int64)
    for t in range(4):
        xi = I(x[t])
        z = I(w["w_gate"] if gated else w["w_up"]) @ xi + I(w["b_act"])
        a = np.maximum(z, 0)
        if gated:
            a = a * (I(w["w_up"]) @ xi)
        y_int = I(w["w_down"]).T @ a + I(w["b_down"])
        assert np.array_equal(oracle.dense_ffn(lay, x[t]), y_int.astype(np.float64))


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("wtype", ["f32", "f16", "q4_0"])
def test_superset_of_true_mask_equals_dense_bitwise(gated, wtype):
    lay, _ = _np_layer(64, 200, 16, gated, wtype, seed=7)
    x = synth.tokens(4, 64, 9).numpy()
    rng = np.random.default_rng(0)
    for t in range(4):
        y_dense = oracle.dense_ffn(lay, x[t])
        T, _ = oracle.true_mask(lay, x[t])
        for extra in (0.0, 0.3, 1.0):
            M = T | (rng.random(lay.d_ff) < extra).astype(np.uint8)
            y = oracle.sparse_ffn(lay, x[t], oracle.compact(M))
            assert np.array_equal(y, y_dense)          # bitwise: skipped terms are exact zeros


@pytest.mark.parametrize("gated", [False, True])
def test_missing_neurons_closed_form(gated):
    """dense - sparse(M) = sum over j in T \\ M of a_j W_down[j]."""
    lay, w = _np_layer(64, 160, 16, gated, "f16", seed=21)
    x = synth.tokens(2, 64, 22).numpy()
    rng = np.random.default_rng(5)
    wd = w["w_down"].astype(np.float64)
    for t in range(2):
        T, _ = oracle.true_mask(lay, x[t])
        M = T & (rng.random(lay.d_ff) < 0.5).astype(np.uint8)
        y_dense, a_all, _ = oracle.dense_ffn(lay, x[t], want_a=True)
        y_sparse = oracle.sparse_ffn(lay, x[t], oracle.compact(M))
        missing = np.flatnonzero(T & (1 - M))
        np.testing.assert_allclose(y_dense - y_sparse, a_all[missing] @ wd[missing], rtol=1e-10,
                                   atol=1e-10)


def test_sparse_brute_force_all_masks_tiny():
    d, F = 6, 9
    rng = np.random.default_rng(4)
    wu = rng.standard_normal((F, d)).astype(np.float32)
    wd = rng.standard_normal((F, d)).astype(np.float32)
    b = rng.standard_normal(F).astype(np.float32)
    bd = rng.standard_normal(d).astype(np.float32)
    lay = oracle.Layer(d, F, 0, wu, wd, b_act=b, b_down=bd)
    x = rng.standard_normal(d).astype(np.float32)
    a = np.maximum(wu.astype(np.float64) @ x + b, 0.0)
    for bits in itertools.product([0, 1], repeat=F):
        m = np.array(bits, dtype=bool)
        y = oracle.sparse_ffn(lay, x, np.flatnonzero(m).astype(np.int32))
        ref = (a[m][:, None] * wd.astype(np.float64)[m]).sum(0) + bd
        np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_neuron_permutation_leaves_output_unchanged():
    L = synth.integer_layer(40, 70, 8, gated=True, wtype="f16", seed=31)
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    perm = np.random.default_rng(2).permutation(70)
    mk = lambda p: oracle.Layer(40, 70, 8, w["w_up"][p], w["w_down"][p], w_gate=w["w_gate"][p],
                                b_act=w["b_act"][p], b_down=w["b_down"], p1=w["p1"], p2=w["p2"][p],
                                p_bias=w["p_bias"][p], threshold=0.5)
    x = synth.integer_tokens(3, 40, 32).numpy()
    L0, L1 = mk(np.arange(70)), mk(perm)
    for t in range(3):
        assert np.array_equal(oracle.dense_ffn(L0, x[t]), oracle.dense_ffn(L1, x[t]))
        _, lg0, m0 = oracle.predict(L0, x[t])
        _, lg1, m1 = oracle.predict(L1, x[t])
        assert np.array_equal(lg1, lg0[perm]) and np.array_equal(m1, m0[perm])


# --- predictor -----------------------------------------------------------------

@pytest.mark.parametrize("shards", [1, 2, 3, 5])
@pytest.mark.parametrize("gated,wtype,act", [(False, "f16", oracle.ACT_RELU), (True, "q4_0", oracle.ACT_RELU),
                                             (True, "f32", oracle.ACT_RELU2)])
def test_neuron_shards_sum_to_the_layer(shards, gated, wtype, act):
    """Neuron sharding: the shards' partial outputs (b_down on shard 0 only) add
    up to the layer output computed with float64 matmuls, and each shard's
    predictor decisions are the layer's decisions on its neurons."""
    d, F, r = 64, 301, 16
    lay, w = _np_layer(d, F, r, gated, wtype, seed=41 + shards, act=act)
    order = np.random.default_rng(shards).permutation(F).astype(np.int32)
    x = np.random.default_rng(7).standard_normal(d).astype(np.float32)
    _, _, mask = oracle.predict(lay, x)
    idx = oracle.compact(mask)
    y_parts = []
    for g in range(shards):
        S = order[g::shards]
        sh = oracle.neuron_shard(lay, S, keep_b_down=(g == 0))
        assert sh.d_ff == S.size
        _, _, m_g = oracle.predict(sh, x)
        assert np.array_equal(m_g, mask[S])
        y_parts.append(oracle.sparse_ffn(sh, x, oracle.compact(m_g)))
    y_ref = oracle.sparse_ffn(lay, x, idx)
    assert np.allclose(np.sum(y_parts, axis=0), y_ref, rtol=1e-12, atol=1e-12)
    # the dense layer the same way, against numpy float64 matmuls
    dense_parts = [oracle.dense_ffn(oracle.neuron_shard(lay, order[g::shards], g == 0), x) for g in range(shards)]
    assert np.allclose(np.sum(dense_parts, axis=0), _dense_np(lay, w, x)[0], rtol=1e-12, atol=1e-12)
    if shards > 1:  # dropping a shard is visible
        assert not np.allclose(np.sum(dense_parts[1:], axis=0), _dense_np(lay, w, x)[0], rtol=1e-6)


def test_predictor_matches_float64_formula():
    lay, w = _np_layer(64, 120, 24, False, "f16", seed=41)
    x = synth.tokens(3, 64, 42).numpy()
    p1 = w["p1"].astype(np.float64)
    p2 = w["p2"].astype(np.float64)
    for t in range(3):
        h, logit, mask = oracle.predict(lay, x[t])
        h_ref = np.maximum(p1 @ x[t].astype(np.float64), 0.0)
        np.testing.assert_allclose(h, h_ref, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(logit, p2 @ h_ref, rtol=1e-12, atol=1e-12)
        assert np.array_equal(mask, (logit > 0.0).astype(np.uint8))


def test_projection_predictor_identity():
    """With P1 = [Q; -Q], P2 = [L, -L]: logit = L (Q x) + b exactly, because
    relu(t) - relu(-t) = t (no ReLU appears in the reference expression)."""
    L = synth.make_layer(96, 150, 32, gated=False, wtype="f32", sparsity=0.8, predictor="projection",
                         seed=5)
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    lay = oracle.Layer(96, 150, 32, w["w_up"], w["w_down"], b_act=w["b_act"], p1=w["p1"], p2=w["p2"],
                       p_bias=w["p_bias"])
    Q = w["p1"][:16].astype(np.float64)
    Lm = w["p2"][:, :16].astype(np.float64)
    for t, x in enumerate(synth.tokens(4, 96, 6).numpy()):
        _, logit, _ = oracle.predict(lay, x)
        np.testing.assert_allclose(logit, Lm @ (Q @ x.astype(np.float64)) + w["p_bias"], rtol=1e-11,
                                   atol=1e-11)


@pytest.mark.parametrize("prefix", [0, 1, 37, 120])
def test_always_on_prefix_in_the_predicted_mask(prefix):
    """Neurons below dense_prefix are in the mask whatever their logit; the
    others follow the float64 formula.  The whole layer as prefix gives the
    all-ones mask, and so the dense FFN, bitwise."""
    lay, w = _np_layer(64, 120, 24, False, "f16", seed=43)
    lay_p = oracle.Layer(64, 120, 24, w["w_up"], w["w_down"], b_act=w["b_act"], b_down=w["b_down"] + 0.25,
                         p1=w["p1"], p2=w["p2"], p_bias=w["p_bias"], threshold=0.0, dense_prefix=prefix)
    p1 = w["p1"].astype(np.float64)
    p2 = w["p2"].astype(np.float64)
    for x in synth.tokens(3, 64, 44).numpy():
        _, logit, mask = oracle.predict(lay_p, x)
        ref = (p2 @ np.maximum(p1 @ x.astype(np.float64), 0.0)) > 0.0
        ref[:prefix] = True
        assert np.array_equal(mask.astype(bool), ref)
        if prefix == 120:
            y = oracle.sparse_ffn(lay_p, x, oracle.compact(mask))
            assert np.array_equal(y, oracle.dense_ffn(lay, x))


def test_predict_union_is_or_of_tokens():
    lay, _ = _np_layer(32, 100, 8, False, "f32", seed=51)
    X = synth.tokens(5, 32, 52).numpy()
    _, union = oracle.predict_union(lay, X)
    ref = np.zeros(100, bool)
    for x in X:
        ref |= oracle.predict(lay, x)[2].astype(bool)
    assert np.array_equal(union.astype(bool), ref)


# --- Q4_0 ----------------------------------------------------------------------

def test_q4_0_roundtrip_exact_on_grid_values():
    rng = np.random.default_rng(61)
    rows, cols = 7, 96
    s = (2.0 ** rng.integers(-6, 3, (rows, cols // 32))).astype(np.float32)
    q = rng.integers(0, 16, (rows, cols)).astype(np.int64)
    q[:, ::32] = 0                                   # each block holds its extreme at code 0
    w = (np.repeat(s, 32, axis=1) * (q - 8)).astype(np.float32)
    blob = oracle.q4_0_quantize(w)
    assert np.array_equal(oracle.dequantize(blob, rows, cols), w.astype(np.float64))


def test_q4_0_layout_and_error_bound():
    rng = np.random.default_rng(62)
    rows, cols = 5, 64
    w = rng.standard_normal((rows, cols)).astype(np.float32)
    blob = oracle.q4_0_quantize(w)
    codes = blob[: rows * cols // 2].reshape(rows, cols // 32, 16)
    scales = blob[rows * cols // 2:].view(np.uint16).reshape(rows, cols // 32).view(np.float16)
    q = np.concatenate([codes & 15, codes >> 4], axis=2).reshape(rows, cols).astype(np.float64)
    deq = np.repeat(scales.astype(np.float64), 32, axis=1) * (q - 8)
    assert np.array_equal(oracle.dequantize(blob, rows, cols), deq)
    for j in range(rows):
        for b in range(cols // 32):
            blk = w[j, 32 * b: 32 * b + 32]
            amax = blk[np.argmax(np.abs(blk))]
            assert scales[j, b] == np.float16(amax / np.float32(-8.0))
            err = np.abs(blk - deq[j, 32 * b: 32 * b + 32])
            sc = abs(float(scales[j, b]))
            # half a step, except the top code 15 which also absorbs w/s in (7.5, 8]
            clamped = q[j, 32 * b: 32 * b + 32] == 15
            bound = np.where(clamped, sc, 0.5 * sc) * (1 + 1e-3) + 1e-7
            assert np.all(err <= bound)


def test_q4_0_hand_worked_block():
    """A block quantised by hand (tests/golden/hand_worked_q4_0.txt): scale
    choice, half-up rounding, the clamp at 15, nibble order and the split
    layout, byte for byte."""
    fields = {}
    for line in open(os.path.join(GOLDEN, "hand_worked_q4_0.txt")):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            fields[k.strip()] = v.split()
    w = np.zeros((1, 32), dtype=np.float32)
    for item in fields["w"]:
        e, v = item.split(":")
        w[0, int(e)] = np.float32(float(v))
    blob = oracle.q4_0_quantize(w)
    assert blob.tobytes() == bytes(int(b, 16) for b in fields["bytes"])
    assert np.array_equal(oracle.dequantize(blob, 1, 32)[0], np.array([float(v) for v in fields["dequant"]]))


def test_q4_0_zero_block():
    blob = oracle.q4_0_quantize(np.zeros((2, 32), np.float32))
    assert np.all(blob[:32] == 0x88) and np.all(blob[32:] == 0)


# --- profiling / hot-first order / stack glue ----------------------------------

def test_hot_first_perm_is_stable_descending_sort():
    rng = np.random.default_rng(71)
    for n in (1, 2, 17, 500):
        counts = rng.integers(0, 6, n).astype(np.int32)
        assert np.array_equal(oracle.hot_first_perm(counts), np.argsort(-counts, kind="stable"))


def test_fire_counts_exact_on_integer_layer():
    L = synth.integer_layer(32, 64, 8, gated=False, wtype="f16", seed=81)
    w = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
    lay = oracle.Layer(32, 64, 8, w["w_up"], w["w_down"], b_act=w["b_act"] + 0.5)
    X = synth.integer_tokens(30, 32, 82).numpy()
    z = X.astype(np.float64) @ w["w_up"].astype(np.float64).T + (w["b_act"] + 0.5)
    assert np.array_equal(oracle.fire_counts(lay, X), (z > 0).sum(0).astype(np.int32))


def test_rms_residual_closed_form():
    rng = np.random.default_rng(91)
    x = rng.standard_normal(300).astype(np.float32)
    y = rng.standard_normal(300)
    out = oracle.rms_residual(x, y)
    v = x.astype(np.float64) + y
    np.testing.assert_allclose(out, v / np.sqrt(np.mean(v * v)), rtol=1e-14)
    assert abs(np.mean(out * out) - 1.0) < 1e-12
    assert np.all(oracle.rms_residual(np.zeros(4, np.float32), np.zeros(4)) == 0)


# --- hand-worked example -------------------------------------------------------

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=", 1)
                vals[k.strip()] = np.array([float(t) for t in v.split()], dtype=np.float64)
    return vals


@pytest.mark.parametrize("act,tag", [(oracle.ACT_RELU, "reglu"), (oracle.ACT_RELU2, "relu2")])
def test_hand_worked_gated_example(act, tag):
    g = _read_golden("hand_worked_reglu.txt")
    d, F, r = 2, 3, 2
    f32 = lambda k, shape: g[k].reshape(shape).astype(np.float32)
    lay = oracle.Layer(d, F, r, f32("w_up", (F, d)), f32("w_down", (F, d)), w_gate=f32("w_gate", (F, d)),
                       b_act=g["b_act"], b_down=g["b_down"], p1=f32("p1", (r, d)), p2=f32("p2", (F, r)),
                       p_bias=g["p_bias"], threshold=float(g["threshold"][0]), act=act)
    x = g["x"].astype(np.float32)
    h, logit, mask = oracle.predict(lay, x)
    assert np.array_equal(h, g["h"]) and np.array_equal(logit, g["logit"])
    idx = oracle.compact(mask)
    assert np.array_equal(idx, g["idx"].astype(np.int32))
    T, _ = oracle.true_mask(lay, x)
    assert np.array_equal(T, np.array([1, 1, 0], dtype=np.uint8))
    assert oracle.recall_precision(mask, T) == (g["recall"][0], g["precision"][0])
    assert np.array_equal(oracle.dense_ffn(lay, x), g["y_dense_" + tag])
    assert np.array_equal(oracle.sparse_ffn(lay, x, idx), g["y_sparse_" + tag])


def test_hand_worked_example():
    g = _read_golden("hand_worked_ffn.txt")
    d, F, r = 3, 4, 2
    lay = oracle.Layer(d, F, r, g["w_up"].reshape(F, d).astype(np.float32),
                       g["w_down"].reshape(F, d).astype(np.float32), b_act=g["b_act"],
                       b_down=g["b_down"], p1=g["p1"].reshape(r, d).astype(np.float32),
                       p2=g["p2"].reshape(F, r).astype(np.float32), p_bias=g["p_bias"],
                       threshold=float(g["threshold"][0]))
    x = g["x"].astype(np.float32)
    h, logit, mask = oracle.predict(lay, x)
    assert np.array_equal(h, g["h"]) and np.array_equal(logit, g["logit"])
    assert np.array_equal(oracle.compact(mask), g["idx"].astype(np.int32))
    assert np.array_equal(oracle.dense_ffn(lay, x), g["y_dense"])
    assert np.array_equal(oracle.sparse_ffn(lay, x, g["idx"].astype(np.int32)), g["y_sparse"])
