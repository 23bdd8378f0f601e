"""Host-side arithmetic of bench.py, on CPU: the algorithmic (needed) bytes that
the roofline divides by, checked against the expected per-token figures worked
out by hand from the configured shapes and densities, and the statistics-only
Q4_0 dequantiser checked against the oracle's."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_predictor_gb300 import synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


# expected active rows at the configured density (n = (1 - sparsity) * d_ff,
# down rows = n) and the resulting needed megabytes per token and layer:
#   predictor (r*d + F*r) * 2 B, n * (R*g + 4) + n * R, x in and y out
@pytest.mark.parametrize("name,n,mb", [
    ("llama7b-reglu-fp16", 1101, 58.0),      # 30.9 predictor + 27.1 FFN
    ("opt30b-relu-fp16-perm", 1434, 114.6),
    ("falcon40b-relu-fp16", 3277, 191.2),
    ("falcon40b-relu-q4_0", 3277, 114.2),
    ("opt175b-relu-fp16-stack12", 2458, 246.7),
])
def test_needed_bytes_at_configured_density(name, n, mb):
    w = synth.WORKLOADS[name]
    pred, ffn = bench.needed_bytes(w, n, n)
    assert (pred + ffn) / 1e6 == pytest.approx(mb, abs=0.15)
    # the predictor term alone: both matrices once, at the predictor element size
    assert pred == (w.rank * w.d_model + w.d_ff * w.rank) * 2


def test_needed_bytes_terms():
    w = synth.WORKLOADS["llama7b-reglu-fp16"]
    # one more predicted neuron adds its gate and up rows plus a 4-byte index;
    # one more non-zero neuron adds its down row; a group of B tokens adds B x/y
    p0, f0 = bench.needed_bytes(w, 100, 50)
    assert bench.needed_bytes(w, 101, 50)[1] - f0 == 2 * 2 * w.d_model + 4
    assert bench.needed_bytes(w, 100, 51)[1] - f0 == 2 * w.d_model
    p4, f4 = bench.needed_bytes(w, 100, 50, batch=4)
    assert p4 == p0 and f4 - f0 == 3 * 2 * 4 * w.d_model


def test_q4_dequant_helper_matches_oracle():
    rows, cols = 7, 96
    blob = oracle.q4_0_quantize(np.random.default_rng(3).standard_normal((rows, cols)).astype(np.float32))
    got = bench.q4_dequant_torch(torch.from_numpy(blob), rows, cols).numpy().astype(np.float64)
    assert np.array_equal(got, oracle.dequantize(blob, rows, cols))


@pytest.mark.parametrize("layers", [1, 3])
def test_reference_arm_prints_one_contract_line(layers, capsys, monkeypatch):
    """The reference arm (the oracle on the host cores) on a small workload:
    one JSON line with the contract's keys, in one or several layers."""
    import argparse
    import json
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    w = synth.Workload("small-stack", 256, 1024, 32, False, "f16", 0.9, 8, layers=layers, predictor="random",
                       seed=7)
    args = argparse.Namespace(gpus=1, steps=2, warmup=3, cpu_seconds=1.0, one_layer=False)
    assert bench.run_reference(args, w) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/layer/token" and line["higher_is_better"] is False
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "us/layer/token", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["cpu_dense"]["value"] > 0
    assert line["config"]["workload"] == "small-stack"


@pytest.mark.parametrize("content,want", [
    (None, None),
    ('{"hbm_gbs": 7012.5, "bf16_tflops": 2100}', 7012.5),
    ('{"hbm_gbs": {"value": 6900, "unit": "GB/s"}}', 6900.0),
    ('{"hbm": {"burst": 7100.0}}', 7100.0),
    ('{"bf16_tflops": 2100}', None),
    ('not json', None),
])
def test_measured_peaks_file(tmp_path, monkeypatch, content, want):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    if content is not None:
        (tmp_path / "MEASURED_PEAKS.json").write_text(content)
    peak, src = bench.measured_peaks()
    if want is None:
        assert (peak, src) == (bench.FALLBACK_HBM_GBS, "fallback")
    else:
        assert (peak, src) == (want, "measured")


def test_committed_traffic_only_for_the_current_kernel_source(tmp_path, monkeypatch):
    """A profile summary's DRAM traffic is used only while its recorded source
    hash matches the kernel sources as they are now; a stale or missing hash,
    or no summary, gives None (the bench line then reports traffic null)."""
    csrc = tmp_path / "activation_sparse_decode_predictor_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["k_layer_b1"]:
        (csrc / f).write_text(f"// {f}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("k_layer_b1")
    assert len(h) == 16
    prof = tmp_path / "profiles" / "k_layer_b1_wl.md"
    assert bench.committed_traffic("k_layer_b1", "wl") is None
    prof.write_text(f"text\ntraffic_bytes_per_launch: 213.1e6\nkernel_source_sha: {h}\n")
    assert bench.committed_traffic("k_layer_b1", "wl") == 213.1e6
    prof.write_text("traffic_bytes_per_launch: 213.1e6\nkernel_source_sha: 0123456789abcdef\n")
    assert bench.committed_traffic("k_layer_b1", "wl") is None
    prof.write_text(f"traffic_bytes_per_launch: 213.1e6\nkernel_source_sha: {h}\n")
    (csrc / "layer_fused.cu").write_text("// changed\n")  # the kernel changed after the capture
    assert bench.committed_traffic("k_layer_b1", "wl") is None
