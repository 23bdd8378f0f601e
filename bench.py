"""Benchmark: microseconds per sparse-FFN layer per decode token, and achieved
HBM GB/s of the dominant kernel against the HBM roofline.

One step = the whole hot path (predictor GEMVs, threshold + union, active-index
compaction, gather up/gate projections, activation, scatter-accumulate down
projection) for every decode token of one batch of synthetic tokens (256 for
the default workload), token by token at batch 1, each token on the next of
R rotating copies of the layer so the step's weight traffic (R x the layer)
is far larger than L2, as consecutive layers of a real model would be.

Default workload: the ReLU-LLaMA-7B-shaped gated FFN layer (d_model 4096,
d_ff 11008, fp16 weights, predictor rank 1024, ~90% Zipf-biased sparsity).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun each rank runs its own token stream on its own GPU (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
--impl reference times the CPU oracle on this machine's host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from activation_sparse_decode_predictor_gb300 import binding as B  # noqa: E402
from activation_sparse_decode_predictor_gb300 import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["sparse_ffn.cu", "common.cuh", "internal.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama7b-reglu-fp16", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--replicas", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU oracle sample")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="decode tokens per step (default: the workload's)")
    ap.add_argument("--quick", action="store_true", help="main timed step only (for profiling runs)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:  # noqa: BLE001
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "activation_sparse_decode_predictor_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload):
    """DRAM bytes per launch of the sparse-FFN kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"k_sparse_b1_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    if m and s and s.group(1) == kernel_source_hash():
        return float(m.group(1))
    return None


class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:  # noqa: BLE001
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------------------------ workload
def needed_bytes(w, n_pred, n_down):
    """Algorithmic bytes of one token through one layer: predictor weights,
    the predicted rows of the up/gate projections (+4 B of index each), the
    down rows of neurons whose activation is non-zero, x in and y out."""
    s_p = 4 if w.wtype == "f32" else 2
    R = {"f32": 4 * w.d_model, "f16": 2 * w.d_model, "q4_0": w.d_model // 32 * 18}[w.wtype]
    g = 2 if w.gated else 1
    pred = (w.rank * w.d_model + w.d_ff * w.rank) * s_p
    ffn = n_pred * (R * g + 4) + n_down * R + w.batch * w.d_model * 4 * 2
    return pred, ffn


def setup_ours(w, replicas, dev):
    torch.cuda.set_device(dev)
    L0 = synth.workload_layer(w, 0, device=f"cuda:{dev}")
    reps = []
    for k in range(replicas):
        Lk = {key: (v.clone() if isinstance(v, torch.Tensor) else v) for key, v in L0.items()}
        reps.append((Lk, B.Layer.from_dict(Lk)))
    X = synth.workload_tokens(w, device=f"cuda:{dev}")
    return L0, reps, X


def active_stats(w, L0, layer, X, ws):
    """Per token: predicted active count, the count with non-zero activation,
    recall and precision of the predictor against the true ReLU mask.  Uses
    the library for the prediction and torch only to count."""
    T = X.shape[0]
    F = w.d_ff
    idx = torch.zeros(T, F, dtype=torch.int32, device=X.device)
    n = torch.zeros(T, dtype=torch.int32, device=X.device)
    for t in range(T):
        B.pi_predict(layer, X[t], idx[t], n[t:t + 1], ws=ws)
    torch.cuda.synchronize()
    w_act = (L0["w_gate"] if w.gated else L0["w_up"]).float()
    z = X @ w_act.T + L0["b_act"]
    true = z > 0
    n_pred, n_down, rec, prec = [], [], [], []
    for t in range(T):
        nt = int(n[t])
        sel = idx[t, :nt].long()
        pm = torch.zeros(F, dtype=torch.bool, device=X.device)
        pm[sel] = True
        n_pred.append(nt)
        n_down.append(int(true[t, sel].sum()))
        inter = int((pm & true[t]).sum())
        rec.append(inter / max(1, int(true[t].sum())))
        prec.append(inter / max(1, nt))
    return idx, n, np.array(n_pred), np.array(n_down), float(np.mean(rec)), float(np.mean(prec)), \
        float(true.float().mean())


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm (first calls set kernel attributes outside capture)
        torch.cuda.synchronize()
        g.capture_begin()
        fn()
        g.capture_end()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps, warmup, stream, barrier=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if barrier:
            barrier()
    return e0.elapsed_time(e1)  # ms


# ------------------------------------------------------------------------------------ CPU oracle
def oracle_sample(w, L0_host, X_host, budget_s):
    """Time the oracle's full per-token path (predictor, compaction, sparse
    FFN) on as many tokens as fit the budget; returns (us per token, tokens)."""
    import oracle
    H = L0_host
    olay = oracle.Layer(w.d_model, w.d_ff, w.rank, H["w_up"], H["w_down"], w_gate=H["w_gate"], b_act=H["b_act"],
                        b_down=H["b_down"], p1=H["p1"], p2=H["p2"], p_bias=H["p_bias"], threshold=H["threshold"])
    t0 = time.perf_counter()
    done = 0
    while done < X_host.shape[0]:
        _, _, m = oracle.predict(olay, X_host[done])
        idx = oracle.compact(m)
        oracle.sparse_ffn(olay, X_host[done], idx)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return (time.perf_counter() - t0) / done * 1e6, done


def host_layer(L0):
    H = {k: (v.detach().cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in L0.items()}
    return H


# ------------------------------------------------------------------------------------ arms
def run_reference(args, w):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    L0 = synth.workload_layer(w, 0, device="cpu")
    H = host_layer(L0)
    X = synth.workload_tokens(w, device="cpu").numpy()
    per_step = []
    tokens_per_sample = None
    budget = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for s in range(args.warmup + args.steps):
        us, ntok = oracle_sample(w, H, X[(s * 7) % X.shape[0]:], budget)
        if s >= args.warmup:
            per_step.append(us)
            tokens_per_sample = ntok
    value = float(np.median(per_step))
    line = {"impl": "reference", "metric": "us_per_ffn_layer_per_token", "value": value,
            "unit": "us/layer/token", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": value * w.tokens / 1000.0, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "d_model": w.d_model, "d_ff": w.d_ff, "rank": w.rank,
                       "gated": w.gated, "weights": w.wtype, "batch": w.batch, "sparsity": w.sparsity},
            "cpu_baseline": {"value": value, "unit": "us/layer/token", "cores": 1, "kind": "oracle",
                             "sample": f"{tokens_per_sample} token(s) per step through one layer (predictor, "
                                       "compaction, sparse FFN), single-threaded C, fp64"},
            "e2e": {"value": value, "unit": "us/layer/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_ours(args, w):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        barrier = dist.barrier
    else:
        barrier = None
    dev = local
    torch.cuda.set_device(dev)
    B.lib()
    L0, reps, X = setup_ours(w, args.replicas, dev)
    if args.tokens:
        X = X[:args.tokens].contiguous()
    T = X.shape[0]
    d = w.d_model
    stream = torch.cuda.Stream()
    ws = B.workspace(B.pi_workspace_bytes(reps[0][1], 1), X.device)
    Y = torch.zeros(T, d, dtype=torch.float32, device=X.device)

    # statistics of the active sets (outside any timed region)
    idx_all, n_all, n_pred, n_down, recall, precision, true_density = active_stats(w, L0, reps[0][1], X, ws)
    pred_b, ffn_b = needed_bytes(w, n_pred, n_down)
    bytes_tok = pred_b + ffn_b                       # per token, arrays
    mean_bytes = float(np.mean(bytes_tok))

    def step():
        for t in range(T):
            B.pi_ffn_layer(reps[t % len(reps)][1], X[t], Y[t], ws=ws)

    g_step = capture(step, stream)
    with Clocks(dev) as clk:
        ms = time_graph(g_step, args.steps, args.warmup, stream, barrier)
    ms_step = ms / args.steps
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([ms_step], device=X.device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_step = float(tt.item())
    us_tok = ms_step * 1000.0 / (T * world)          # whole job: all ranks' tokens in the max time

    peak, peak_src = measured_peaks()
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token",
                              "quick": True, "workload": w.name, "tokens_per_step": T,
                              "layer_gbs": mean_bytes / (us_tok * world * 1e-6) / 1e9,
                              "device_status": B.pi_sync_status(ws)}))
        return 0

    # the dominant kernel alone: the sparse FFN on the predicted lists (same rotation)
    def sparse_only():
        for t in range(T):
            B.pi_sparse_ffn(reps[t % len(reps)][1], X[t], idx_all[t], n_all[t:t + 1], Y[t], ws=ws)

    def predict_only():
        for t in range(T):
            B.pi_predict(reps[t % len(reps)][1], X[t], idx_all[t], n_all[t:t + 1], ws=ws)

    ksteps = max(10, args.steps // 4)
    g_sp = capture(sparse_only, stream)
    ms_sp = time_graph(g_sp, ksteps, args.warmup, stream) / ksteps
    g_pr = capture(predict_only, stream)
    ms_pr = time_graph(g_pr, ksteps, args.warmup, stream) / ksteps
    us_sp = ms_sp * 1000.0 / T
    us_pr = ms_pr * 1000.0 / T
    ffn_gbs = float(np.mean(ffn_b)) / (us_sp * 1e-6) / 1e9
    pred_gbs = float(pred_b) / (us_pr * 1e-6) / 1e9
    layer_gbs = mean_bytes / (us_tok * world * 1e-6) / 1e9

    # end to end through the public API: pinned host tokens in, outputs back
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(T, d, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(X)
    e2e_steps = max(3, args.steps // 20)
    with torch.cuda.stream(stream):
        def e2e_step():
            Xd.copy_(Xh, non_blocking=True)
            for t in range(T):
                B.pi_ffn_layer(reps[t % len(reps)][1], Xd[t], Y[t], ws=ws)
            Yh.copy_(Y, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
    us_e2e = e0.elapsed_time(e1) / e2e_steps * 1000.0 / T
    st = B.pi_sync_status(ws)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        us_cpu, ntok = oracle_sample(w, host_layer(L0), X.cpu().numpy(), args.cpu_seconds)
        cpu = {"value": us_cpu, "unit": "us/layer/token", "cores": 1, "kind": "oracle",
               "sample": f"first {ntok} of {T} tokens through one layer (predictor, compaction, sparse FFN), "
                         "single-threaded C oracle, fp64"}

    if rank == 0:
        line = {
            "metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if w.wtype == "f16" else w.wtype,
            "data": "synthetic",
            "config": {"workload": w.name, "d_model": d, "d_ff": w.d_ff, "rank": w.rank, "gated": w.gated,
                       "weights": w.wtype, "accumulate": "f32", "batch": w.batch, "tokens_per_step": T,
                       "sparsity": w.sparsity, "layer_replicas": len(reps),
                       "l2": f"inputs larger than L2: {len(reps)} rotating layer copies, "
                             f"{len(reps) * mean_bytes / 1e6:.0f} MB needed bytes per rotation",
                       "n_active_mean": float(np.mean(n_pred)), "n_nonzero_mean": float(np.mean(n_down)),
                       "true_density": true_density, "predictor_recall": recall, "predictor_precision": precision,
                       "needed_bytes_per_token": mean_bytes, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "k_sparse_b1 (pi_sparse_ffn)", "achieved": ffn_gbs,
                         "peak": peak, "unit": "GB/s", "frac": ffn_gbs / peak,
                         "traffic": committed_traffic(w.name), "peak_source": peak_src},
            "kernels": {"predict_us": us_pr, "predict_gbs": pred_gbs, "predict_frac": pred_gbs / peak,
                        "sparse_ffn_us": us_sp, "sparse_ffn_gbs": ffn_gbs, "layer_gbs": layer_gbs,
                        "layer_frac": layer_gbs / peak},
            "e2e": {"value": us_e2e, "unit": "us/layer/token", "h2d_bytes_per_step": int(Xh.numel() * 4),
                    "d2h_bytes_per_step": int(Yh.numel() * 4), "path": "pi_ffn_layer per token, direct calls"},
            "gpu_launches": 3 * T * args.steps,
            "clocks": clk.summary(),
            "device_status": st,
        }
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
