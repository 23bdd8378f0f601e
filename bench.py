"""Benchmark: microseconds per sparse-FFN layer per decode token, and achieved
HBM GB/s of the dominant kernel against the HBM roofline.

One step = the whole hot path (predictor GEMVs, threshold + union, active-index
compaction, gather up/gate projections, activation, scatter-accumulate down
projection) for every decode token of one batch of synthetic tokens.

Default workload: the OPT-175B-shaped stack of 12 non-gated ReLU FFN layers
(d_model 12288, d_ff 49152, fp16 weights, predictor rank 1024, ~95%
Zipf-biased sparsity), 128 decode tokens per step, each token through all 12
distinct layers with the residual + RMS rescale between them, timed end to
end; its 29 GB of weights are far larger than L2.  Single-layer workloads run
each token on the next of R rotating copies of the layer, so a step's weight
traffic (R x the layer) is far larger than L2, as consecutive layers of a real
model would be.

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
# sources of the kernel each roofline line describes (a committed ncu traffic
# figure counts only while its recorded hash matches these files)
KERNEL_SOURCES = {
    "k_layer_b1": ["layer_fused.cu", "ffn_rows.cuh", "common.cuh", "internal.h"],
    "k_union": ["union_mma.cu", "ffn_rows.cuh", "common.cuh", "internal.h"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="opt175b-relu-fp16-stack12", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--replicas", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU oracle sample")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="decode tokens per step (default: the workload's)")
    ap.add_argument("--quick", action="store_true", help="main timed step only (for profiling runs)")
    ap.add_argument("--one-layer", action="store_true",
                    help="multi-layer workloads: time one layer on rotating copies instead of the stack")
    ap.add_argument("--batch", type=int, default=0,
                    help="tokens decoded together through the union path (default: the workload's)")
    ap.add_argument("--dense-prefix", default="0",
                    help="always-on prefix of the hot-first order: a neuron count, or 'auto' for the neurons that "
                         "fired on more than half of the profiling tokens (implies the hot-first order)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------ helpers
def measured_peaks():
    """HBM copy bandwidth (GB/s) from MEASURED_PEAKS.json when present: a
    number under hbm_gbs (or hbm_GBps / hbm), or an object holding one under
    value / burst / median / mean; else the fallback figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = next((v[q] for q in ("value", "burst", "median", "mean") if q in v), None)
                if isinstance(v, (int, float)) and v > 0:
                    return float(v), "measured"
        except Exception:  # noqa: BLE001 -- an unreadable file means the fallback
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "activation_sparse_decode_predictor_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, tag):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    profiles/<kernel>_<tag>.md, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{tag}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    if m and s and s.group(1) == kernel_source_hash(kernel):
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


def job_time(ms_step, world, device):
    """Time per step of the whole job: the slowest rank's (every rank calls this)."""
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([float(ms_step)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())
    return ms_step


def whole_job_us_per_token(ms_step, tokens_per_rank, world):
    """All ranks' tokens processed in the slowest rank's time (weak scaling)."""
    return ms_step * 1000.0 / (tokens_per_rank * world)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------------------------ workload
def needed_bytes(w, n_pred, n_down, batch=1, prefix=0):
    """Algorithmic bytes of one group of `batch` tokens through one layer:
    predictor weights (read once for the group; no P2 rows for an always-on
    prefix), the predicted (union) rows of the up/gate projections (+4 B of
    index each; the prefix rows are part of that list), the down rows of
    neurons whose activation is non-zero for at least one token, x in and y
    out."""
    s_p = 4 if w.wtype == "f32" else 2
    R = {"f32": 4 * w.d_model, "f16": 2 * w.d_model, "q4_0": w.d_model // 32 * 18}[w.wtype]
    g = 2 if w.gated else 1
    pred = (w.rank * w.d_model + (w.d_ff - prefix) * w.rank) * s_p
    ffn = n_pred * (R * g + 4) + n_down * R + batch * w.d_model * 4 * 2
    return pred, ffn


def q4_dequant_torch(blob, rows, cols):
    """Q4_0 split blob -> fp32 matrix with plain torch ops (statistics only)."""
    codes = blob[: rows * cols // 2].view(rows, cols // 32, 16)
    scales = blob[rows * cols // 2:].view(torch.float16).view(rows, cols // 32, 1).float()
    q = torch.cat([codes & 15, codes >> 4], dim=2).float() - 8.0
    return (q * scales).reshape(rows, cols)


def top_share(counts, frac=0.26):
    """Share of all firings carried by the `frac` most frequently firing
    neurons (the power-law locality statistic of the pages)."""
    c = np.sort(np.asarray(counts, dtype=np.float64))[::-1]
    k = max(1, int(round(frac * c.size)))
    return float(c[:k].sum() / max(1.0, c.sum()))


def hot_first(w, L0, dev, prefix="0"):
    """Offline profiling pass: w.profile_tokens synthetic tokens (a token stream
    of their own; 1024 when the workload names none) through pi_fire_counts on
    the layer as generated, the hot-first order from pi_hot_first_perm, then
    every per-neuron array (rows of w_up / w_gate / w_down / p2, entries of
    b_act / p_bias) permuted with pi_permute_rows.  An always-on prefix is set
    from `prefix` (a count, or 'auto': the neurons that fired on more than half
    of the profiling tokens).  Returns the permuted layer and statistics of
    the order."""
    F = w.d_ff
    lay = B.Layer.from_dict(L0)
    T = w.profile_tokens or 1024
    Xp = synth.workload_tokens(w, n=T, device=f"cuda:{dev}", stream=1)
    counts = torch.zeros(F, dtype=torch.int32, device=Xp.device)
    B.pi_fire_counts(lay, Xp, counts)
    c = counts.cpu().numpy()
    perm = B.pi_hot_first_perm(c)
    perm_d = torch.from_numpy(perm).to(Xp.device)
    out = dict(L0)
    for k in ("w_up", "w_gate", "w_down", "p2", "b_act", "p_bias"):
        if L0.get(k) is not None:
            out[k] = B.pi_permute_rows(L0[k], perm_d)
    torch.cuda.synchronize()
    cs = c[perm].astype(np.float64)
    H = int(np.sum(c > T // 2)) if prefix == "auto" else int(prefix)
    out["dense_prefix"] = H
    stats = {"profile_tokens": int(T),
             "first_quarter_share_profile": float(cs[: F // 4].sum() / max(1.0, cs.sum())),
             "dense_prefix": H}
    return out, perm, stats


def setup_ours(w, replicas, dev, prefix="0"):
    torch.cuda.set_device(dev)
    L0 = synth.workload_layer(w, 0, device=f"cuda:{dev}")
    perm_stats = None
    if w.permute or prefix != "0":
        L0, _, perm_stats = hot_first(w, L0, dev, prefix)
    if w.wtype == "q4_0":
        # the generator returns fp16 matrices; store them as Q4_0 with the library's quantiser
        for k in ("w_up", "w_gate", "w_down"):
            if L0[k] is not None:
                L0[k] = B.pi_quantize_q4_0(L0[k])
        L0["wtype_code"] = B.PI_Q4_0
        torch.cuda.synchronize()
    reps = []
    for k in range(replicas):
        Lk = {key: (v.clone() if isinstance(v, torch.Tensor) else v) for key, v in L0.items()}
        reps.append((Lk, B.Layer.from_dict(Lk)))
    # consecutive calls run consecutive copies, as a decode step runs consecutive
    # layers: each copy names the one after it (a scheduling hint)
    for k in range(replicas):
        reps[k][1].set_next(reps[(k + 1) % replicas][1])
    X = synth.workload_tokens(w, device=f"cuda:{dev}")
    return L0, reps, X, perm_stats


def active_stats(w, L0, layer, X, ws, ws1, batch):
    """Per group of `batch` tokens: predicted (union) active count and the count
    of those rows with a non-zero activation for some token of the group; per
    token: recall and precision of the predictor against the true ReLU mask,
    and the true mask itself.  Uses the library for the predictions and torch
    only to count."""
    T = X.shape[0]
    G = T // batch
    F = w.d_ff
    idx = torch.zeros(G, F, dtype=torch.int32, device=X.device)
    n = torch.zeros(G, dtype=torch.int32, device=X.device)
    for gi in range(G):
        xg = X[gi * batch:(gi + 1) * batch] if batch > 1 else X[gi]
        B.pi_predict(layer, xg, idx[gi], n[gi:gi + 1], ws=ws)
    idx1 = torch.zeros(F, dtype=torch.int32, device=X.device)
    n1 = torch.zeros(T, dtype=torch.int32, device=X.device)
    own = torch.zeros(T, F, dtype=torch.bool, device=X.device)
    for t in range(T):
        B.pi_predict(layer, X[t], idx1, n1[t:t + 1], ws=ws1)
        own[t, idx1[: int(n1[t])].long()] = True
    torch.cuda.synchronize()
    w_act = L0["w_gate"] if w.gated else L0["w_up"]
    w_act = q4_dequant_torch(w_act, F, w.d_model) if w.wtype == "q4_0" else w_act.float()
    z = X @ w_act.T + L0["b_act"]
    true = z > 0
    n_pred, n_down = [], []
    for gi in range(G):
        nt = int(n[gi])
        sel = idx[gi, :nt].long()
        n_pred.append(nt)
        n_down.append(int(true[gi * batch:(gi + 1) * batch][:, sel].any(dim=0).sum()))
    inter = (own & true).sum(dim=1).float()
    rec = float((inter / true.sum(dim=1).clamp(min=1)).mean())
    prec = float((inter / own.sum(dim=1).clamp(min=1)).mean())
    return dict(idx=idx, n=n, n_pred=np.array(n_pred), n_down=np.array(n_down), recall=rec, precision=prec,
                true_density=float(true.float().mean()), true=true)


def true_lists(true):
    """Ascending true-active lists [T, F] (int32, device) and their lengths [T]."""
    T, F = true.shape
    idx = torch.zeros(T, F, dtype=torch.int32, device=true.device)
    n = true.sum(dim=1).to(torch.int32)
    for t in range(T):
        nz = torch.nonzero(true[t]).flatten().to(torch.int32)
        idx[t, : nz.numel()] = nz
    return idx, n


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


def roofline_obj(kernel, achieved, peak, peak_src, traffic, **extra):
    r = {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src}
    r.update(extra)
    return r


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


def host_layer(L0, w=None):
    """Host copy of a layer for the oracle; a Q4_0 workload's fp16 matrices are
    quantised by the oracle's own quantiser."""
    H = {k: (v.detach().cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in L0.items()}
    if w is not None and w.wtype == "q4_0":
        import oracle
        for k in ("w_up", "w_gate", "w_down"):
            if H[k] is not None and H[k].dtype != np.uint8:
                H[k] = oracle.q4_0_quantize(H[k].astype(np.float32))
    return H


def oracle_stack_sample(w, olays, X_host, budget_s):
    """Time the oracle through every layer of a stack (predictor, compaction,
    sparse FFN, residual + rescale) on as many tokens as fit the budget;
    returns (us per layer per token, tokens)."""
    import oracle
    t0 = time.perf_counter()
    done = 0
    while done < X_host.shape[0] and (done == 0 or time.perf_counter() - t0 < budget_s):
        xo = X_host[done]
        for ol in olays:
            _, _, m = oracle.predict(ol, xo)
            yo = oracle.sparse_ffn(ol, xo, oracle.compact(m))
            xo = oracle.rms_residual(xo, yo).astype(np.float32)
        done += 1
    return (time.perf_counter() - t0) / (done * len(olays)) * 1e6, done


def oracle_dense_us(olay, x):
    """Context for the reference arm: the oracle's dense FFN (every neuron) on
    one token, microseconds."""
    import oracle
    t0 = time.perf_counter()
    oracle.dense_ffn(olay, x)
    return (time.perf_counter() - t0) * 1e6


def oracle_layer(w, H):
    import oracle
    return oracle.Layer(w.d_model, w.d_ff, w.rank, H["w_up"], H["w_down"], w_gate=H["w_gate"], b_act=H["b_act"],
                        b_down=H["b_down"], p1=H["p1"], p2=H["p2"], p_bias=H["p_bias"], threshold=H["threshold"])


# ------------------------------------------------------------------------------------ arms
def reference_layers(w):
    """The workload's layers as host arrays for the oracle, drawn by the same
    seeded generator as the GPU arm (on the GPU when there is one, so both arms
    see the same numbers).  A hot-first neuron order is not applied here: it
    only renames neurons, and the oracle's work per token does not depend on
    the order."""
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    out = []
    for l in range(w.layers):
        L = synth.workload_layer(w, l, device=dev)
        out.append(oracle_layer(w, host_layer(L, w)))
        del L
    X = synth.workload_tokens(w, device=dev).cpu().numpy()
    return out, X


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, single-threaded, on a
    bounded sample of the same workload per step.  ms_per_step is the wall time
    of the sample each step actually ran (tokens_per_step of them)."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    stack = w.layers > 1 and not args.one_layer
    if not stack and w.layers > 1:
        w = synth.Workload(**{**w.__dict__, "layers": 1})
    olays, X = reference_layers(w)
    budget = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    per_step, wall_ms, ntoks = [], [], []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if stack:
            us, ntok = oracle_stack_sample(w, olays, X[(s * 7) % X.shape[0]:], budget)
        else:
            us, ntok = oracle_sample_layer(olays[0], X[(s * 7) % X.shape[0]:], budget)
        if s >= args.warmup:
            per_step.append(us)
            wall_ms.append((time.perf_counter() - t0) * 1000.0)
            ntoks.append(ntok)
    value = float(np.median(per_step))
    what = (f"token(s) per step through all {w.layers} layers (predictor, compaction, sparse FFN, residual + "
            "rescale)" if stack else "token(s) per step through one layer (predictor, compaction, sparse FFN)")
    line = {"impl": "reference", "metric": "us_per_ffn_layer_per_token", "value": value,
            "unit": "us/layer/token", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": float(np.median(wall_ms)), "tokens_per_step": int(np.median(ntoks)),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {**workload_config(w, 1, stack), "hot_first_order": False},
            "cpu_baseline": {"value": value, "unit": "us/layer/token", "cores": 1, "kind": "oracle",
                             "sample": f"{int(np.median(ntoks))} {what}, single-threaded C, fp64"},
            "e2e": {"value": value, "unit": "us/layer/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "cpu_dense": {"value": oracle_dense_us(olays[0], X[0]), "unit": "us/layer/token",
                          "sample": "1 token through the first layer, every neuron, single-threaded C oracle, fp64"}}
    print(json.dumps(line))
    return 0


def oracle_sample_layer(olay, X_host, budget_s):
    import oracle
    t0 = time.perf_counter()
    done = 0
    while done < X_host.shape[0] and (done == 0 or time.perf_counter() - t0 < budget_s):
        _, _, m = oracle.predict(olay, X_host[done])
        oracle.sparse_ffn(olay, X_host[done], oracle.compact(m))
        done += 1
    return (time.perf_counter() - t0) / done * 1e6, done


def workload_config(w, batch, stack):
    c = {"workload": w.name, "d_model": w.d_model, "d_ff": w.d_ff, "rank": w.rank, "gated": w.gated,
         "weights": w.wtype, "accumulate": "f32", "batch": batch, "sparsity": w.sparsity,
         "hot_first_order": bool(w.permute)}
    if stack:
        c["layers"] = w.layers
    return c


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
    L0, reps, X, perm_stats = setup_ours(w, args.replicas, dev, args.dense_prefix)
    H = int(L0.get("dense_prefix", 0))
    if args.tokens:
        X = X[:args.tokens].contiguous()
    bsz = args.batch or w.batch
    T = X.shape[0] // bsz * bsz
    X = X[:T].contiguous()
    G = T // bsz                                     # groups of bsz tokens decoded together
    d = w.d_model
    stream = torch.cuda.Stream()
    ws = B.workspace(B.pi_workspace_bytes(reps[0][1], bsz), X.device)
    ws1 = ws if bsz == 1 else B.workspace(B.pi_workspace_bytes(reps[0][1], 1), X.device)
    Y = torch.zeros(T, d, dtype=torch.float32, device=X.device)
    Xg = [X[gi * bsz:(gi + 1) * bsz] if bsz > 1 else X[gi] for gi in range(G)]
    Yg = [Y[gi * bsz:(gi + 1) * bsz] if bsz > 1 else Y[gi] for gi in range(G)]

    # statistics of the active sets (outside any timed region)
    S = active_stats(w, L0, reps[0][1], X, ws, ws1, bsz)
    pred_b, ffn_b = needed_bytes(w, S["n_pred"], S["n_down"], bsz, H)
    bytes_grp = pred_b + ffn_b                       # per group, arrays
    mean_bytes = float(np.mean(bytes_grp)) / bsz     # per token
    fire = S["true"].sum(dim=0).cpu().numpy()

    def step():
        for gi in range(G):
            B.pi_ffn_layer(reps[gi % len(reps)][1], Xg[gi], Yg[gi], ws=ws)

    g_step = capture(step, stream)
    with Clocks(dev) as clk:
        ms = time_graph(g_step, args.steps, args.warmup, stream, barrier)
    ms_step = job_time(ms / args.steps, world, X.device)
    us_tok = whole_job_us_per_token(ms_step, T, world)

    peak, peak_src = measured_peaks()
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token",
                              "quick": True, "workload": w.name, "tokens_per_step": T,
                              "layer_gbs": mean_bytes / (us_tok * world * 1e-6) / 1e9,
                              "device_status": B.pi_sync_status(ws)}))
        return 0

    # the sparse FFN alone on the predicted lists (same rotation), and the predictor alone
    idx_all, n_all = S["idx"], S["n"]

    def sparse_only():
        for gi in range(G):
            B.pi_sparse_ffn(reps[gi % len(reps)][1], Xg[gi], idx_all[gi], n_all[gi:gi + 1], Yg[gi], ws=ws)

    def predict_only():
        for gi in range(G):
            B.pi_predict(reps[gi % len(reps)][1], Xg[gi], idx_all[gi], n_all[gi:gi + 1], ws=ws)

    ksteps = max(10, args.steps // 4)
    g_sp = capture(sparse_only, stream)
    ms_sp = time_graph(g_sp, ksteps, args.warmup, stream) / ksteps
    g_pr = capture(predict_only, stream)
    ms_pr = time_graph(g_pr, ksteps, args.warmup, stream) / ksteps
    us_sp = ms_sp * 1000.0 / G                      # per group
    us_pr = ms_pr * 1000.0 / G
    ffn_gbs = float(np.mean(ffn_b)) / (us_sp * 1e-6) / 1e9
    pred_gbs = float(pred_b) / (us_pr * 1e-6) / 1e9
    layer_gbs = mean_bytes / (us_tok * world * 1e-6) / 1e9
    kernels = {"per": "token" if bsz == 1 else f"group of {bsz} tokens",
               "predict_us": us_pr, "predict_gbs": pred_gbs, "predict_frac": pred_gbs / peak,
               "sparse_ffn_us": us_sp, "sparse_ffn_gbs": ffn_gbs, "sparse_ffn_frac": ffn_gbs / peak,
               "layer_gbs": layer_gbs, "layer_frac": layer_gbs / peak}

    if bsz == 1:
        # measurement mode (i): the sparse FFN alone on the TRUE active lists, at
        # exactly the generator's sparsity (kernel roofline without the predictor)
        tidx, tn = true_lists(S["true"])

        def sparse_true():
            for t in range(T):
                B.pi_sparse_ffn(reps[t % len(reps)][1], X[t], tidx[t], tn[t:t + 1], Y[t], ws=ws)

        g_tr = capture(sparse_true, stream)
        ms_tr = time_graph(g_tr, ksteps, args.warmup, stream) / ksteps
        us_tr = ms_tr * 1000.0 / T
        n_true = tn.cpu().numpy()
        tr_b = float(np.mean(needed_bytes(w, n_true, n_true, 1)[1]))
        kernels.update({"true_mask_sparse_ffn_us": us_tr, "true_mask_sparse_ffn_gbs": tr_b / (us_tr * 1e-6) / 1e9,
                        "true_mask_sparse_ffn_frac": tr_b / (us_tr * 1e-6) / 1e9 / peak,
                        "true_mask_n_mean": float(np.mean(n_true))})

    # end to end through the public API: pinned host tokens in, outputs back
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(T, d, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(X)
    e2e_steps = max(3, args.steps // 4)
    with torch.cuda.stream(stream):
        Xdg = [Xd[gi * bsz:(gi + 1) * bsz] if bsz > 1 else Xd[gi] for gi in range(G)]

        def e2e_step():
            Xd.copy_(Xh, non_blocking=True)
            for gi in range(G):
                B.pi_ffn_layer(reps[gi % len(reps)][1], Xdg[gi], Yg[gi], ws=ws)
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
        H0 = host_layer(L0) if w.wtype != "q4_0" else host_layer(synth.workload_layer(w, 0, device=X.device), w)
        us_cpu, ntok = oracle_sample(w, H0, X.cpu().numpy(), args.cpu_seconds)
        cpu = {"value": us_cpu, "unit": "us/layer/token", "cores": 1, "kind": "oracle",
               "sample": f"first {ntok} of {T} tokens through one layer (predictor, compaction, sparse FFN), "
                         "single-threaded C oracle, fp64"}

    if bsz == 1:
        # one kernel per token and layer: the whole step is k_layer_b1 back to back
        launches_per_group = 1
        roofline = roofline_obj("k_layer_b1 (pi_ffn_layer)", layer_gbs, peak, peak_src,
                                committed_traffic("k_layer_b1", w.name))
        roofline_layer = None
    else:
        # predictor (2 kernels) + k_union_prep + k_union_up + k_union_down per group
        launches_per_group = 8
        roofline = roofline_obj("k_union_prep + k_union_up + k_union_down (pi_sparse_ffn)", ffn_gbs, peak, peak_src,
                                committed_traffic("k_union", f"{w.name}_b{bsz}"))
        # the whole layer, predictor bytes included, over the timed step
        roofline_layer = roofline_obj("pi_ffn_layer (predictor + compaction + union FFN)", layer_gbs, peak, peak_src,
                                      None)

    if rank == 0:
        cfg = workload_config(w, bsz, False)
        cfg["hot_first_order"] = bool(perm_stats)
        cfg.update({"dense_prefix": H, "tokens_per_step": T, "layer_replicas": len(reps),
                    "l2": f"inputs larger than L2: {len(reps)} rotating layer copies, "
                          f"{len(reps) * mean_bytes / 1e6:.0f} MB needed bytes per rotation",
                    "n_active_mean": float(np.mean(S["n_pred"])), "n_nonzero_mean": float(np.mean(S["n_down"])),
                    "true_density": S["true_density"], "predictor_recall": S["recall"],
                    "predictor_precision": S["precision"], "top26_firing_share": top_share(fire),
                    "needed_bytes_per_token": mean_bytes, "parallelism": f"replicas x{world}"})
        if perm_stats:
            cfg["hot_first"] = perm_stats
            cfg["hot_first"]["first_quarter_share_decode"] = float(fire[: w.d_ff // 4].sum() / max(1, fire.sum()))
        line = {
            "metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if w.wtype == "f16" else w.wtype,
            "data": "synthetic", "config": cfg, "roofline": roofline, "kernels": kernels,
            "e2e": {"value": us_e2e, "unit": "us/layer/token", "h2d_bytes_per_step": int(Xh.numel() * 4),
                    "d2h_bytes_per_step": int(Yh.numel() * 4), "path": "pi_ffn_layer per group, direct calls"},
            "gpu_launches": launches_per_group * G * args.steps,
            "clocks": clk.summary(),
            "device_status": st,
        }
        if roofline_layer:
            line["roofline_layer"] = roofline_layer
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_stack(args, w):
    """Workloads of several layers (the OPT-175B-shaped stack): each token goes
    through `w.layers` distinct layers, each layer's output plus its input
    rescaled into the next layer's input, and the whole token is timed end to
    end.  Layer 0 runs pi_ffn_layer on the token; every later layer runs
    pi_ffn_layer_chain, whose kernel applies the glue to the previous layer's
    input and output itself; one pi_rms_residual finishes the token.  Metric:
    us per layer per token (step time / tokens / layers).  The roofline's
    dominant kernel, k_layer_b1, is also timed alone: the same layer calls back
    to back on the recorded inputs of every layer."""
    world, rank, local = dist_env()
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        barrier = dist.barrier
    dev = local
    torch.cuda.set_device(dev)
    B.lib()
    nl = w.layers
    Ls = [synth.workload_layer(w, l, device=f"cuda:{dev}") for l in range(nl)]
    stack_prefix = []
    if args.dense_prefix != "0":  # hot-first order and an always-on prefix for every layer
        for l in range(nl):
            Ls[l], _, st_ = hot_first(w, Ls[l], dev, args.dense_prefix)
            stack_prefix.append(st_["dense_prefix"])
    lays = [B.Layer.from_dict(L) for L in Ls]
    for l in range(nl):
        lays[l].set_next(lays[(l + 1) % nl])  # the next layer of the stack (layer 0 of the next token)
    X = synth.workload_tokens(w, device=f"cuda:{dev}")
    if args.tokens:
        X = X[:args.tokens].contiguous()
    T, d = X.shape
    ws = B.workspace(B.pi_workspace_bytes(lays[0], 1), X.device)
    ya = torch.empty(d, dtype=torch.float32, device=X.device)
    xs = [torch.empty(d, dtype=torch.float32, device=X.device) for _ in range(2)]
    ys = [torch.empty(d, dtype=torch.float32, device=X.device) for _ in range(2)]
    Xout = torch.empty(T, d, dtype=torch.float32, device=X.device)
    stream = torch.cuda.Stream()

    def token(xin, xout, rec_x=None, rec_y=None):
        B.pi_ffn_layer(lays[0], xin, ys[0], ws=ws)
        xp, yp = xin, ys[0]
        if rec_x is not None:
            rec_x[0].copy_(xin)
            rec_y[0].copy_(ys[0])
        for l in range(1, nl):
            xn, yn = xs[l % 2], ys[l % 2]
            B.pi_ffn_layer_chain(lays[l], xp, yp, xn, yn, ws=ws)
            if rec_x is not None:
                rec_x[l].copy_(xn)
                rec_y[l].copy_(yn)
            xp, yp = xn, yn
        B.pi_rms_residual(xp, yp, xout)

    def step(Xin=X):
        for t in range(T):
            token(Xin[t], Xout[t])

    # statistics on the chained inputs of every layer (outside any timed region)
    Xl = torch.empty(nl, T, d, dtype=torch.float32, device=X.device)
    Yl = torch.empty(nl, T, d, dtype=torch.float32, device=X.device)
    for t in range(T):
        token(X[t], Xout[t], rec_x=[Xl[l, t] for l in range(nl)], rec_y=[Yl[l, t] for l in range(nl)])
    torch.cuda.synchronize()
    n_pred, n_down, recs, precs, dens, fire = [], [], [], [], [], []
    trues = []
    for l in range(nl):
        S = active_stats(w, Ls[l], lays[l], Xl[l], ws, ws, 1)
        n_pred.append(S["n_pred"])
        n_down.append(S["n_down"])
        recs.append(S["recall"])
        precs.append(S["precision"])
        dens.append(S["true_density"])
        fire.append(S["true"].sum(dim=0).cpu().numpy())
        trues.append(S["true"])
    n_pred, n_down = np.concatenate(n_pred), np.concatenate(n_down)
    Hm = float(np.mean(stack_prefix)) if stack_prefix else 0.0
    pred_b, ffn_b = needed_bytes(w, n_pred, n_down, 1, Hm)
    mean_bytes = float(np.mean(pred_b + ffn_b))  # per token and layer

    g_step = capture(step, stream)
    with Clocks(dev) as clk:
        ms = time_graph(g_step, args.steps, args.warmup, stream, barrier)
    ms_step = job_time(ms / args.steps, world, X.device)
    us_tok = whole_job_us_per_token(ms_step, T * nl, world)  # per layer per token
    layer_gbs = mean_bytes / (us_tok * world * 1e-6) / 1e9
    peak, peak_src = measured_peaks()
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token",
                              "quick": True, "workload": w.name, "tokens_per_step": T, "layer_gbs": layer_gbs,
                              "device_status": B.pi_sync_status(ws)}))
        return 0

    # the dominant kernel alone: every layer's k_layer_b1 (as the step calls it) on its
    # recorded inputs, back to back, without the one glue launch per token
    ksteps = max(4, args.steps // 4)
    xscratch = torch.empty(d, dtype=torch.float32, device=X.device)

    def kernel_only():
        for t in range(T):
            B.pi_ffn_layer(lays[0], Xl[0, t], ya, ws=ws)
            for l in range(1, nl):
                B.pi_ffn_layer_chain(lays[l], Xl[l - 1, t], Yl[l - 1, t], xscratch, ya, ws=ws)

    g_k = capture(kernel_only, stream)
    ms_k = time_graph(g_k, ksteps, min(args.warmup, 3), stream) / ksteps
    us_k = ms_k * 1000.0 / (T * nl)
    k_gbs = mean_bytes / (us_k * 1e-6) / 1e9

    # measurement mode (i): the sparse FFN alone on every layer's TRUE active lists
    tl = [true_lists(tr) for tr in trues]

    def sparse_true():
        for t in range(T):
            for l in range(nl):
                B.pi_sparse_ffn(lays[l], Xl[l, t], tl[l][0][t], tl[l][1][t:t + 1], ya, ws=ws)

    g_tr = capture(sparse_true, stream)
    ms_tr = time_graph(g_tr, ksteps, min(args.warmup, 3), stream) / ksteps
    us_tr = ms_tr * 1000.0 / (T * nl)
    n_true = np.concatenate([x[1].cpu().numpy() for x in tl])
    tr_b = float(np.mean(needed_bytes(w, n_true, n_true, 1)[1]))
    del tl

    # end to end: pinned host tokens in, the stack's outputs back
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(T, d, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(X)
    e2e_steps = max(2, args.steps // 10)
    with torch.cuda.stream(stream):
        def e2e_step():
            Xd.copy_(Xh, non_blocking=True)
            step(Xd)
            Yh.copy_(Xout, non_blocking=True)
        e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
    us_e2e = e0.elapsed_time(e1) / e2e_steps * 1000.0 / (T * nl)
    st = B.pi_sync_status(ws)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        olays = [oracle_layer(w, host_layer(Ls[l], w)) for l in range(nl)]
        us_cpu, done = oracle_stack_sample(w, olays, X.cpu().numpy(), args.cpu_seconds)
        cpu = {"value": us_cpu, "unit": "us/layer/token", "cores": 1, "kind": "oracle",
               "sample": f"first {done} of {T} tokens through all {nl} layers (predictor, compaction, sparse FFN, "
                         "residual + rescale), single-threaded C oracle, fp64"}
        del olays

    if rank == 0:
        fire_all = np.concatenate(fire)
        cfg = workload_config(w, 1, True)
        if stack_prefix:
            cfg["hot_first_order"] = True
            cfg["dense_prefix_per_layer"] = stack_prefix
        cfg.update({"tokens_per_step": T,
                    "l2": f"inputs larger than L2: {nl} distinct layers, "
                          f"{nl * mean_bytes / 1e6:.0f} MB needed bytes per token",
                    "n_active_mean": float(np.mean(n_pred)), "n_nonzero_mean": float(np.mean(n_down)),
                    "true_density_per_layer": [round(x, 4) for x in dens],
                    "predictor_recall": float(np.mean(recs)), "predictor_precision": float(np.mean(precs)),
                    "top26_firing_share": float(np.mean([top_share(f) for f in fire])),
                    "needed_bytes_per_token_layer": mean_bytes, "parallelism": f"replicas x{world}"})
        del fire_all
        line = {
            "metric": "us_per_ffn_layer_per_token", "value": us_tok, "unit": "us/layer/token", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16" if w.wtype == "f16" else w.wtype,
            "data": "synthetic", "config": cfg,
            "roofline": roofline_obj("k_layer_b1 (pi_ffn_layer), timed alone back to back on the stack's inputs",
                                     k_gbs, peak, peak_src, committed_traffic("k_layer_b1", w.name),
                                     launch_us=us_k),
            "roofline_layer": roofline_obj("stack end to end (k_layer_b1, one glue kernel per token)", layer_gbs,
                                           peak, peak_src, None),
            "kernels": {"per": "layer and token", "layer_kernel_us": us_k, "layer_kernel_gbs": k_gbs,
                        "layer_kernel_frac": k_gbs / peak, "step_us_per_layer": us_tok,
                        "true_mask_sparse_ffn_us": us_tr, "true_mask_sparse_ffn_gbs": tr_b / (us_tr * 1e-6) / 1e9,
                        "true_mask_sparse_ffn_frac": tr_b / (us_tr * 1e-6) / 1e9 / peak,
                        "true_mask_n_mean": float(np.mean(n_true))},
            "e2e": {"value": us_e2e, "unit": "us/layer/token", "h2d_bytes_per_step": int(Xh.numel() * 4),
                    "d2h_bytes_per_step": int(Yh.numel() * 4),
                    "path": "pi_ffn_layer, then pi_ffn_layer_chain per layer, pi_rms_residual per token"},
            "gpu_launches": (nl + 1) * T * args.steps,
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
    if w.layers > 1 and not args.one_layer:
        return run_stack(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
