"""Seeded synthetic inputs shared by the tests, the benchmark and the CPU oracle.

This module only draws inputs: it holds none of the sparse-FFN arithmetic (no
predictor evaluation, no masking, no compaction, no quantisation).  Whatever it
returns is fed unchanged to both the CUDA library and the oracle.

Recipe (the pages measure real OPT / LLaMA / Falcon checkpoints on Wikipedia
text; none of that is available, so seeded Gaussian stand-ins of the same
shapes are used):

* tokens  x ~ N(0, 1), float32.
* FFN weights  ~ N(0, std = 1/sqrt(fan_in)): fan_in = d_model for the up / gate
  projections, d_ff for the down projection (stored neuron-major [d_ff, d_model]).
* Power-law firing (PowerInfer summary page, "关键结果": about 26% of neurons
  carry 80% of the activations).  Neuron of popularity rank k fires with
  probability p_k = min(0.99, c * k^-s), s = 1.1, with c found by bisection so
  that mean(p) = 1 - sparsity.  The bias of the projection feeding the
  activation is b_j = ||w_j|| * ndtri(p_{pi(j)}), so that P(w_j.x + b_j > 0) =
  p_{pi(j)} for x ~ N(0, I); pi is a seeded random rank -> neuron map, which
  scatters the hot neurons (so a hot-first permutation has work to do).
  Gated layers put the bias on the gate; b_down = 0.
* Predictor, random kind (tiny config): P1 ~ N(0, 1/sqrt(d_model)),
  P2 ~ N(0, 1/sqrt(rank)), no bias, threshold 0.
* Predictor, projection kind (the larger configs; the pages give neither the
  predictor's form nor its training, and no training data exists here):
  Q = k = rank/2 random orthonormal directions of the input space,
  P1 = [Q; -Q], P2 = [L, -L] / ||L_j|| with L = W_act Q^T, p_bias = b.  Because
  relu(t) - relu(-t) = t, its logit is b_j + (w_j projected on span Q).x / s_j,
  distributed N(b_j, 1) like the true pre-activation, so threshold 0 gives the
  configured density; its recall is limited by how much of w_j lies in span Q.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    d_model: int
    d_ff: int
    rank: int
    gated: bool
    wtype: str            # "f32" | "f16" | "q4_0"
    sparsity: float       # expected fraction of neurons that do NOT fire
    tokens: int
    batch: int = 1
    layers: int = 1
    predictor: str = "projection"   # "random" | "projection"
    permute: bool = False           # hot-first permutation from a profiling pass
    profile_tokens: int = 0
    zipf_s: float = 1.1
    seed: int = 0


WORKLOADS = {
    "tiny-relu-fp32": Workload("tiny-relu-fp32", 512, 2048, 64, False, "f32", 0.90, 64,
                               predictor="random", seed=1000),
    "llama7b-reglu-fp16": Workload("llama7b-reglu-fp16", 4096, 11008, 1024, True, "f16", 0.90, 256,
                                   seed=1001),
    "opt30b-relu-fp16-perm": Workload("opt30b-relu-fp16-perm", 7168, 28672, 1024, False, "f16", 0.95,
                                      256, permute=True, profile_tokens=1024, seed=1002),
    "falcon40b-relu-fp16": Workload("falcon40b-relu-fp16", 8192, 32768, 1024, False, "f16", 0.90, 256,
                                    seed=1003),
    "falcon40b-relu-q4_0": Workload("falcon40b-relu-q4_0", 8192, 32768, 1024, False, "q4_0", 0.90, 256,
                                    seed=1003),
    "opt175b-relu-fp16-stack12": Workload("opt175b-relu-fp16-stack12", 12288, 49152, 1024, False, "f16",
                                          0.95, 128, layers=12, seed=1004),
}


def zipf_probs(n: int, density: float, s: float = 1.1, pmax: float = 0.99) -> np.ndarray:
    """p_k = min(pmax, c k^-s), k = 1..n, with mean(p) = density (bisection on c)."""
    k = np.arange(1, n + 1, dtype=np.float64)
    base = k ** (-s)
    lo, hi = 0.0, 1.0
    while np.minimum(pmax, hi * base).mean() < density:
        hi *= 2.0
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(pmax, c * base).mean() < density:
            lo = c
        else:
            hi = c
    return np.minimum(pmax, hi * base)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, std, seed, device="cpu", dtype=torch.float32) -> torch.Tensor:
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return (t * float(std)).to(dtype)


def tokens(n: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    """n decode-token activations x ~ N(0, 1), float32 [n, d]."""
    return randn((n, d), 1.0, seed, device)


def _storage(t: torch.Tensor, wtype: str) -> torch.Tensor:
    return t.to(torch.float32 if wtype == "f32" else torch.float16)


def make_layer(d_model: int, d_ff: int, rank: int, *, gated: bool, wtype: str = "f16",
               sparsity: float = 0.9, predictor: str = "projection", zipf_s: float = 1.1,
               seed: int = 0, device="cpu") -> dict:
    """One synthetic FFN layer plus predictor, as torch tensors on `device`.

    Matrices come back in their storage dtype (float32 for "f32", float16
    otherwise -- "q4_0" layers are returned in float16 and quantised by the
    caller with the library or the oracle).  Keys: w_up, w_gate (or None),
    w_down, b_act, b_down, p1, p2, p_bias (or None), threshold, plus the shape.
    """
    dev = torch.device(device)
    sd = seed * 1000
    w_up = randn((d_ff, d_model), d_model ** -0.5, sd + 1, dev)
    w_gate = randn((d_ff, d_model), d_model ** -0.5, sd + 2, dev) if gated else None
    w_down = randn((d_ff, d_model), d_ff ** -0.5, sd + 3, dev)
    w_act = w_gate if gated else w_up
    # fp16 storage changes the row norms slightly; use the stored rows
    w_act_st = _storage(w_act, wtype).to(torch.float32)
    norms = w_act_st.norm(dim=1)

    p = torch.from_numpy(zipf_probs(d_ff, 1.0 - sparsity, zipf_s)).to(dev)
    rank_of = torch.randperm(d_ff, generator=_gen(sd + 4, dev), device=dev)  # neuron j has rank rank_of[j]
    p_neuron = p[rank_of]
    b_act = (norms.double() * torch.special.ndtri(p_neuron)).to(torch.float32)
    b_down = torch.zeros(d_model, dtype=torch.float32, device=dev)

    ptype = torch.float32 if wtype == "f32" else torch.float16
    if predictor == "random":
        p1 = randn((rank, d_model), d_model ** -0.5, sd + 5, dev, ptype)
        p2 = randn((d_ff, rank), rank ** -0.5, sd + 6, dev, ptype)
        p_bias = None
    elif predictor == "projection":
        k = rank // 2
        g = randn((d_model, k), 1.0, sd + 5, dev)
        q, _ = torch.linalg.qr(g.cpu())             # [d, k] orthonormal columns (host LAPACK)
        q = q.to(dev)
        Q = q.T.contiguous()                        # [k, d]
        Lm = w_act_st @ Q.T                         # [d_ff, k]
        s = Lm.norm(dim=1, keepdim=True).clamp_min(1e-12)
        Lm = Lm / s
        p1 = torch.cat([Q, -Q], 0).to(ptype)
        p2 = torch.cat([Lm, -Lm], 1).to(ptype)
        p_bias = b_act.clone()
    else:
        raise ValueError(predictor)

    return dict(d_model=d_model, d_ff=d_ff, rank=rank, gated=gated, wtype=wtype,
                w_up=_storage(w_up, wtype), w_gate=None if w_gate is None else _storage(w_gate, wtype),
                w_down=_storage(w_down, wtype), b_act=b_act, b_down=b_down,
                p1=p1.contiguous(), p2=p2.contiguous(), p_bias=p_bias, threshold=0.0)


def workload_layer(w: Workload, layer: int = 0, device="cpu") -> dict:
    return make_layer(w.d_model, w.d_ff, w.rank, gated=w.gated, wtype=w.wtype, sparsity=w.sparsity,
                      predictor=w.predictor, zipf_s=w.zipf_s, seed=w.seed * 100 + layer, device=device)


def workload_tokens(w: Workload, n: int | None = None, device="cpu", stream: int = 0) -> torch.Tensor:
    """Decode tokens of the workload (stream 0) or its profiling pass (stream 1)."""
    return tokens(w.tokens if n is None else n, w.d_model, w.seed * 100 + 77 + stream, device)


def random_mask(n: int, density: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.random(n) < density).astype(np.uint8)


def integer_layer(d_model: int, d_ff: int, rank: int, *, gated: bool, wtype: str, seed: int,
                  device="cpu") -> dict:
    """Small-integer weights and biases (|w| <= 3, |b| <= 8): with small integer
    tokens every partial sum is an integer far below 2^24, so any summation
    order gives the same fp32 result."""
    gen = _gen(seed, "cpu")

    def ri(shape, lo, hi):
        return torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)

    dt = torch.float32 if wtype == "f32" else torch.float16
    out = dict(d_model=d_model, d_ff=d_ff, rank=rank, gated=gated, wtype=wtype,
               w_up=ri((d_ff, d_model), -3, 3).to(dt),
               w_gate=ri((d_ff, d_model), -3, 3).to(dt) if gated else None,
               w_down=ri((d_ff, d_model), -3, 3).to(dt),
               b_act=ri((d_ff,), -8, 8), b_down=ri((d_model,), -4, 4),
               p1=ri((rank, d_model), -2, 2).to(dt), p2=ri((d_ff, rank), -2, 2).to(dt),
               p_bias=ri((d_ff,), -8, 8), threshold=0.5)
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in out.items()}


def integer_tokens(n: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    gen = _gen(seed, "cpu")
    return torch.randint(-2, 3, (n, d), generator=gen).to(torch.float32).to(device)
