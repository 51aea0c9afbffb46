"""Seeded synthetic inputs for the fused MoE forward.

This module is shared by the tests and the benchmark.  It holds none of the
layer's arithmetic: it draws random numbers and runs a harness router
(softmax -> top-k -> renormalise, which is not part of the layer).  The FP4
weights are drawn directly in their quantised form, as random E2M1 codes and
random UE8M0 exponents, so no quantiser lives here.

Workloads (all seeded, seed 0):
  tiny    T=64,   H=256,  I=128,  E=8,   k=2, uniform router
  mid     T=4096, H=2048, I=768,  E=64,  k=6, uniform router
  share   T=8192, H=7168, I=2048, E=32 local of 256 global, k=8; top-8 of the
          256 global experts, entries outside experts 0..31 set to -1
  full    T=8192, H=7168, I=2048, E=256, k=8, router logits + log Zipf(1.2)
          per-expert bias (load imbalance)
  decode  T=128,  H=7168, I=2048, E=256, k=8, uniform router

x ~ N(0,1) cast to bf16.  Weights W1 [E,2I,H], W2 [E,H,I] have the
distribution of N(0, 1/sqrt(K)) quantised to MXFP4 (one UE8M0 per 32 along
K): each E2M1 magnitude index is drawn from the probabilities that |2z|,
z ~ N(0,1), lies nearest to that E2M1 magnitude, the sign is a fair coin,
and each 32-block's exponent is s0 or s0+1 with the probability that makes
E[w^2] = 1/K.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SF_VEC = 32
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    router: str  # "uniform" | "zipf" | "share"
    global_experts: int = 0

    @property
    def flops_per_entry(self) -> int:
        """6*H*I: L1 (2*H*2I) + L2 (2*I*H) multiply-adds counted as 2 FLOPs."""
        return 6 * self.H * self.I


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 128, 8, 2, "uniform"),
    "mid": Workload("mid", 4096, 2048, 768, 64, 6, "uniform"),
    "share": Workload("share", 8192, 7168, 2048, 32, 8, "share", global_experts=256),
    "full": Workload("full", 8192, 7168, 2048, 256, 8, "zipf"),
    "decode": Workload("decode", 128, 7168, 2048, 256, 8, "uniform"),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0,1) as bf16 [T,H]."""
    g = _gen(seed, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_routing(w: Workload, seed: int = 1, device="cpu"):
    """Harness router.  Returns (topk_idx int64 [T,k], topk_w float32 [T,k])."""
    g = _gen(seed, device)
    n_glob = w.global_experts if w.router == "share" else w.E
    logits = torch.randn(w.T, n_glob, generator=g, device=device, dtype=torch.float32)
    if w.router == "zipf":
        r = torch.arange(1, n_glob + 1, device=device, dtype=torch.float64)
        p = r.pow(-1.2)
        p = p / p.sum()
        logits = logits + p.log().to(torch.float32)[None, :]
    probs = torch.softmax(logits, dim=-1)
    topv, topi = torch.topk(probs, w.k, dim=-1)
    topw = topv / topv.sum(dim=-1, keepdim=True)
    if w.router == "share":
        topi = torch.where(topi < w.E, topi, torch.full_like(topi, -1))
    return topi.to(torch.int64).contiguous(), topw.to(torch.float32).contiguous()


def _e2m1_magnitude_probs():
    """P(|2z| nearest to each E2M1 magnitude), z ~ N(0,1), and E[v^2]."""
    edges = [0.0] + [(a + b) / 2 for a, b in zip(_E2M1_MAG[:-1], _E2M1_MAG[1:])] + [math.inf]
    cdf = [math.erf((e / 2.0) / math.sqrt(2.0)) if e != math.inf else 1.0 for e in edges]
    probs = [cdf[i + 1] - cdf[i] for i in range(8)]
    ev2 = sum(p * m * m for p, m in zip(probs, _E2M1_MAG))
    return probs, ev2


def weight_exponent_recipe(K: int):
    """(s0, p_up): each 32-block exponent is s0+1 with probability p_up, else s0,
    so that E[w^2] = 1/K for w = v * 2^s."""
    _, ev2 = _e2m1_magnitude_probs()
    target = 1.0 / K
    s0 = math.floor(0.5 * math.log2(target / ev2))
    p_up = (target / (ev2 * 4.0 ** s0) - 1.0) / 3.0
    return s0, min(max(p_up, 0.0), 1.0)


def make_weights(E: int, N: int, K: int, seed: int, device="cpu"):
    """MXFP4 weights [E,N,K]: (q uint8 [E,N,K/2], two codes per byte with the
    even K index in the low nibble; sf uint8 [E,N,K/32], biased exponents)."""
    assert K % SF_VEC == 0
    g = _gen(seed, device)
    probs, _ = _e2m1_magnitude_probs()
    cum = torch.tensor([sum(probs[: i + 1]) for i in range(7)], device=device, dtype=torch.float32)
    s0, p_up = weight_exponent_recipe(K)
    q = torch.empty(E, N, K // 2, dtype=torch.uint8, device=device)
    sf = torch.empty(E, N, K // SF_VEC, dtype=torch.uint8, device=device)
    for e in range(E):
        u = torch.rand(N, K, generator=g, device=device, dtype=torch.float32)
        mag = torch.bucketize(u, cum, right=True).to(torch.uint8)  # 0..7
        sign = (torch.rand(N, K, generator=g, device=device) < 0.5).to(torch.uint8) << 3
        nib = mag | sign
        q[e] = nib[:, 0::2] | (nib[:, 1::2] << 4)
        up = (torch.rand(N, K // SF_VEC, generator=g, device=device) < p_up).to(torch.uint8)
        sf[e] = (127 + s0) + up
    return q, sf


def make_inputs(w: Workload, seed: int = 0, device="cpu", weight_device=None):
    """All inputs of one workload.  Weight tensors may be drawn on another
    device (e.g. the GPU for the big workloads)."""
    wd = device if weight_device is None else weight_device
    x = make_x(w.T, w.H, seed * 10 + 0, device)
    idx, tw = make_routing(w, seed * 10 + 1, device)
    w1q, w1sf = make_weights(w.E, 2 * w.I, w.H, seed * 10 + 2, wd)
    w2q, w2sf = make_weights(w.E, w.H, w.I, seed * 10 + 3, wd)
    return dict(x=x, topk_idx=idx, topk_w=tw, w1q=w1q, w1sf=w1sf, w2q=w2q, w2sf=w2sf)
