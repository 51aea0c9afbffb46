"""Seeded synthetic inputs for the fused MoE forward.

This module is shared by the tests and the benchmark.  It holds none of the
layer's arithmetic: it draws random numbers, runs a harness router (softmax
-> top-k -> renormalise, which is not part of the layer) and turns Gaussian
weights into the MXFP4 bytes the layer takes as input (the layer never
quantises weights; this is how its inputs are made).

Workloads (all seeded, seed 0):
  tiny    T=64,   H=256,  I=128,  E=8,   k=2, uniform router
  mid     T=4096, H=2048, I=768,  E=64,  k=6, uniform router
  share   T=8192, H=7168, I=2048, E=32 local of 256 global, k=8; top-8 of the
          256 global experts, entries outside experts 0..31 set to -1
  full    T=8192, H=7168, I=2048, E=256, k=8, router logits + log Zipf(1.2)
          per-expert bias (load imbalance)
  decode  T=128,  H=7168, I=2048, E=256, k=8, uniform router

x ~ N(0,1) cast to bf16.  Weights W1 [E,2I,H], W2 [E,H,I] are drawn as
N(0, 1/sqrt(K)) (standard deviation 1/sqrt(K), K the reduction length) and
quantised to MXFP4 along K, one expert at a time on the weights' device: per
32-block the UE8M0 scale 2^e with the smallest e such that amax <= 6 * 2^e
(clamped to [-126, 127], 2^0 for an all-zero block), then every value / 2^e
rounded to the nearest E2M1 value (0, .5, 1, 1.5, 2, 3, 4, 6), ties to the
even code, sign in bit 3.  Codes are packed two per byte, the even K index in
the low nibble.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SF_VEC = 32


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


# midpoints between consecutive E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6
_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def quantize_mxfp4(w: torch.Tensor):
    """MXFP4 bytes of a float tensor [N, K] (K a multiple of 32): (q uint8
    [N, K/2], sf uint8 [N, K/32] biased exponents), by the rule in the module
    docstring.  The scale exponent is read off frexp(amax) = f * 2^q (f in
    [0.5, 1)): 6 * 2^e >= amax first holds at e = q - 3 when f <= 0.75 and at
    e = q - 2 otherwise; both comparisons are exact."""
    N, K = w.shape
    assert K % SF_VEC == 0
    # float32 throughout: amax, frexp, the power-of-two scaling and the
    # comparisons with the (exactly representable) midpoints are all exact
    b = w.to(torch.float32).reshape(N, K // SF_VEC, SF_VEC)
    amax = b.abs().amax(dim=-1)
    f, q = torch.frexp(amax)
    e = torch.where(f <= 0.75, q - 3, q - 2)
    e = torch.where(amax > 0, e, torch.zeros_like(e)).clamp(-126, 127)
    v = b * torch.ldexp(torch.ones_like(amax), -e)[..., None]
    a = v.abs()
    mids = torch.tensor(_E2M1_MIDS, dtype=torch.float32, device=w.device)
    code = torch.bucketize(a, mids, right=False)          # midpoints strictly below a
    tie = (code < len(_E2M1_MIDS)) & (a == mids[code.clamp(max=len(_E2M1_MIDS) - 1)])
    code = code + (tie & (code % 2 == 1)).to(code.dtype)   # a tie goes to the even code
    neg = (v < 0) | ((v == 0) & torch.signbit(v))
    nib = (code | (neg.to(code.dtype) << 3)).to(torch.uint8).reshape(N, K)
    qb = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return qb.contiguous(), (e + 127).to(torch.uint8).contiguous()


def make_weights(E: int, N: int, K: int, seed: int, device="cpu"):
    """MXFP4 weights [E,N,K] quantised from N(0, 1/sqrt(K)): (q uint8
    [E,N,K/2], two codes per byte with the even K index in the low nibble;
    sf uint8 [E,N,K/32], biased exponents)."""
    assert K % SF_VEC == 0
    g = _gen(seed, device)
    q = torch.empty(E, N, K // 2, dtype=torch.uint8, device=device)
    sf = torch.empty(E, N, K // SF_VEC, dtype=torch.uint8, device=device)
    std = 1.0 / math.sqrt(K)
    for e in range(E):
        w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * std
        q[e], sf[e] = quantize_mxfp4(w)
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
