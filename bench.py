"""Benchmark of the fused MoE layer forward on GB300.

One step = the whole hot path on one batch: moe_plan (one kernel:
route_fused for up to 256 experts, route_small for more experts and at most
2048 top-k entries) + moe_forward (dispatch_quant, the fused expert kernel,
combine), on the full
skewed workload T=8192, H=7168, I=2048, E=256, k=8 by default.  Inputs are
synthetic and seeded, resident in HBM before timing; L2 is flushed (a 512 MB
buffer is written) before every timed step, outside the timed events.
FLOPs = 6 * N * H * I with N the number of valid top-k entries.

The default run also times the decode-shaped workload (T=128, same layer
sizes), whose bound is the weight stream from HBM, and reports it in a
`decode` object of the same JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload full]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

With N > 1 (torchrun), each rank runs an independent replica of the layer on
its own GPU (the layer does not shard on one node: weak scaling, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_layer_counts_gb300 import inputs  # noqa: E402

METRIC = "MoE fwd TFLOP/s & tokens/s (T=8192,H=7168,I=2048,E=256,k=8); % FP8 peak"
STAGES = ("route", "dispatch", "experts", "combine")             # what moe_forward runs (fused expert kernel)
STAGES_SEPARATE = ("route", "dispatch", "expert_l1", "expert_l2", "combine")
ROUTE_CHUNK = 2048  # top-k entries the one-CTA plan (more than 256 experts) handles
FUSED_PLAN_EXPERTS = 256  # experts up to which the plan is one multi-CTA launch
FLUSH_BYTES = 512 << 20
# FLOPs of one oracle sample (about 7 s on 16 host cores at the full layer size)
ORACLE_SAMPLE_FLOP = 4.0e11
# the reference arm's whole run (warm-up + timed calls) stays within about this much
# oracle work (a few minutes on 16 host cores): many steps take smaller samples
REFERENCE_RUN_FLOP = 1.2e13


def kernels_per_step(w, fused=True) -> int:
    """Kernels of the library one step launches: the plan (route_fused for up
    to FUSED_PLAN_EXPERTS experts, route_small for more experts and at most
    ROUTE_CHUNK top-k entries, otherwise route_count, route_scan and
    route_slot), dispatch_quant,
    the expert kernel(s) and combine.  Counters are zeroed by memset nodes,
    not kernels of the library."""
    one = w.T * w.k <= ROUTE_CHUNK or w.E <= FUSED_PLAN_EXPERTS
    return (1 if one else 3) + (3 if fused else 4)


def peaks():
    """Roofline denominators measured on this GPU pool: copy bandwidth and the
    bf16 GEMM rate as a burst (the GEMMs here are timed inside a short run of
    steps at the maximum SM clock); FP8 (the MXF8F6F4 rate) is 2x bf16, the
    nominal ratio of the two dense tensor rates."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        return dict(hbm_gbs=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    return rank, world


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) == 7:
                try:
                    self.samples.append((float(f[0]), float(f[1]), f[3:]))
                except ValueError:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for _, _, r in self.samples for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples), "sm_max_mhz": max(s[1] for s in self.samples),
                "reasons": reasons, "samples": len(self.samples)}


def kernel_source_hash() -> str:
    src = os.path.join(ROOT, "moe_expert_layer_counts_gb300", "csrc", "expert_gemm.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def measured_traffic(workload: str):
    """Per-launch DRAM bytes of the fused expert kernel on this workload from the
    committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "expert_traffic.json")
    if not os.path.exists(path):
        return None
    m = json.load(open(path))
    if m.get("kernel_sha") != kernel_source_hash():
        return None
    return m.get("bytes_per_launch", {}).get(workload)


# ------------------------------------------------------------------ oracle legs
def oracle_sample(w, flop=ORACLE_SAMPLE_FLOP):
    """The token sample both oracle timings (cpu_baseline and the reference
    arm) use: evenly spaced tokens, as many as make about `flop` of layer
    work at k entries per token (all tokens of the small workloads)."""
    import numpy as np
    n = min(w.T, max(32, int(flop / (6.0 * w.H * w.I * w.k))))
    step = max(1, w.T // n)
    return np.arange(0, w.T, step, dtype=np.int32)[:n], step


def _oracle_args(d):
    import numpy as np
    x = d["x"].cpu().view(torch.int16).numpy().view(np.uint16)
    idx = d["topk_idx"].cpu().numpy()
    tw = d["topk_w"].cpu().numpy()
    ws = [d[n].cpu().numpy() for n in ("w1q", "w1sf", "w2q", "w2sf")]
    return x, idx, tw, ws


def _sample_note(w, toks, step, n_valid):
    return (f"{len(toks)} tokens (every {step}th) of the {w.name} workload, {n_valid} valid entries, the same "
            f"sample in every call; weights of each touched expert dequantised inside the timing")


def cpu_baseline(w, d):
    """The oracle, as it stands, on the host cores: one untimed call, then one
    timed call on the sample of oracle_sample()."""
    import oracle
    oracle.build()
    x, idx, tw, ws = _oracle_args(d)
    toks, step = oracle_sample(w)
    oracle.forward(x, idx, tw, w.E, *ws, tokens=toks)
    t0 = time.perf_counter()
    oracle.forward(x, idx, tw, w.E, *ws, tokens=toks)
    dt = time.perf_counter() - t0
    n_valid = int((idx[toks] >= 0).sum())
    return dict(value=6.0 * n_valid * w.H * w.I / dt / 1e12, unit="TFLOP/s", cores=oracle.num_threads(),
                kind="oracle", seconds=dt, tokens_per_s=len(toks) / dt, sample=_sample_note(w, toks, step, n_valid))


def run_reference(args, w, rank, world):
    """Reference arm: the CPU oracle timed as it stands, on rank 0 only; every
    step is one oracle call on the sample of oracle_sample()."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    d = inputs.make_inputs(w, device="cpu", weight_device="cuda" if torch.cuda.is_available() else "cpu")
    x, idx, tw, ws = _oracle_args(d)
    # the cpu_baseline sample unless the run's step count would make the whole
    # run take more than a few minutes
    toks, step = oracle_sample(w, min(ORACLE_SAMPLE_FLOP, REFERENCE_RUN_FLOP / (args.warmup + args.steps)))
    n_valid = int((idx[toks] >= 0).sum())
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(x, idx, tw, w.E, *ws, tokens=toks)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = 6.0 * n_valid * w.H * w.I * args.steps / total / 1e12
    note = _sample_note(w, toks, step, n_valid)
    line = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
                ms_per_step=1e3 * total / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=f"{w.name}: T={w.T} H={w.H} I={w.I} E={w.E} k={w.k}", sample=note),
                cpu_baseline=dict(value=value, unit="TFLOP/s", cores=oracle.num_threads(), kind="oracle",
                                  sample=note),
                e2e=dict(value=value, unit="TFLOP/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU legs
class Layer:
    """One workload's inputs, prepared weights and workspace on the GPU."""

    def __init__(self, moe, w, dev):
        self.moe, self.w = moe, w
        self.d = inputs.make_inputs(w, seed=0, device=dev)
        self.W1 = moe.MXFP4Weight.prepare(self.d["w1q"], self.d["w1sf"], layer=1)
        self.W2 = moe.MXFP4Weight.prepare(self.d["w2q"], self.d["w2sf"], layer=2)
        self.ws = moe.alloc_workspace(w.T, w.k, w.E, w.H, w.I, dev)
        self.y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device=dev)
        idx = self.d["topk_idx"]
        self.n_valid = int((idx >= 0).sum().item())
        self.touched = int(torch.unique(idx[idx >= 0]).numel())
        counts = torch.bincount(idx[idx >= 0].flatten(), minlength=w.E)
        self.max_count = int(counts.max().item()) if self.n_valid else 0
        self.flops = 6.0 * self.n_valid * w.H * w.I
        # FP4 codes + UE8M0 scales of every touched expert (W1 and W2)
        self.weight_bytes = self.touched * 3 * w.H * w.I * (0.5 + 1.0 / 32)

    def step(self, ev=None, fused=True, options=None):
        """One step; with fused=False the two expert layers run as two
        launches (moe_expert_l1, moe_expert_l2) so that each can be timed."""
        m, w, d = self.moe, self.w, self.d
        rec = iter(ev) if ev else None
        if rec: next(rec).record()
        p = m.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I, workspace=self.ws)
        if rec: next(rec).record()
        m.dispatch(p, d["x"], options=options)
        if rec: next(rec).record()
        if fused:
            m.expert_fused(p, self.W1, self.W2, options=options)
        else:
            m.expert_l1(p, self.W1, options=options)
            if rec: next(rec).record()
            m.expert_l2(p, self.W2)
        if rec: next(rec).record()
        m.combine(p, self.y)
        if rec: next(rec).record()
        return p

    def expert_bytes(self):
        """Algorithmic bytes of one fused expert launch: the touched experts' W1
        and W2 (codes + scales), the pool rows read (codes + scales) and the
        bf16 L2 rows written (h stays an intermediate of the launch)."""
        w = self.w
        return self.weight_bytes + self.n_valid * w.H * (1 + 1.0 / 32) + self.n_valid * w.H * 2


def timed_steps(L, args, world, flush, dev, fused=True, options=None):
    """W untimed steps, then K steps bracketed by barrier + synchronize, each
    after an L2 flush (outside the events); CUDA events per stage."""
    moe = L.moe
    stages = STAGES if fused else STAGES_SEPARATE
    for _ in range(args.warmup):
        flush.fill_(1)
        p = L.step(fused=fused, options=options)
    torch.cuda.synchronize()
    status = moe.plan_check(p)
    assert status == 0, moe.error_string(status)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for i in range(args.steps):
            flush.fill_(i & 255)
            p = L.step(evs[i], fused=fused, options=options)
        torch.cuda.synchronize()
    barrier(world)
    status = moe.plan_check(p)
    assert status == 0, moe.error_string(status)
    stage_ms = {s: 0.0 for s in stages}
    total_ms = 0.0
    for e in evs:
        total_ms += e[0].elapsed_time(e[-1])
        for j, s in enumerate(stages):
            stage_ms[s] += e[j].elapsed_time(e[j + 1])
    t_max = max_over_ranks(total_ms / 1e3, world)
    return t_max, {s: v / args.steps for s, v in stage_ms.items()}, clk.summary()


def weight_stream(L, step_s, pk):
    gbs = L.weight_bytes / step_s / 1e9
    return dict(touched_experts=L.touched, bytes_per_step=L.weight_bytes, gbs=gbs, pct_hbm=gbs / pk["hbm_gbs"],
                note=f"touched experts' FP4 + UE8M0 weight bytes per step / step time, vs {pk['source']} "
                     f"HBM copy bandwidth {pk['hbm_gbs']} GB/s")


def roofline(L, stage_ms, pk, mma):
    """The dominant kernel, the fused expert kernel (both GEMMs): tensor-bound
    against the FP8 peak (and the measured block-scaled MMA ceiling) when
    experts hold more than 16 rows, otherwise bound by its weight stream from
    HBM."""
    w = L.w
    t_s = stage_ms["experts"] / 1e3
    kernel = "expert_gemm_kernel<3> (L1 + L2 fused)"
    if L.max_count <= 16:
        gb = L.expert_bytes()
        ach = gb / t_s / 1e9
        return dict(kernel=kernel, bound="hbm", achieved=ach, peak=pk["hbm_gbs"], unit="GB/s",
                    frac=ach / pk["hbm_gbs"], traffic=measured_traffic(w.name),
                    algorithmic=f"touched W1 + W2 (codes + scales) + pool rows read + L2 rows written = {gb:.4g} B "
                                f"per launch",
                    peak_note=f"{pk['source']} HBM copy bandwidth")
    fl = 6.0 * L.n_valid * w.H * w.I
    ach = fl / t_s / 1e12
    fp8 = 2.0 * pk["bf16"]
    r = dict(kernel=kernel, bound="tensor", achieved=ach, peak=fp8, unit="TFLOP/s",
             frac=ach / fp8, traffic=measured_traffic(w.name),
             algorithmic=f"6*N*H*I = {fl:.4g} FLOP per launch (valid rows only)",
             peak_note=f"FP8 = 2 x {pk['source']} burst bf16 cuBLAS rate ({pk['bf16']} TF/s), the nominal FP8/bf16 "
                       f"ratio of the dense tensor rates")
    if mma:
        r.update(frac_vs_mma=ach / mma["tflops"], mma_ceiling_tflops=mma["tflops"],
                 frac_vs_stream=ach / mma["stream"]["tflops"], stream_ceiling_tflops=mma["stream"]["tflops"])
    return r


def separate_leg(L, args, world, flush, dev, pk):
    """The same steps with the two expert layers as two launches: per-layer
    times and tensor rates (L1 4*N*H*I, L2 2*N*H*I FLOP)."""
    t, stage_ms, _ = timed_steps(L, args, world, flush, dev, fused=False)
    w = L.w
    fp8 = 2.0 * pk["bf16"]
    out = dict(ms_per_step=1e3 * t / args.steps, stage_ms=stage_ms)
    for name, f in (("expert_l1", 4.0), ("expert_l2", 2.0)):
        tf = f * L.n_valid * w.H * w.I / (stage_ms[name] / 1e3) / 1e12
        out[name] = dict(tflops=tf, frac_fp8=tf / fp8)
    return out


def gather_leg(L, args, world, flush, dev):
    """The same steps with layer 1 gathering its A rows by token from
    token-major x (moe_options_t.a_operand = MOE_A_GATHER: dispatch writes each
    token's codes once instead of k pool rows; same results)."""
    t, stage_ms, _ = timed_steps(L, args, world, flush, dev, options=L.moe.Options(a_operand=L.moe.A_GATHER))
    return dict(ms_per_step=1e3 * t / args.steps, value=world * L.flops * args.steps / t / 1e12, unit="TFLOP/s",
                stage_ms=stage_ms,
                note="A operand of layer 1 gathered by token with TMA tile::gather4 (32 four-row requests per "
                     "128-row stage) instead of one 128-row box of the expert-major pool")


def mma_ceiling(moe, dev):
    """The block-scaled MMA (the GEMMs' instruction) issued back to back on every
    SM from fixed shared-memory operands: the tensor pipe's rate on this GPU.
    Beside it, the same MMAs fed by the layer-1 tile's own operand stream (TMA
    ring, scale copies, no epilogue) from L2-resident operands, with the SM
    clocks sampled while it runs: what this tile shape can reach with its
    operands moving, under the board's power limit."""
    tflops, ctas, ms = moe.selftest_mma_rate(kblocks=16384, repeats=3)
    with ClockSampler(dev.index) as clk:
        s_tf, s_ctas, s_ms = moe.selftest_stream_rate(kblocks=16384, repeats=20)
    return dict(tflops=tflops, ctas=ctas, ms=ms,
                note="moe_selftest_mma_rate: M=128 N=256 K=32 kind::mxf8f6f4 block-scaled MMAs, one CTA per SM, "
                     "16384 x 4 per CTA, best of 3 launches",
                stream=dict(tflops=s_tf, ctas=s_ctas, ms=s_ms, clocks=clk.summary(),
                            note="moe_selftest_stream_rate: the same MMAs fed by the layer-1 tile's 4-stage TMA ring "
                                 "(128-row E4M3 A box, 256-row E2M1 B box, scale copies), no epilogue, one CTA per "
                                 "SM, 16384 k-blocks per CTA, best of 20 launches"))


def decode_leg(moe, args, world, flush, dev, pk):
    """The decode-shaped workload, timed like the main one."""
    w = inputs.WORKLOADS["decode"]
    L = Layer(moe, w, dev)
    t, stage_ms, clk = timed_steps(L, args, world, flush, dev)
    step_s = t / args.steps
    out = dict(workload=f"{w.name}: T={w.T} H={w.H} I={w.I} E={w.E} k={w.k}", ms_per_step=1e3 * step_s,
               value=world * L.flops / step_s / 1e12, unit="TFLOP/s", tokens_per_s=world * w.T / step_s,
               stage_ms=stage_ms, weight_stream=weight_stream(L, step_s, pk), roofline=roofline(L, stage_ms, pk, None),
               clocks=clk, gpu_launches=kernels_per_step(w) * args.steps,
               separate_kernels=separate_leg(L, args, world, flush, dev, pk))
    del L
    torch.cuda.empty_cache()
    return out


def e2e_legs(L, args, world, flush):
    """End to end through the public API: pinned host inputs -> GPU -> pinned
    host y, three ways (a pipelined stream of steps, one step at a time, one
    step as a replayed CUDA graph)."""
    moe, w, d = L.moe, L.w, L.d
    hx = d["x"].cpu().pin_memory()
    hidx = d["topk_idx"].cpu().pin_memory()
    htw = d["topk_w"].cpu().pin_memory()
    hy = torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory()
    gx, gidx, gtw = torch.empty_like(d["x"]), torch.empty_like(d["topk_idx"]), torch.empty_like(d["topk_w"])
    e2e_ms = 0.0
    for i in range(args.warmup + args.e2e_steps):
        flush.fill_(3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gx.copy_(hx, non_blocking=True)
        gidx.copy_(hidx, non_blocking=True)
        gtw.copy_(htw, non_blocking=True)
        pp = moe.plan(gidx, gtw, w.E, w.H, w.I, workspace=L.ws)
        moe.forward(gx, L.W1, L.W2, pp, L.y)
        hy.copy_(L.y, non_blocking=True)
        b.record()
        b.synchronize()
        if i >= args.warmup:
            e2e_ms += a.elapsed_time(b)
    e2e_t = max_over_ranks(e2e_ms / 1e3, world)
    serial = world * L.flops * args.e2e_steps / e2e_t / 1e12

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gx.copy_(hx, non_blocking=True)
            gidx.copy_(hidx, non_blocking=True)
            gtw.copy_(htw, non_blocking=True)
            gp = moe.plan(gidx, gtw, w.E, w.H, w.I, workspace=L.ws)
            moe.forward(gx, L.W1, L.W2, gp, L.y)
            hy.copy_(L.y, non_blocking=True)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph_ms = 0.0
    for i in range(args.warmup + args.e2e_steps):
        flush.fill_(3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        if i >= args.warmup:
            graph_ms += a.elapsed_time(b)
    status = moe.plan_check(gp)
    assert status == 0, moe.error_string(status)
    graph_t = max_over_ranks(graph_ms / 1e3, world)
    graph_val = world * L.flops * args.e2e_steps / graph_t / 1e12
    # a stream of steps as a serving loop runs them: copies in, compute and copies out on three streams, two
    # buffer sets, so step i+1's inputs arrive and step i-1's output leaves while step i computes (every step's
    # copies stay inside the timed region; no L2 flush: the weights and the pool exceed L2 on these workloads)
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    gx2 = [torch.empty_like(d["x"]) for _ in range(2)]
    gidx2 = [torch.empty_like(d["topk_idx"]) for _ in range(2)]
    gtw2 = [torch.empty_like(d["topk_w"]) for _ in range(2)]
    y2 = [torch.empty_like(d["x"]) for _ in range(2)]
    hy2 = [torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_in.wait_stream(torch.cuda.current_stream())
        start.record(s_in)
        pl = None
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_comp[b])
            with torch.cuda.stream(s_in):
                gx2[b].copy_(hx, non_blocking=True)
                gidx2[b].copy_(hidx, non_blocking=True)
                gtw2[b].copy_(htw, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            if i >= 2:
                s_comp.wait_event(ev_out[b])
            pl = moe.plan(gidx2[b], gtw2[b], w.E, w.H, w.I, workspace=L.ws, stream=s_comp)
            moe.forward(gx2[b], L.W1, L.W2, pl, y2[b], stream=s_comp)
            ev_comp[b].record(s_comp)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                hy2[b].copy_(y2[b], non_blocking=True)
            ev_out[b].record(s_out)
        end.record(s_out)
        end.synchronize()
        return start.elapsed_time(end), pl

    pipelined(args.warmup)
    torch.cuda.synchronize()
    pipe_ms, pl = pipelined(args.e2e_steps)
    status = moe.plan_check(pl, stream=s_comp)
    assert status == 0, moe.error_string(status)
    pipe_t = max_over_ranks(pipe_ms / 1e3, world)
    pipe_val = world * L.flops * args.e2e_steps / pipe_t / 1e12
    h2d = hx.numel() * 2 + hidx.numel() * 8 + htw.numel() * 4
    d2h = hy.numel() * 2
    return dict(value=pipe_val, unit="TFLOP/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                ms_per_step=1e3 * pipe_t / args.e2e_steps,
                note="a stream of steps through the public API: each step copies its inputs in from pinned host "
                     "memory and its y out; copies in, compute and copies out run on three streams with two "
                     "buffer sets, so the copies of neighbouring steps overlap the compute",
                serial=dict(value=serial, unit="TFLOP/s", ms_per_step=1e3 * e2e_t / args.e2e_steps,
                            note="one step at a time: copy in, plan, forward, copy out, wait"),
                graph=dict(value=graph_val, unit="TFLOP/s", ms_per_step=1e3 * graph_t / args.e2e_steps,
                           note="one step at a time, captured once in a CUDA graph and replayed"))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="full", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode leg of the default run")
    ap.add_argument("--e2e-steps", type=int, default=50)
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    w = inputs.WORKLOADS[args.workload]
    rank, world = dist_init(args)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import moe_expert_layer_counts_gb300 as moe
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    mma = mma_ceiling(moe, dev)
    L = Layer(moe, w, dev)
    t_max, stage_ms, clk = timed_steps(L, args, world, flush, dev)
    value = world * L.flops * args.steps / t_max / 1e12
    step_s = t_max / args.steps
    separate = separate_leg(L, args, world, flush, dev, pk)
    gathered = gather_leg(L, args, world, flush, dev)
    e2e = e2e_legs(L, args, world, flush)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, L.d)
    fp8 = 2.0 * pk["bf16"]
    line = dict(
        metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=1e3 * step_s, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="e4m3 x e2m1 -> fp32 (MXFP8 x MXFP4, UE8M0/32)", data="synthetic",
        config=dict(workload=f"{w.name}: T={w.T} H={w.H} I={w.I} E={w.E} k={w.k}", T=w.T, H=w.H, I=w.I, E=w.E,
                    k=w.k, valid_entries=L.n_valid, l2="flushed before every timed step (512 MB write)",
                    parallelism=f"replicas x{world}"),
        tokens_per_s=world * w.T / step_s,
        weight_stream=weight_stream(L, step_s, pk),
        pct_fp8_peak=value / world / fp8,
        fp8_peak_tflops=dict(value=fp8, note=f"2 x {pk['source']} burst bf16 cuBLAS rate ({pk['bf16']} TF/s)"),
        pct_mma_ceiling=value / world / mma["tflops"],
        mma_ceiling=mma,
        stage_ms=stage_ms,
        roofline=roofline(L, stage_ms, pk, mma),
        separate_kernels=separate,
        a_gather=gathered,
        e2e=e2e,
        gpu_launches=kernels_per_step(w) * args.steps,
        clocks=clk,
        cpu_baseline=cpu,
    )
    del L, e2e
    torch.cuda.empty_cache()
    if w.name != "decode" and not args.no_decode:
        line["decode"] = decode_leg(moe, args, world, flush, dev, pk)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
