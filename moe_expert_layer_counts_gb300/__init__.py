"""Python binding of libmoe (include/moe.h): argument marshalling only.

Every step of the layer runs in the CUDA kernels of ``csrc/``; this module
turns torch tensors into device pointers and the current torch stream into a
``cudaStream_t``, calls the C ABI, and raises on a non-zero status.  PyTorch
provides device memory and streams, nothing else.  If the compiled library is
missing, loading fails loudly; there is no other implementation to fall back
to.

Names follow the C ABI: ``plan`` (moe_plan), ``dispatch``, ``expert_l1``,
``expert_l2``, ``expert_fused``, ``combine``, ``forward`` (moe_forward), ``plan_check``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
_lib = None
_lock = threading.Lock()

BLOCK_M = 128

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4
ERR_BAD_EXPERT_ID = 5
ERR_TIMEOUT = 6
ERR_TOO_LARGE = 8
ERR_DEBUG_BOUNDS = 9   # debug builds (MOE_DEBUG) only
SF_PAIRS_ADJACENT = 0
SF_PAIRS_HALVES = 1

EXPORT = dict(count=0, off=1, poff=2, slot_of=3, row_token=4, row_topk=5, row_weight=6, block_expert=7,
              n_blocks=8, pool_q=9, pool_sf=10, h_q=11, h_sf=12, l2_out=13, error=14, pool_rows=15,
              max_count=16, x_q=17)
_EXPORT_DTYPE = dict(count=torch.int32, off=torch.int32, poff=torch.int32, slot_of=torch.int32,
                     row_token=torch.int32, row_topk=torch.int32, row_weight=torch.float32,
                     block_expert=torch.int32, n_blocks=torch.int32, pool_q=torch.uint8, pool_sf=torch.uint8,
                     h_q=torch.uint8, h_sf=torch.uint8, l2_out=torch.bfloat16, error=torch.int32,
                     max_count=torch.int32, x_q=torch.uint8)

# every function declared in include/moe.h
SYMBOLS = ("moe_plan_workspace_bytes", "moe_weight_scales_bytes", "moe_prepare_weight_scales", "moe_plan",
           "moe_dispatch", "moe_expert_l1", "moe_expert_l2", "moe_combine", "moe_forward", "moe_plan_check",
           "moe_plan_export", "moe_error_string", "moe_expert_offsets_static", "moe_selftest_bounded_wait",
           "moe_selftest_mma_rate", "moe_expert_fused", "moe_selftest_fused_wait", "moe_selftest_stream_rate")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {error_string(status)} (status {status})")


class Plan(ctypes.Structure):
    """moe_plan_t: caller-owned opaque storage."""
    _fields_ = [("opaque", ctypes.c_uint64 * 24)]


class Weights(ctypes.Structure):
    """moe_weights_t."""
    _fields_ = [("q", ctypes.c_void_p), ("sf_mma", ctypes.c_void_p), ("E", ctypes.c_int32),
                ("N", ctypes.c_int32), ("K", ctypes.c_int32)]


SCALE_CEIL = 0
SCALE_OCP_FLOOR = 1


A_POOL = 0
A_GATHER = 1


class Options(ctypes.Structure):
    """moe_options_t: activation_clamp (> 0 limits bf16 gate/up to [-c, c]; 0 = off),
    scale_rule (SCALE_CEIL / SCALE_OCP_FLOOR for the activation scales), fast_math
    (1: fast SwiGLU with exact decisions, 0: exact everywhere; same bytes), a_operand
    (A_POOL: layer 1 reads the expert-major pool; A_GATHER: dispatch writes x once
    token-major and layer 1 gathers rows by token; same bytes)."""
    _fields_ = [("activation_clamp", ctypes.c_float), ("scale_rule", ctypes.c_int32),
                ("fast_math", ctypes.c_int32), ("a_operand", ctypes.c_int32), ("reserved", ctypes.c_int32 * 4)]

    def __init__(self, activation_clamp: float = 0.0, scale_rule: int = SCALE_CEIL, fast_math: int = 1,
                 a_operand: int = A_POOL):
        super().__init__(float(activation_clamp), int(scale_rule), int(fast_math), int(a_operand))


def _opts(options: "Options | None"):
    return None if options is None else ctypes.byref(options)


def lib():
    """Load libmoe.so (it must have been built: see build.py)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libmoe.so not built at {LIB_PATH}; run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.moe_plan_workspace_bytes.restype = sz
            L.moe_plan_workspace_bytes.argtypes = [i32] * 5
            L.moe_weight_scales_bytes.restype = sz
            L.moe_weight_scales_bytes.argtypes = [i32] * 3
            L.moe_prepare_weight_scales.restype = i32
            L.moe_prepare_weight_scales.argtypes = [P, i32, i32, i32, i32, P, sz, P]
            L.moe_plan.restype = i32
            L.moe_plan.argtypes = [ctypes.POINTER(Plan), P, P, i32, i32, i32, i32, i32, P, sz, P]
            OP = ctypes.POINTER(Options)
            L.moe_dispatch.restype = i32
            L.moe_dispatch.argtypes = [ctypes.POINTER(Plan), P, OP, P]
            L.moe_combine.restype = i32
            L.moe_combine.argtypes = [ctypes.POINTER(Plan), P, P]
            L.moe_expert_l1.restype = i32
            L.moe_expert_l1.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Weights), OP, P]
            L.moe_expert_l2.restype = i32
            L.moe_expert_l2.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Weights), P]
            L.moe_expert_fused.restype = i32
            L.moe_expert_fused.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Weights), ctypes.POINTER(Weights),
                                           OP, P]
            L.moe_selftest_fused_wait.restype = i32
            L.moe_selftest_fused_wait.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Weights),
                                                  ctypes.POINTER(Weights), P]
            L.moe_forward.restype = i32
            L.moe_forward.argtypes = [P, ctypes.POINTER(Weights), ctypes.POINTER(Weights), ctypes.POINTER(Plan), P,
                                      OP, P]
            L.moe_plan_check.restype = i32
            L.moe_plan_check.argtypes = [ctypes.POINTER(Plan), P]
            L.moe_plan_export.restype = i32
            L.moe_plan_export.argtypes = [ctypes.POINTER(Plan), i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            L.moe_expert_offsets_static.restype = i32
            L.moe_expert_offsets_static.argtypes = [P, i32, i32, i32, P, P, P, P]
            L.moe_selftest_bounded_wait.restype = i32
            L.moe_selftest_bounded_wait.argtypes = [i32, ctypes.c_uint64, P, P]
            L.moe_selftest_mma_rate.restype = i32
            L.moe_selftest_mma_rate.argtypes = [i32, P, ctypes.POINTER(i32), P]
            L.moe_selftest_stream_rate.restype = i32
            L.moe_selftest_stream_rate.argtypes = [P, P, P, P, i32, P, ctypes.POINTER(i32), P]
            L.moe_error_string.restype = ctypes.c_char_p
            L.moe_error_string.argtypes = [i32]
            _lib = L
    return _lib


def error_string(status: int) -> str:
    return lib().moe_error_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != OK:
        raise MoeError(rc, where)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------------- sizes
def plan_workspace_bytes(T: int, k: int, E: int, H: int, I: int) -> int:
    return int(lib().moe_plan_workspace_bytes(T, k, E, H, I))


def weight_scales_bytes(E: int, N: int, K: int) -> int:
    return int(lib().moe_weight_scales_bytes(E, N, K))


# ----------------------------------------------------------------- weights
class MXFP4Weight:
    """An [E, N, K] MXFP4 weight on the device: packed codes plus scales in
    the tensor-core layout (made once by ``prepare``)."""

    def __init__(self, q: torch.Tensor, sf_mma: torch.Tensor, E: int, N: int, K: int):
        self.q, self.sf_mma, self.E, self.N, self.K = q, sf_mma, E, N, K
        self.c = Weights(q.data_ptr(), sf_mma.data_ptr(), E, N, K)

    @classmethod
    def prepare(cls, q: torch.Tensor, sf: torch.Tensor, layer: int, stream=None) -> "MXFP4Weight":
        """q: uint8 [E,N,K/2] packed e2m1; sf: uint8 [E,N,K/32]; both on the GPU.
        layer 1 = W1 (gate rows then up rows), layer 2 = W2."""
        assert layer in (1, 2)
        E, N, K2 = q.shape
        K = 2 * K2
        assert sf.shape == (E, N, K // 32) and q.is_cuda and sf.is_cuda
        q = q.contiguous()
        sf = sf.contiguous()
        nbytes = weight_scales_bytes(E, N, K)
        if nbytes == 0:
            raise MoeError(ERR_UNSUPPORTED, "weight_scales_bytes")
        out = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        pairing = SF_PAIRS_HALVES if layer == 1 else SF_PAIRS_ADJACENT
        _check(lib().moe_prepare_weight_scales(_ptr(sf), E, N, K, pairing, _ptr(out), nbytes, _stream(stream)),
               "moe_prepare_weight_scales")
        return cls(q, out, E, N, K)


# ----------------------------------------------------------------- plan
class MoePlan:
    """A dispatch plan plus the workspace it lives in."""

    def __init__(self, c_plan: Plan, workspace: torch.Tensor, T, k, E, H, I):
        self.c, self.workspace = c_plan, workspace
        self.T, self.k, self.E, self.H, self.I = T, k, E, H, I

    def export(self, what: str):
        """View of an internal array of the plan (see MOE_EXPORT_* in moe.h)."""
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().moe_plan_export(ctypes.byref(self.c), EXPORT[what], ctypes.byref(off), ctypes.byref(nb)),
               "moe_plan_export")
        if what == "pool_rows":
            return nb.value
        raw = self.workspace[off.value: off.value + nb.value]
        return raw.view(_EXPORT_DTYPE[what])


def alloc_workspace(T, k, E, H, I, device=None) -> torch.Tensor:
    n = plan_workspace_bytes(T, k, E, H, I)
    if n == 0:
        raise MoeError(ERR_UNSUPPORTED, "plan_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def plan(topk_idx: torch.Tensor, topk_w: torch.Tensor, E: int, H: int, I: int,
         workspace: torch.Tensor | None = None, stream=None) -> MoePlan:
    """moe_plan: counts, offsets, stable slots.  topk_idx int64 [T,k], topk_w float32 [T,k]."""
    T, k = topk_idx.shape
    assert topk_idx.dtype == torch.int64 and topk_w.dtype == torch.float32
    topk_idx = topk_idx.contiguous()
    topk_w = topk_w.contiguous()
    if workspace is None:
        workspace = alloc_workspace(T, k, E, H, I, topk_idx.device)
    p = Plan()
    _check(lib().moe_plan(ctypes.byref(p), _ptr(topk_idx), _ptr(topk_w), T, k, E, H, I, _ptr(workspace),
                          workspace.numel(), _stream(stream)), "moe_plan")
    return MoePlan(p, workspace, T, k, E, H, I)


def dispatch(p: MoePlan, x: torch.Tensor, options: Options | None = None, stream=None):
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    _check(lib().moe_dispatch(ctypes.byref(p.c), _ptr(x), _opts(options), _stream(stream)), "moe_dispatch")


def expert_l1(p: MoePlan, W1: MXFP4Weight, options: Options | None = None, stream=None):
    _check(lib().moe_expert_l1(ctypes.byref(p.c), ctypes.byref(W1.c), _opts(options), _stream(stream)),
           "moe_expert_l1")


def expert_l2(p: MoePlan, W2: MXFP4Weight, stream=None):
    _check(lib().moe_expert_l2(ctypes.byref(p.c), ctypes.byref(W2.c), _stream(stream)), "moe_expert_l2")


def expert_fused(p: MoePlan, W1: MXFP4Weight, W2: MXFP4Weight, options: Options | None = None, stream=None):
    """moe_expert_fused: both expert layers in one persistent launch."""
    _check(lib().moe_expert_fused(ctypes.byref(p.c), ctypes.byref(W1.c), ctypes.byref(W2.c), _opts(options),
                                  _stream(stream)), "moe_expert_fused")


def selftest_fused_wait(p: MoePlan, W1: MXFP4Weight, W2: MXFP4Weight, stream=None):
    """moe_selftest_fused_wait: the fused launch with no row block ever ready
    (every layer-2 wait expires); read the outcome with plan_check."""
    _check(lib().moe_selftest_fused_wait(ctypes.byref(p.c), ctypes.byref(W1.c), ctypes.byref(W2.c),
                                         _stream(stream)), "moe_selftest_fused_wait")


def combine(p: MoePlan, y: torch.Tensor, stream=None):
    assert y.dtype == torch.bfloat16 and y.is_contiguous()
    _check(lib().moe_combine(ctypes.byref(p.c), _ptr(y), _stream(stream)), "moe_combine")


def forward(x: torch.Tensor, W1: MXFP4Weight, W2: MXFP4Weight, p: MoePlan, y: torch.Tensor | None = None,
            options: Options | None = None, stream=None) -> torch.Tensor:
    """moe_forward: dispatch + L1 + L2 + combine.  Returns y [T,H] bf16."""
    if y is None:
        y = torch.empty_like(x)
    assert x.dtype == torch.bfloat16 and x.is_contiguous() and y.is_contiguous()
    _check(lib().moe_forward(_ptr(x), ctypes.byref(W1.c), ctypes.byref(W2.c), ctypes.byref(p.c), _ptr(y),
                             _opts(options), _stream(stream)), "moe_forward")
    return y


def plan_check(p: MoePlan, stream=None) -> int:
    """Synchronise and return the device-side status (0, ERR_BAD_EXPERT_ID, ERR_TIMEOUT)."""
    return int(lib().moe_plan_check(ctypes.byref(p.c), _stream(stream)))


def expert_offsets_static(topk_idx: torch.Tensor, E: int, stream=None):
    """moe_expert_offsets_static: (count [E], offsets [E+1], padded offsets [E+1]) int32,
    computed with the library's fixed scratch instead of a caller workspace.  Only the
    three outputs are allocated here (by torch); the C entry point allocates nothing."""
    T, k = topk_idx.shape
    assert topk_idx.dtype == torch.int64
    topk_idx = topk_idx.contiguous()
    count = torch.empty(E, dtype=torch.int32, device=topk_idx.device)
    off = torch.empty(E + 1, dtype=torch.int32, device=topk_idx.device)
    poff = torch.empty(E + 1, dtype=torch.int32, device=topk_idx.device)
    _check(lib().moe_expert_offsets_static(_ptr(topk_idx), T, k, E, _ptr(count), _ptr(off), _ptr(poff),
                                           _stream(stream)), "moe_expert_offsets_static")
    return count, off, poff


def selftest_bounded_wait(arrive: bool, timeout_ns: int, stream=None):
    """moe_selftest_bounded_wait: (status, elapsed_us) of one device-side bounded
    mbarrier wait that is (arrive=True) or is not completed."""
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    _check(lib().moe_selftest_bounded_wait(int(bool(arrive)), int(timeout_ns), _ptr(out), _stream(stream)),
           "moe_selftest_bounded_wait")
    torch.cuda.synchronize()
    st, us = (int(v) for v in out.cpu())
    return st, us


MMA_FLOP_PER_KBLOCK = 4 * 2 * 128 * 256 * 32


def selftest_mma_rate(kblocks: int = 16384, repeats: int = 3, stream=None):
    """moe_selftest_mma_rate timed with CUDA events: the best of `repeats`
    launches (after one warm-up), as (TFLOP/s, CTAs, ms per launch)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream() if stream is None else stream
    ctas = ctypes.c_int(0)
    best = None
    for i in range(repeats + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        _check(lib().moe_selftest_mma_rate(int(kblocks), _ptr(status), ctypes.byref(ctas),
                                           ctypes.c_void_p(s.cuda_stream)), "moe_selftest_mma_rate")
        b.record(s)
        b.synchronize()
        _check(int(status.item()), "moe_selftest_mma_rate (device)")
        if i > 0:
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
    tflops = ctas.value * kblocks * MMA_FLOP_PER_KBLOCK / (best / 1e3) / 1e12
    return tflops, ctas.value, best


def selftest_stream_rate(kblocks: int = 8192, repeats: int = 3, stream=None):
    """moe_selftest_stream_rate timed with CUDA events on synthetic operands
    (finite E4M3 codes, random E2M1 codes, unit scales): the best of `repeats`
    launches (after one warm-up), as (TFLOP/s, CTAs, ms per launch)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    # E4M3 codes with bit 3 clear: never 0x7F / 0xFF (NaN)
    a = (torch.randint(0, 256, (2048 * 7168,), dtype=torch.int32, device=dev, generator=g) & 0xF7).to(torch.uint8)
    b = torch.randint(0, 256, (2 * 2048 * 3584,), dtype=torch.int32, device=dev, generator=g).to(torch.uint8)
    sfa = torch.full((16 * 56 * 512,), 127, dtype=torch.uint8, device=dev)
    sfb = torch.full((16 * 56 * 1024,), 127, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream() if stream is None else stream
    ctas = ctypes.c_int(0)
    best = None
    for i in range(repeats + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        _check(lib().moe_selftest_stream_rate(_ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb), int(kblocks), _ptr(status),
                                              ctypes.byref(ctas), ctypes.c_void_p(s.cuda_stream)),
               "moe_selftest_stream_rate")
        e1.record(s)
        e1.synchronize()
        _check(int(status.item()), "moe_selftest_stream_rate (device)")
        if i > 0:
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
    tflops = ctas.value * kblocks * MMA_FLOP_PER_KBLOCK / (best / 1e3) / 1e12
    return tflops, ctas.value, best
