"""Plain CPU oracle of the fused MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python
binding) never imports it, and it shares no code with them.

The arithmetic lives in ``moe_oracle.c`` (plain C, double accumulation); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Every function cites the passage of the analysed pages it follows in the C
source.  All functions here are pinned by the ``-m "not gpu"`` tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK_M = 128
SF_VEC = 32


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.or_e4m3_decode.restype = f64
            L.or_e4m3_decode.argtypes = [i32]
            L.or_e4m3_encode.restype = i32
            L.or_e4m3_encode.argtypes = [f64]
            L.or_e2m1_decode.restype = f64
            L.or_e2m1_decode.argtypes = [i32]
            L.or_e2m1_encode.restype = i32
            L.or_e2m1_encode.argtypes = [f64]
            L.or_ue8m0_ceil.restype = i32
            L.or_ue8m0_ceil.argtypes = [f64, f64]
            L.or_ue8m0_value.restype = f64
            L.or_ue8m0_value.argtypes = [i32]
            L.or_ue8m0_floor.argtypes = [f64, i32]
            L.or_ue8m0_floor.restype = i32
            L.or_quant_mx_e4m3_rule.argtypes = [P, i32, P, P, i32]
            L.or_quant_mx_e4m3_rule.restype = None
            L.or_bf16_decode.restype = ctypes.c_float
            L.or_bf16_decode.argtypes = [ctypes.c_uint16]
            L.or_bf16_encode.restype = ctypes.c_uint16
            L.or_bf16_encode.argtypes = [ctypes.c_float]
            L.or_quant_mx_e4m3.restype = None
            L.or_quant_mx_e4m3.argtypes = [P, i32, P, P]
            L.or_quant_mx_e2m1.restype = None
            L.or_quant_mx_e2m1.argtypes = [P, i32, P, P]
            L.or_plan.restype = i32
            L.or_plan.argtypes = [P, P, i32, i32, i32, i64, P, P, P, P, P, P, P]
            L.or_quant_x.restype = None
            L.or_quant_x.argtypes = [P, i32, i32, i32, P, P, i32]
            L.or_forward.restype = i32
            L.or_forward.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P, i64,
                                     ctypes.c_float, i32, i32]
            L.or_l2_combine.restype = i32
            L.or_l2_combine.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, i64, P, i32, P, i32]
            L.or_combine.restype = None
            L.or_combine.argtypes = [P, P, i32, i32, i32, P]
            L.or_bruteforce_token.restype = i32
            L.or_bruteforce_token.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, ctypes.c_float, i32, P]
            L.or_num_threads.restype = i32
            L.or_num_threads.argtypes = []
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codecs
def e4m3_decode(code: int) -> float:
    return lib().or_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().or_e4m3_encode(float(v))


def e2m1_decode(nib: int) -> float:
    return lib().or_e2m1_decode(int(nib))


def e2m1_encode(v: float) -> int:
    return lib().or_e2m1_encode(float(v))


SCALE_RULE_CEIL = 0
SCALE_RULE_OCP_FLOOR = 1


def ue8m0_floor(amax: float, emax_elem: int) -> int:
    """UE8M0 byte of the OCP MX floor rule: 2^(floor(log2 amax) - emax_elem)."""
    return lib().or_ue8m0_floor(float(amax), int(emax_elem))


def ue8m0_ceil(amax: float, maxnorm: float) -> int:
    return lib().or_ue8m0_ceil(float(amax), float(maxnorm))


def ue8m0_value(byte: int) -> float:
    return lib().or_ue8m0_value(int(byte))


def bf16_decode(bits: int) -> float:
    return lib().or_bf16_decode(int(bits))


def bf16_encode(v: float) -> int:
    return lib().or_bf16_encode(float(v))


def quant_mx_e4m3(v: np.ndarray, scale_rule: int = SCALE_RULE_CEIL):
    """MX E4M3 of a float32 vector (length a multiple of 32) -> (codes, scale bytes)."""
    v = _c(v, np.float32).ravel()
    codes = np.zeros(v.size, np.uint8)
    sf = np.zeros(v.size // SF_VEC, np.uint8)
    lib().or_quant_mx_e4m3_rule(_p(v), v.size, _p(codes), _p(sf), int(scale_rule))
    return codes, sf


def quant_mx_e2m1(v: np.ndarray):
    """MXFP4 of a float32 vector -> (nibbles one per byte, sf u8)."""
    v = _c(v, np.float32).ravel()
    nib = np.zeros(v.size, np.uint8)
    sf = np.zeros(v.size // SF_VEC, np.uint8)
    lib().or_quant_mx_e2m1(_p(v), v.size, _p(nib), _p(sf))
    return nib, sf


# ---------------------------------------------------------------- plan
def pool_capacity(T: int, k: int, E: int) -> int:
    """Upper bound of the padded pool rows: N + min(E, N)*(BLOCK_M-1), rounded up."""
    n = T * k
    cap = n + min(E, n) * (BLOCK_M - 1)
    return max(BLOCK_M, (cap + BLOCK_M - 1) // BLOCK_M * BLOCK_M)


def plan(topk_idx: np.ndarray, topk_w: np.ndarray, E: int, p_cap: int | None = None):
    """Routing plan.  Returns dict with count, off, poff, slot_of, row_token,
    row_topk, row_weight and status (0 ok, 1 bad expert id seen)."""
    idx = _c(topk_idx, np.int64)
    T, k = idx.shape
    w = _c(topk_w, np.float32)
    if p_cap is None:
        p_cap = pool_capacity(T, k, E)
    out = dict(
        count=np.zeros(E, np.int32), off=np.zeros(E + 1, np.int32), poff=np.zeros(E + 1, np.int32),
        slot_of=np.zeros(max(T * k, 1), np.int32), row_token=np.zeros(p_cap, np.int32),
        row_topk=np.zeros(p_cap, np.int32), row_weight=np.zeros(p_cap, np.float32),
    )
    st = lib().or_plan(_p(idx), _p(w), T, k, E, p_cap, _p(out["count"]), _p(out["off"]), _p(out["poff"]),
                       _p(out["slot_of"]), _p(out["row_token"]), _p(out["row_topk"]), _p(out["row_weight"]))
    out["slot_of"] = out["slot_of"][: T * k]
    out["status"] = st
    out["p_cap"] = p_cap
    return out


def quant_x(x_bf16_bits: np.ndarray, nthreads: int = 0, scale_rule: int = SCALE_RULE_CEIL):
    """Token-major MXFP8 of x given as uint16 bf16 bits [T,H] -> (q [T,H], sf [T,H/32])."""
    x = _c(x_bf16_bits, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), np.uint8)
    sf = np.zeros((T, H // SF_VEC), np.uint8)
    lib().or_quant_x(_p(x), T, H, int(scale_rule), _p(q), _p(sf), nthreads)
    return q, sf


def forward(x_bf16_bits, topk_idx, topk_w, E, w1q, w1sf, w2q, w2sf, tokens=None,
            want_pool=False, nthreads: int = 0, activation_clamp: float = 0.0,
            scale_rule: int = SCALE_RULE_CEIL):
    """Oracle forward.  x: uint16 bf16 bits [T,H]; w1q uint8 [E,2I,H/2]; w1sf uint8
    [E,2I,H/32]; w2q uint8 [E,H,I/2]; w2sf uint8 [E,H,I/32].
    tokens: optional int array of tokens to compute (y rows in that order).
    want_pool: also return per-pool-row hq [p_cap,I], hsf [p_cap,I/32], o [p_cap,H] and the
    pre-requantisation h [p_cap,I] (float32); with a token subset only the pool rows of those
    tokens are filled (the others stay zero).
    activation_clamp: > 0 limits the bf16 gate and up values to [-c, c] before SwiGLU.
    scale_rule: SCALE_RULE_CEIL or SCALE_RULE_OCP_FLOOR for the activation (x and h) scales.
    Returns dict(y=uint16 bf16 bits, status, and pool arrays if asked)."""
    x = _c(x_bf16_bits, np.uint16)
    T, H = x.shape
    idx = _c(topk_idx, np.int64)
    k = idx.shape[1] if idx.ndim == 2 else 1
    w = _c(topk_w, np.float32)
    w1q, w1sf, w2q, w2sf = (_c(a, np.uint8) for a in (w1q, w1sf, w2q, w2sf))
    I = w2q.shape[2] * 2
    assert w1q.shape == (E, 2 * I, H // 2) and w1sf.shape == (E, 2 * I, H // SF_VEC)
    assert w2q.shape == (E, H, I // 2) and w2sf.shape == (E, H, I // SF_VEC)
    p_cap = pool_capacity(T, k, E)
    res = {}
    if tokens is None:
        toks_p, ntok = None, T
    else:
        toks = _c(tokens, np.int32)
        toks_p, ntok = _p(toks), toks.size
    y = np.zeros((ntok, H), np.uint16)
    hq = hsf = o = hf = None
    if want_pool:
        hq = np.zeros((p_cap, I), np.uint8)
        hsf = np.zeros((p_cap, I // SF_VEC), np.uint8)
        o = np.zeros((p_cap, H), np.uint16)
        hf = np.zeros((p_cap, I), np.float32)
    st = lib().or_forward(_p(x), _p(idx), _p(w), T, k, E, H, I, _p(w1q), _p(w1sf), _p(w2q), _p(w2sf),
                          toks_p, ntok, _p(y),
                          _p(hq) if hq is not None else None, _p(hsf) if hsf is not None else None,
                          _p(o) if o is not None else None, _p(hf) if hf is not None else None, p_cap,
                          float(activation_clamp), int(scale_rule), nthreads)
    res.update(y=y, status=st)
    if hq is not None:
        res.update(hq=hq, hsf=hsf, o=o, h=hf)
    return res


def l2_combine(topk_idx, topk_w, E, w2q, w2sf, hq_pool, hsf_pool, tokens, nthreads: int = 0):
    """L2 + combine of the listed tokens from given requantised L1 outputs
    (hq_pool uint8 [p_cap, I], hsf_pool uint8 [p_cap, I/32], indexed by the
    plan's pool rows): the second half of forward(), to replay the layer
    from another implementation's h.  Returns y (uint16 bf16 bits [ntok, H])."""
    idx = _c(topk_idx, np.int64)
    T, k = idx.shape
    w = _c(topk_w, np.float32)
    w2q, w2sf = _c(w2q, np.uint8), _c(w2sf, np.uint8)
    H, I = w2q.shape[1], w2q.shape[2] * 2
    hq, hsf = _c(hq_pool, np.uint8), _c(hsf_pool, np.uint8)
    p_cap = hq.shape[0]
    assert hq.shape == (p_cap, I) and hsf.shape == (p_cap, I // SF_VEC) and p_cap >= pool_capacity(T, k, E)
    toks = _c(tokens, np.int32)
    y = np.zeros((toks.size, H), np.uint16)
    st = lib().or_l2_combine(_p(idx), _p(w), T, k, E, H, I, _p(w2q), _p(w2sf), _p(hq), _p(hsf), p_cap, _p(toks),
                             toks.size, _p(y), nthreads)
    assert st in (0, 1), st
    return y


def combine(o_pool: np.ndarray, slot_of: np.ndarray, T: int, k: int):
    o = _c(o_pool, np.uint16)
    H = o.shape[1]
    s = _c(slot_of, np.int32)
    y = np.zeros((T, H), np.uint16)
    lib().or_combine(_p(o), _p(s), T, k, H, _p(y))
    return y


def bruteforce_token(x_row_bits, idx_row, w_row, E, w1q, w1sf, w2q, w2sf, activation_clamp: float = 0.0,
                     scale_rule: int = SCALE_RULE_CEIL):
    x = _c(x_row_bits, np.uint16).ravel()
    idx = _c(idx_row, np.int64).ravel()
    w = _c(w_row, np.float32).ravel()
    w1q, w1sf, w2q, w2sf = (_c(a, np.uint8) for a in (w1q, w1sf, w2q, w2sf))
    H = x.size
    I = w2q.shape[2] * 2
    y = np.zeros(H, np.uint16)
    st = lib().or_bruteforce_token(_p(x), _p(idx), _p(w), idx.size, E, H, I, _p(w1q), _p(w1sf),
                                   _p(w2q), _p(w2sf), float(activation_clamp), int(scale_rule), _p(y))
    return y, st


def num_threads() -> int:
    return lib().or_num_threads()
