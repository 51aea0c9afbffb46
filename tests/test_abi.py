"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-only entry points answer without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libmoe():
    from moe_expert_layer_counts_gb300 import build as b
    b.build()
    return ctypes.CDLL(b.LIB)


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"^\s*(?:size_t|int|const char\*)\s+(moe_\w+)\s*\(", txt, flags=re.M))
    return sorted(names)


def test_exports_every_declared_symbol(libmoe):
    import moe_expert_layer_counts_gb300 as m
    names = header_functions()
    assert len(names) >= 12
    assert set(names) == set(m.SYMBOLS)
    for n in names:
        assert hasattr(libmoe, n), n


def test_host_only_sizes(libmoe):
    f = libmoe.moe_plan_workspace_bytes
    f.restype = ctypes.c_size_t
    full = f(8192, 8, 256, 7168, 2048)
    assert full > 2 * 10 ** 9
    assert f(0, 8, 256, 7168, 2048) > 0          # empty batch is valid
    assert f(64, 2, 8, 256, 128) < full
    for bad in [(64, 0, 8, 256, 128), (64, 33, 8, 256, 128), (64, 2, 0, 256, 128), (64, 2, 2000, 256, 128),
                (64, 2, 8, 200, 128), (64, 2, 8, 256, 100), (-1, 2, 8, 256, 128)]:
        assert f(*bad) == 0, bad
    g = libmoe.moe_weight_scales_bytes
    g.restype = ctypes.c_size_t
    assert g(256, 4096, 7168) == 256 * 32 * 56 * 512
    assert g(1, 100, 128) == 0


def test_argument_errors_before_any_device_call(libmoe):
    libmoe.moe_plan.restype = ctypes.c_int
    libmoe.moe_plan.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_size_t,
                                                                               ctypes.c_void_p]
    assert libmoe.moe_plan(None, None, None, 4, 2, 8, 256, 128, None, 0, None) == 1  # MOE_ERR_INVALID_ARG
    plan = ctypes.create_string_buffer(192)
    # misaligned workspace pointer
    assert libmoe.moe_plan(plan, 16, 16, 4, 2, 8, 256, 128, 8, 1 << 30, None) == 1
    # unsupported shape
    assert libmoe.moe_plan(plan, 16, 16, 4, 2, 8, 200, 128, 256, 1 << 30, None) == 2
    # workspace too small
    assert libmoe.moe_plan(plan, 16, 16, 4, 2, 8, 256, 128, 256, 16, None) == 3
    libmoe.moe_forward.restype = ctypes.c_int
    libmoe.moe_forward.argtypes = [ctypes.c_void_p] * 7
    assert libmoe.moe_forward(None, None, None, plan, None, None, None) == 1  # plan never filled
    # options out of range are rejected before any device call
    import moe_expert_layer_counts_gb300 as moe
    assert ctypes.sizeof(moe.Options) == 32
    for bad in (moe.Options(scale_rule=2), moe.Options(fast_math=3), moe.Options(activation_clamp=-1.0),
                moe.Options(activation_clamp=float("nan")), moe.Options(a_operand=2)):
        assert libmoe.moe_forward(None, None, None, plan, None, ctypes.addressof(bad), None) == 1
    libmoe.moe_error_string.restype = ctypes.c_char_p
    for s in range(8):
        assert libmoe.moe_error_string(s)


def test_selftest_argument_errors_without_a_device(libmoe):
    """The calibration self-tests check their arguments before touching the
    device: null, misaligned or out-of-range arguments are MOE_ERR_INVALID_ARG."""
    f = libmoe.moe_selftest_stream_rate
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int),
                                          ctypes.c_void_p]
    ctas = ctypes.c_int(0)
    ok = 1 << 20  # any 16-byte aligned address; never dereferenced on these paths
    assert f(None, ok, ok, ok, 16, ok, ctypes.byref(ctas), None) == 1
    assert f(ok, ok, ok, ok + 8, 16, ok, ctypes.byref(ctas), None) == 1   # misaligned scale pointer
    assert f(ok, ok, ok, ok, 0, ok, ctypes.byref(ctas), None) == 1        # no k-blocks
    assert f(ok, ok, ok, ok, (1 << 20) + 1, ok, ctypes.byref(ctas), None) == 1
    assert f(ok, ok, ok, ok, 16, None, ctypes.byref(ctas), None) == 1     # no status word
    g = libmoe.moe_selftest_mma_rate
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.c_void_p]
    assert g(0, ok, ctypes.byref(ctas), None) == 1
    assert g(16, None, ctypes.byref(ctas), None) == 1


def test_debug_build_exports_the_same_symbols():
    """The MOE_DEBUG variant (device bounds checks on plan tables) builds for
    sm_103a and exports exactly what include/moe.h declares."""
    from moe_expert_layer_counts_gb300 import build as b
    lib = ctypes.CDLL(b.build(debug=True))
    for n in header_functions():
        assert hasattr(lib, n), n
    lib.moe_error_string.restype = ctypes.c_char_p
    assert b"debug" in lib.moe_error_string(9)
