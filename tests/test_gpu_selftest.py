"""Failure detection without a GPU fault: the library's bounded mbarrier wait
gives up at its deadline and reports MOE_ERR_TIMEOUT, and the context stays
usable afterwards."""
import pytest

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_completes_when_arrived(moe):
    st, us = moe.selftest_bounded_wait(True, 1_000_000_000)
    assert st == moe.OK
    assert 15 <= us < 100_000


def test_bounded_wait_times_out_and_context_stays_usable(moe, oracle):
    st, us = moe.selftest_bounded_wait(False, 20_000_000)   # 20 ms, nothing arrives
    assert st == moe.ERR_TIMEOUT
    assert 20_000 <= us < 500_000
    # the GPU context is still good: a full forward runs and matches the oracle
    w = inputs.WORKLOADS["tiny"]
    d, W1, W2 = gh.setup(moe, w)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E)


def test_bounded_wait_argument_checks(moe):
    for args in ((True, 0), (True, 3_000_000_000)):
        with pytest.raises(moe.MoeError):
            moe.selftest_bounded_wait(*args)


def test_mma_rate_calibration(moe):
    """The block-scaled MMA ceiling kernel completes (status OK) on every SM and
    reports a rate in the plausible band of this GPU's FP8 tensor pipe."""
    tflops, ctas, ms = moe.selftest_mma_rate(kblocks=2048, repeats=1)
    assert ctas >= 100
    assert 1000.0 < tflops < 20000.0, tflops
    with pytest.raises(moe.MoeError):
        moe.selftest_mma_rate(kblocks=0)


def test_stream_rate_calibration(moe):
    """The operand-stream ceiling kernel (the GEMM tile's TMA ring, scale
    copies and MMAs, no epilogue) completes with status OK on every SM, at a
    rate no higher than the bare MMA ceiling allows."""
    mma, _, _ = moe.selftest_mma_rate(kblocks=2048, repeats=1)
    tflops, ctas, ms = moe.selftest_stream_rate(kblocks=1024, repeats=1)
    assert ctas >= 100
    assert 500.0 < tflops < 1.1 * mma, (tflops, mma)
    with pytest.raises(moe.MoeError):
        moe.selftest_stream_rate(kblocks=0)
