"""The fused expert kernel (both layers in one persistent launch, layer-2
tiles gated by per-row-block readiness counters): the same bytes as the two
separate launches, and a bounded wait that expires cleanly."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def _valid_rows(p):
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    return np.nonzero(row_token[:P] >= 0)[0]


def _expert_outputs(p, w):
    rows = _valid_rows(p)
    cap = p.export("pool_rows")
    hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
    hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), cap, w.I)[rows]
    o = gh.bits(p.export("l2_out").view(-1, w.H))[rows]
    return hq, hsf, o


def _ragged_case():
    """Experts of 1, 16, 17, 127, 128, 129, 300 rows and an empty one (the wide
    ring, partly filled blocks of every A box size, blocks spanning experts)."""
    counts = {0: 1, 1: 16, 2: 17, 3: 127, 4: 128, 5: 129, 7: 300}
    flat = np.concatenate([np.full(n, e) for e, n in counts.items()])
    w = inputs.Workload("ragged", flat.size, 384, 256, 8, 1, "uniform")
    idx = np.random.default_rng(2).permutation(flat).reshape(w.T, 1)
    tw = np.random.default_rng(3).random((w.T, 1)).astype(np.float32)
    return w, idx, tw


@pytest.mark.parametrize("name", ["tiny", "mid", "ragged", "decode", "share", "full"])
def test_fused_equals_two_launches(moe, name):
    """h codes, h scales and the bf16 L2 rows of every routed pool row are
    bit-identical between moe_expert_fused and moe_expert_l1 + moe_expert_l2
    (the same arithmetic in the same order; only the scheduling differs)."""
    if name == "ragged":
        w, idx, tw = _ragged_case()
        d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    else:
        w = inputs.WORKLOADS[name]
        d, W1, W2 = gh.setup(moe, w)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    moe.dispatch(p, d["x"])
    moe.expert_l1(p, W1)
    moe.expert_l2(p, W2)
    assert moe.plan_check(p) == 0
    sep = _expert_outputs(p, w)
    p.export("h_q").zero_()
    p.export("l2_out").zero_()
    moe.expert_fused(p, W1, W2)
    assert moe.plan_check(p) == 0
    fused = _expert_outputs(p, w)
    for a, b, what in zip(fused, sep, ("h codes", "h scales", "L2 rows")):
        np.testing.assert_array_equal(a, b, err_msg=f"{name}: {what}")


def test_fused_forward_ragged_against_oracle(moe, oracle):
    w, idx, tw = _ragged_case()
    d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="ragged fused forward")


def test_fused_wait_expires_cleanly_and_context_stays_usable(moe, oracle):
    """No row block ever becomes ready: every layer-2 tile's bounded wait runs
    out after 1 s, the launch records MOE_ERR_TIMEOUT (where = a layer-2 tile
    waiting on its block) and exits without a fault; the next forward on the
    same context matches the oracle."""
    w = inputs.WORKLOADS["tiny"]
    d, W1, W2 = gh.setup(moe, w)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    moe.dispatch(p, d["x"])
    moe.selftest_fused_wait(p, W1, W2)
    assert moe.plan_check(p) == moe.ERR_TIMEOUT
    err = p.export("error").cpu().numpy()
    assert err[1] == 1 + 80, err
    p2 = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p2)
    assert moe.plan_check(p2) == 0
    gh.check_forward(oracle, p2, y, gh.host(d), w.E, what="after time-out")
