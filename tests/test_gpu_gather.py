"""Layer 1 with its A rows gathered by token from token-major MXFP8 x
(tile::gather4 loads; the "skip the pool" option, moe_options_t.a_operand =
MOE_A_GATHER): dispatch writes each token's codes once, bit-exact to the
oracle's quantisation, and the expert kernel produces the same bytes as with
the expert-major pool."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def _ragged():
    counts = {0: 1, 1: 16, 2: 17, 3: 127, 4: 128, 5: 129, 7: 300}
    flat = np.concatenate([np.full(n, e) for e, n in counts.items()])
    w = inputs.Workload("ragged", flat.size, 384, 256, 8, 1, "uniform")
    idx = np.random.default_rng(4).permutation(flat).reshape(w.T, 1)
    tw = np.random.default_rng(5).random((w.T, 1)).astype(np.float32)
    return w, idx, tw


def _setup(moe, name):
    if name == "ragged":
        w, idx, tw = _ragged()
        d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    else:
        w = inputs.WORKLOADS[name]
        d, W1, W2 = gh.setup(moe, w)
    return w, d, W1, W2


def _outputs(p, w):
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    cap = p.export("pool_rows")
    hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
    hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), cap, w.I)[rows]
    o = gh.bits(p.export("l2_out").view(-1, w.H))[rows]
    return hq, hsf, o


@pytest.mark.parametrize("name", ["tiny", "mid", "ragged", "decode", "share"])
def test_gathered_rows_give_the_pool_results(moe, oracle, name):
    w, d, W1, W2 = _setup(moe, name)
    pool_opts, gather_opts = moe.Options(), moe.Options(a_operand=moe.A_GATHER)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y_pool = moe.forward(d["x"], W1, W2, p, options=pool_opts)
    assert moe.plan_check(p) == 0
    ref = _outputs(p, w)
    # gathered: fused kernel (moe_forward) and the layer-1 kernel alone
    p.export("pool_q").fill_(0xAA)        # the gathered path must not read the pool's codes
    p.export("h_q").zero_()
    p.export("l2_out").zero_()
    y_gather = moe.forward(d["x"], W1, W2, p, options=gather_opts)
    assert moe.plan_check(p) == 0
    for a, b, what in zip(_outputs(p, w), ref, ("h codes", "h scales", "L2 rows")):
        np.testing.assert_array_equal(a, b, err_msg=f"{name} fused: {what}")
    np.testing.assert_array_equal(gh.bits(y_gather), gh.bits(y_pool))
    p.export("h_q").zero_()
    moe.expert_l1(p, W1, options=gather_opts)
    assert moe.plan_check(p) == 0
    np.testing.assert_array_equal(_outputs(p, w)[0], ref[0], err_msg=f"{name} layer 1 alone")
    # the token-major codes are the oracle's quantisation of x, bit for bit
    if name in ("tiny", "mid", "ragged"):
        xq, _ = oracle.quant_x(gh.bits(d["x"]))
        np.testing.assert_array_equal(p.export("x_q").cpu().numpy().reshape(w.T, w.H), xq)


def test_gathered_forward_against_oracle(moe, oracle):
    w, d, W1, W2 = _setup(moe, "ragged")
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p, options=moe.Options(a_operand=moe.A_GATHER))
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="gathered A rows")
