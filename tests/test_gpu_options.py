"""GPU parity of the layer options (activation clamp, OCP floor scale rule,
fast_math) against the oracle with the same options."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_dispatch_floor_rule_bit_exact(moe, oracle):
    w = inputs.WORKLOADS["mid"]
    x = inputs.make_x(w.T, w.H, 0, "cuda") * 37.0          # wide range: many blocks with amax > 448/2^e
    x = x.to(torch.bfloat16)
    idx, tw = (t.cuda() for t in inputs.make_routing(w, 1))
    p = moe.plan(idx, tw, w.E, w.H, w.I)
    moe.dispatch(p, x, options=moe.Options(scale_rule=moe.SCALE_OCP_FLOOR))
    assert moe.plan_check(p) == 0
    xq, xsf = oracle.quant_x(gh.bits(x), scale_rule=oracle.SCALE_RULE_OCP_FLOOR)
    xq_c, _ = oracle.quant_x(gh.bits(x))
    assert np.mean(xq != xq_c) > 0.01                        # the rule matters on this data
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    toks = row_token[rows]
    pool = p.export("pool_q").cpu().numpy().reshape(-1, w.H)
    np.testing.assert_array_equal(pool[rows], xq[toks])
    sf = gh.sf_rows_from_mma(p.export("pool_sf").cpu().numpy(), p.export("pool_rows"), w.H)
    np.testing.assert_array_equal(sf[rows], xsf[toks])


@pytest.mark.parametrize("name", ["tiny", "mid"])
@pytest.mark.parametrize("clamp,rule", [(0.75, 1), (0.0, 1), (0.75, 0)])
def test_forward_with_options_against_oracle(moe, oracle, name, clamp, rule):
    w = inputs.WORKLOADS[name]
    d, W1, W2 = gh.setup(moe, w)
    h = gh.host(d)
    opts = moe.Options(activation_clamp=clamp, scale_rule=rule)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p, options=opts)
    assert moe.plan_check(p) == 0
    ref = gh.check_forward(oracle, p, y, h, w.E, what=f"y {name} clamp={clamp} rule={rule}",
                           activation_clamp=clamp, scale_rule=rule)
    # the requantised L1 output: codes and scales as the oracle's (up to rare bf16 gate/up differences)
    cap = p.export("pool_rows")
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
    hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), cap, w.I)[rows]
    assert np.mean(hq != ref["hq"][rows]) <= 1e-5
    assert np.mean(hsf != ref["hsf"][rows]) <= 1e-5
    if name == "tiny":  # the options change the result
        base = oracle.forward(h["x"], h["topk_idx"], h["topk_w"], w.E, h["w1q"], h["w1sf"], h["w2q"], h["w2sf"])
        assert not np.array_equal(ref["y"], base["y"])


def test_fast_math_off_gives_the_same_bytes(moe):
    """fast_math=0 computes every SwiGLU value by the exact formula; the fast
    path recomputes exactly wherever an integer decision could change, so both
    give identical requantised activations and outputs."""
    w = inputs.WORKLOADS["mid"]
    d, W1, W2 = gh.setup(moe, w)
    outs = []
    for fast in (1, 0):
        p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
        y = moe.forward(d["x"], W1, W2, p, options=moe.Options(fast_math=fast))
        assert moe.plan_check(p) == 0
        P = int(p.export("poff").cpu().numpy()[-1])
        rows = np.nonzero(p.export("row_token").cpu().numpy()[:P] >= 0)[0]
        hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
        hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), p.export("pool_rows"), w.I)[rows]
        outs.append((gh.bits(y), hq, hsf))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_invalid_options_are_rejected(moe):
    w = inputs.WORKLOADS["tiny"]
    d, W1, W2 = gh.setup(moe, w)
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    for bad in (moe.Options(scale_rule=5), moe.Options(fast_math=2), moe.Options(activation_clamp=-0.5)):
        with pytest.raises(moe.MoeError) as ei:
            moe.forward(d["x"], W1, W2, p, options=bad)
        assert ei.value.status == moe.ERR_INVALID_ARG
    r = moe.Options()
    r.reserved[2] = 1
    with pytest.raises(moe.MoeError):
        moe.expert_l1(p, W1, options=r)
    assert moe.plan_check(p) == 0
