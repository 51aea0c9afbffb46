"""Per-stage GPU parity: the gathered MXFP8 pool (bit-exact), the L1 output
(requantised h: codes equal to the oracle's), L2 on injected oracle
activations, and combine on injected oracle L2 rows (bit-exact)."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def _plan_and_dispatch(moe, w, d):
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    moe.dispatch(p, d["x"])
    return p


@pytest.mark.parametrize("name", ["tiny", "mid", "decode", "full"])
def test_dispatch_pool_bit_exact(moe, oracle, name):
    w = inputs.WORKLOADS[name]
    d = dict(x=inputs.make_x(w.T, w.H, 0, "cuda"))
    d["topk_idx"], d["topk_w"] = (t.cuda() for t in inputs.make_routing(w, 1))
    p = _plan_and_dispatch(moe, w, d)
    assert moe.plan_check(p) == 0
    xq, xsf = oracle.quant_x(gh.bits(d["x"]))
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    toks = row_token[rows]
    pool = p.export("pool_q").cpu().numpy().reshape(-1, w.H)
    np.testing.assert_array_equal(pool[rows], xq[toks])
    sf = gh.sf_rows_from_mma(p.export("pool_sf").cpu().numpy(), p.export("pool_rows"), w.H)
    np.testing.assert_array_equal(sf[rows], xsf[toks])


@pytest.mark.parametrize("rule", [0, 1])
def test_dispatch_pool_bit_exact_at_extreme_magnitudes(moe, oracle, rule):
    """Token rows scaled by 2^s for s from -140 to +120 (bf16 subnormals, the
    ends of the UE8M0 range where the scale exponent clamps, exact zeros,
    single huge or tiny values inside a block): pool codes and scale bytes
    equal the oracle's under both scale rules."""
    w = inputs.Workload("extreme", 96, 1024, 128, 4, 2, "uniform")
    x = inputs.make_x(w.T, w.H, 5, "cpu").float()
    s = torch.linspace(-140, 120, w.T).round()
    x = x * torch.exp2(s)[:, None]
    x[3] = 0.0                                   # an all-zero row
    x[7, :32] = 0.0                              # an all-zero block
    x[11, 5] = 3.0e38                            # one huge value among ordinary ones
    x[13, 40] = 1.0e-40                          # one bf16 subnormal among ordinary ones
    x[17] = x[17] * 0 + torch.where(torch.arange(w.H) % 2 == 0, 1.0e-38, -1.0e-39)
    d = dict(x=x.to(torch.bfloat16).cuda())
    d["topk_idx"], d["topk_w"] = (t.cuda() for t in inputs.make_routing(w, 1))
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    moe.dispatch(p, d["x"], options=moe.Options(scale_rule=rule))
    assert moe.plan_check(p) == 0
    xq, xsf = oracle.quant_x(gh.bits(d["x"]), scale_rule=rule)
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    toks = row_token[rows]
    pool = p.export("pool_q").cpu().numpy().reshape(-1, w.H)
    np.testing.assert_array_equal(pool[rows], xq[toks])
    sf = gh.sf_rows_from_mma(p.export("pool_sf").cpu().numpy(), p.export("pool_rows"), w.H)
    np.testing.assert_array_equal(sf[rows], xsf[toks])


def _deq_e4m3(codes, sf):
    tab = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    v = tab[codes.astype(np.int64)]
    return v * np.exp2(sf.astype(np.float64) - 127).repeat(32, axis=-1)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_expert_layers_against_oracle_pool(moe, oracle, name):
    w = inputs.WORKLOADS[name]
    d, W1, W2 = gh.setup(moe, w)
    h = gh.host(d)
    p = _plan_and_dispatch(moe, w, d)
    moe.expert_l1(p, W1)
    assert moe.plan_check(p) == 0
    ref = gh.oracle_forward(oracle, h, w.E, want_pool=True)
    cap = p.export("pool_rows")
    row_token = p.export("row_token").cpu().numpy()
    P = int(p.export("poff").cpu().numpy()[-1])
    rows = np.nonzero(row_token[:P] >= 0)[0]
    # L1: requantised SwiGLU*w, E4M3 codes + UE8M0 scales.  Every integer
    # decision is taken by the exact formula, so codes differ only where the
    # fp32 tensor-core accumulation rounds gate/up to another bf16 than the
    # oracle's double sum does (rare).
    hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
    hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), cap, w.I)[rows]
    code_mism = np.mean(hq != ref["hq"][rows])
    sf_mism = np.mean(hsf != ref["hsf"][rows])
    a = _deq_e4m3(hq, hsf)
    b = _deq_e4m3(ref["hq"][rows], ref["hsf"][rows])
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert code_mism <= 1e-5 and sf_mism <= 1e-5 and rel <= 1e-4, (code_mism, sf_mism, rel)

    # L2 on the oracle's own h (injected): bf16 rows in pool order
    hq_all = p.export("h_q").view(-1, w.I)
    inj = np.zeros((cap, w.I), np.uint8)
    inj[rows] = ref["hq"][rows]
    hq_all.copy_(torch.from_numpy(inj).cuda())
    sf_rows = np.full((cap, w.I // 32), 127, np.uint8)
    sf_rows[rows] = ref["hsf"][rows]
    p.export("h_sf").copy_(torch.from_numpy(gh.sf_mma_from_rows(sf_rows)).cuda())
    moe.expert_l2(p, W2)
    assert moe.plan_check(p) == 0
    o = gh.bits(p.export("l2_out").view(-1, w.H))[rows]
    o_ref = ref["o"][rows]
    mism = np.mean(o != o_ref)
    ov, rv = gh.bf16_values(o), gh.bf16_values(o_ref)
    rel2 = np.linalg.norm(ov - rv) / np.linalg.norm(rv)
    assert mism <= 1e-4 and rel2 <= 1e-4, (mism, rel2)

    # combine on the oracle's own L2 rows (injected): bit-exact
    o_inj = np.zeros((cap, w.H), np.uint16)
    o_inj[rows] = o_ref
    p.export("l2_out").view(torch.int16).copy_(torch.from_numpy(o_inj.view(np.int16)).cuda().view(-1))
    y = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    moe.combine(p, y)
    y_ref = oracle.combine(o_inj, p.export("slot_of").cpu().numpy(), w.T, w.k)
    np.testing.assert_array_equal(gh.bits(y), y_ref)
