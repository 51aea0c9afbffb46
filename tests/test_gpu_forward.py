"""End-to-end GPU forward against the oracle: all rows on the small
workloads, sampled tokens at full size, and the degenerate cases."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def run(moe, w, d, W1, W2):
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p)
    return p, y


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_forward_all_tokens(moe, oracle, name):
    w = inputs.WORKLOADS[name]
    d, W1, W2 = gh.setup(moe, w)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what=name)


@pytest.mark.parametrize("name", ["share", "full", "decode"])
def test_forward_sampled_tokens_full_size(moe, oracle, name):
    w = inputs.WORKLOADS[name]
    d, W1, W2 = gh.setup(moe, w)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    h = gh.host(d)
    rng = np.random.default_rng(0)
    toks = np.unique(np.concatenate([[0, 1, w.T - 1], rng.choice(w.T, 29, replace=False)])).astype(np.int32)
    if name == "share":  # include tokens with no local expert (y must be 0)
        none = np.nonzero((h["topk_idx"] < 0).all(1))[0][:3]
        toks = np.unique(np.concatenate([toks, none])).astype(np.int32)
    ref = gh.check_forward(oracle, p, y, h, w.E, tokens=toks, what=name)
    yb = gh.bits(y)[toks]
    # the requantised L1 output of the sampled tokens' pool rows, code by code
    # (wide ring, 128-row A boxes and the full-size layer-1 epilogue here;
    # the narrow ring on decode): the same bar as on the small workloads
    slots = p.export("slot_of").cpu().numpy().reshape(w.T, w.k)[toks]
    rows = slots[slots >= 0]
    hq = p.export("h_q").cpu().numpy().reshape(-1, w.I)[rows]
    hsf = gh.sf_rows_from_mma(p.export("h_sf").cpu().numpy(), p.export("pool_rows"), w.I)[rows]
    assert rows.size > 0
    assert np.mean(hq != ref["hq"][rows]) <= 1e-5 and np.mean(hsf != ref["hsf"][rows]) <= 1e-5
    if name == "share":
        for t in np.nonzero((h["topk_idx"][toks] < 0).all(1))[0]:
            assert np.all(yb[t] == 0)
    # output rows are finite everywhere
    assert torch.isfinite(y.float()).all()


def test_forward_deterministic(moe):
    w = inputs.WORKLOADS["mid"]
    d, W1, W2 = gh.setup(moe, w)
    _, y1 = run(moe, w, d, W1, W2)
    _, y2 = run(moe, w, d, W1, W2)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_forward_edge_routings(moe, oracle):
    w = inputs.Workload("edge", 512, 256, 128, 8, 4, "uniform")
    rng = np.random.default_rng(3)
    cases = {}
    # one expert gets every entry (duplicates inside a token)
    cases["one_expert"] = np.full((w.T, w.k), 3)
    # experts with 0, 1, 127, 128, 129 rows
    flat = np.concatenate([np.full(n, e) for e, n in {1: 1, 2: 127, 3: 128, 4: 129}.items()])
    flat = np.concatenate([flat, np.full(w.T * w.k - flat.size, -1)])
    cases["ragged"] = rng.permutation(flat).reshape(w.T, w.k)
    # all entries skipped
    cases["none"] = -np.ones((w.T, w.k))
    for name, idx in cases.items():
        tw = rng.random((w.T, w.k)).astype(np.float32)
        d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
        p, y = run(moe, w, d, W1, W2)
        assert moe.plan_check(p) == 0
        gh.check_forward(oracle, p, y, gh.host(d), w.E, what=name)
        if name == "none":
            assert torch.all(y.view(torch.int16) == 0)


def test_bad_expert_ids_reported(moe, oracle):
    w = inputs.WORKLOADS["tiny"]
    idx, tw = inputs.make_routing(w)
    idx = idx.clone()
    idx[5, 1] = w.E          # out of range: skipped and reported
    idx[9, 0] = -3
    d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == moe.ERR_BAD_EXPERT_ID
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="bad ids")


def test_empty_batch_forward(moe):
    w = inputs.Workload("empty", 0, 256, 128, 8, 2, "uniform")
    d, W1, W2 = gh.setup(moe, inputs.Workload("w", 4, 256, 128, 8, 2, "uniform"))
    idx = torch.zeros(0, 2, dtype=torch.int64, device="cuda")
    tw = torch.zeros(0, 2, dtype=torch.float32, device="cuda")
    p = moe.plan(idx, tw, w.E, w.H, w.I)
    y = torch.empty(0, w.H, dtype=torch.bfloat16, device="cuda")
    moe.forward(torch.empty(0, w.H, dtype=torch.bfloat16, device="cuda"), W1, W2, p, y)
    assert moe.plan_check(p) == 0


def test_odd_h_tail_tile(moe, oracle):
    """H = 384: the last L2 output tile holds 128 valid columns of 256."""
    w = inputs.Workload("oddH", 96, 384, 256, 4, 2, "uniform")
    d, W1, W2 = gh.setup(moe, w)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="oddH")


def test_largest_expert_count_and_topk(moe, oracle):
    """E = 1024 experts and k = 32 (the library's limits): most experts get one
    or two rows, so nearly every pool block is a 16-row-A block, and combine
    sums 32 entries per token."""
    w = inputs.Workload("maxEk", 64, 256, 128, 1024, 32, "uniform")
    d, W1, W2 = gh.setup(moe, w)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="E=1024 k=32")


def test_partial_blocks_on_every_a_box_size(moe, oracle):
    """A block loads the smallest A box (16, 32, 64 or 128 rows) that holds its
    valid rows; counts on both sides of each switch, and 144 = 128 + 16 for a
    second block."""
    counts = {0: 16, 1: 17, 2: 32, 3: 33, 4: 64, 5: 65, 6: 144, 7: 100}
    flat = np.concatenate([np.full(n, e) for e, n in counts.items()])
    w = inputs.Workload("boxes", flat.size, 256, 128, len(counts), 1, "uniform")
    idx = np.random.default_rng(5).permutation(flat).reshape(w.T, 1)
    tw = np.full((w.T, 1), 0.5, np.float32)
    d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what="partial blocks")


@pytest.mark.parametrize("largest,H", [(16, 1024), (17, 1024), (16, 384)])
def test_ring_shape_switch(moe, oracle, largest, H):
    """With no expert above 16 rows the GEMMs run the 6-stage narrow ring
    (16-row A stages), otherwise the 4-stage wide ring: 200 experts of 1 to 16
    rows plus one of `largest`, H = 1024 (8 k-blocks per L1 tile) so that each
    CTA's ring wraps several times over its tiles; H = 384 adds a half-empty
    last L2 output tile to the narrow ring."""
    rng = np.random.default_rng(11)
    counts = rng.integers(1, 17, size=200)
    counts[0] = 16
    counts[1] = largest
    flat = np.concatenate([np.full(n, e) for e, n in enumerate(counts)])
    w = inputs.Workload("ring", flat.size, H, 256, counts.size, 1, "uniform")
    idx = rng.permutation(flat).reshape(w.T, 1)
    tw = np.full((w.T, 1), 0.75, np.float32)
    d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw)
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    assert int(p.export("max_count").cpu()[0]) == largest
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what=f"ring, largest count {largest}, H {H}")


def test_forward_per_token_scales(moe, oracle):
    """Token rows scaled by 2^s for s from -40 to +30 (the UE8M0 scales of x,
    the accumulators and the requantised h all move with them, within fp32
    range): every token's output agrees with the oracle's, token by token
    (relative L2 <= 5e-3 each), so no scale is clamped or lost on the way."""
    w = inputs.Workload("scaled", 96, 1024, 256, 4, 2, "uniform")
    d, W1, W2 = gh.setup(moe, w)
    s = torch.linspace(-40, 30, w.T, device="cuda").round()
    d["x"] = (d["x"].float() * torch.exp2(s)[:, None]).to(torch.bfloat16).contiguous()
    p, y = run(moe, w, d, W1, W2)
    assert moe.plan_check(p) == 0
    h = gh.host(d)
    ref = gh.oracle_forward(oracle, h, w.E)["y"]
    a = torch.from_numpy(gh.bits(y).view(np.int16)).view(torch.bfloat16).double()
    b = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double()
    rel = (torch.linalg.norm(a - b, dim=1) / torch.linalg.norm(b, dim=1).clamp_min(1e-300))
    assert torch.isfinite(a).all()
    assert rel.max().item() <= 5e-3, (rel.argmax().item(), rel.max().item())
