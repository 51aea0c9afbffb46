"""The expert-offsets entry point that allocates nothing.

Some callers of this library cannot call cudaMalloc: a plugin running inside a
host framework that owns all device memory, or a serving loop whose memory
budget is fixed after start-up.  They cannot hand moe_plan() a workspace, so
moe_expert_offsets_static() computes the same per-expert counts, offsets and
row-block-padded offsets with scratch kept in a fixed array inside the
library.  This test calls it through the C ABI on two different routings in a
row (and the first again), and checks every result against the tables that
moe_plan() computes with a workspace; the results are integers, so they must
be equal.  It is collected last and also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def _offsets_static(moe, idx, E):
    L = moe.lib()
    T, k = idx.shape
    count = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    poff = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    rc = L.moe_expert_offsets_static(ctypes.c_void_p(idx.data_ptr()), T, k, E, ctypes.c_void_p(count.data_ptr()),
                                     ctypes.c_void_p(off.data_ptr()), ctypes.c_void_p(poff.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == moe.OK, moe.error_string(rc)
    torch.cuda.synchronize()
    return count.cpu().numpy(), off.cpu().numpy(), poff.cpu().numpy()


def _with_workspace(moe, idx, tw, E):
    p = moe.plan(idx, tw, E, 256, 128)
    assert moe.plan_check(p) == 0
    return p.export("count").cpu().numpy(), p.export("off").cpu().numpy(), p.export("poff").cpu().numpy()


def test_offsets_static_matches_plan_on_consecutive_calls(moe):
    runs = []
    for name in ("full", "mid", "full"):
        w = inputs.WORKLOADS[name]
        idx, tw = (t.cuda() for t in inputs.make_routing(w))
        got = _offsets_static(moe, idx, w.E)
        want = _with_workspace(moe, idx, tw, w.E)
        for g, r in zip(got, want):
            np.testing.assert_array_equal(g, r)
        runs.append(got)
    for g, r in zip(runs[0], runs[2]):
        np.testing.assert_array_equal(g, r)


def _oracle_tables(oracle, idx_np, E):
    r = oracle.plan(idx_np, np.ones(idx_np.shape, np.float32), E)
    return r["count"], r["off"], r["poff"]


def test_offsets_static_edge_cases_against_oracle(moe, oracle):
    """Edge cases, compared directly with the oracle's plan (which skips every
    id outside [0, E)): an empty batch, one expert, ids of -1 and ids out of
    range (skipped here without a report), a single entry, and a batch that
    fits one routing chunk next to one that needs several."""
    rng = np.random.default_rng(17)
    cases = []
    cases.append(("T=0", np.zeros((0, 4), np.int64), 8))
    cases.append(("E=1", np.zeros((300, 2), np.int64), 1))
    bad = rng.integers(0, 16, (500, 3)).astype(np.int64)
    bad[rng.random(bad.shape) < 0.2] = -1
    bad[3, 1], bad[77, 0], bad[400, 2] = 16, -2, 1 << 40
    cases.append(("bad ids", bad, 16))
    cases.append(("one entry", np.array([[5]], np.int64), 6))
    cases.append(("one chunk", rng.integers(0, 40, (256, 8)).astype(np.int64), 40))
    cases.append(("many chunks", rng.integers(-1, 300, (4000, 6)).astype(np.int64), 300))
    for name, idx_np, E in cases:
        idx = torch.from_numpy(idx_np).cuda()
        got = _offsets_static(moe, idx, E)
        want = _oracle_tables(oracle, idx_np, E)
        for g, r in zip(got, want):
            np.testing.assert_array_equal(g, r, err_msg=name)


def test_offsets_static_rejects_sizes_beyond_its_scratch(moe):
    L = moe.lib()
    idx = torch.zeros(1, 1, dtype=torch.int64, device="cuda")
    out = torch.zeros(2048, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(out.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # more than 262144 entries, and more than 32768 chunk-expert cells
    assert L.moe_expert_offsets_static(ctypes.c_void_p(idx.data_ptr()), 300000, 1, 8, p, p, p, s) == moe.ERR_TOO_LARGE
    assert L.moe_expert_offsets_static(ctypes.c_void_p(idx.data_ptr()), 65536, 2, 1024, p, p, p, s) == moe.ERR_TOO_LARGE
    assert "fixed scratch" in moe.error_string(moe.ERR_TOO_LARGE)
