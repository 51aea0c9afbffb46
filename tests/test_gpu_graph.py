"""The layer replays from a CUDA graph: plan + forward are captured once
(no host synchronisation, no allocation inside the library) and replayed on
new inputs copied into the captured buffers; outputs equal eager calls."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_plan_and_forward_replay_from_a_cuda_graph(moe, name):
    w = inputs.WORKLOADS[name]
    d, W1, W2 = gh.setup(moe, w, seed=0)
    ws = moe.alloc_workspace(w.T, w.k, w.E, w.H, w.I)
    sx, sidx, stw = d["x"].clone(), d["topk_idx"].clone(), d["topk_w"].clone()
    sy = torch.empty_like(sx)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (first-call set-up happens here)
        p = moe.plan(sidx, stw, w.E, w.H, w.I, workspace=ws)
        moe.forward(sx, W1, W2, p, sy)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        p = moe.plan(sidx, stw, w.E, w.H, w.I, workspace=ws)
        moe.forward(sx, W1, W2, p, sy)
    for seed in (1, 2):
        d2 = inputs.make_inputs(w, seed=seed, device="cuda")
        sx.copy_(d2["x"]); sidx.copy_(d2["topk_idx"]); stw.copy_(d2["topk_w"])
        g.replay()
        torch.cuda.synchronize()
        assert moe.plan_check(p) == 0
        eager = moe.forward(d2["x"], W1, W2, moe.plan(d2["topk_idx"], d2["topk_w"], w.E, w.H, w.I))
        np.testing.assert_array_equal(gh.bits(sy), gh.bits(eager))
