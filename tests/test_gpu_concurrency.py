"""Several host threads use the library at once, each with its own stream
and workspace: plans and forwards of different batches overlap on the GPU.
None of the library's kernels needs its CTAs to be resident together (a
waiting CTA of the plan takes untaken chunks itself; a layer-2 tile of the
fused expert kernel only waits on layer-1 tiles held by running CTAs), so
two fused launches that share the SMs finish, and every output equals the
same forward run alone."""
import threading

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_concurrent_streams_and_threads(moe):
    w = inputs.WORKLOADS["mid"]
    d, W1, W2 = gh.setup(moe, w, seed=0)
    batches = [inputs.make_inputs(w, seed=s, device="cuda") for s in (1, 2, 3)]
    # each batch alone, one after another
    alone = []
    for b in batches:
        p = moe.plan(b["topk_idx"], b["topk_w"], w.E, w.H, w.I)
        alone.append(gh.bits(moe.forward(b["x"], W1, W2, p)))
        assert moe.plan_check(p) == moe.OK
    torch.cuda.synchronize()
    results, errors = [None] * len(batches), []

    def worker(i):
        try:
            b = batches[i]
            s = torch.cuda.Stream()
            ws = moe.alloc_workspace(w.T, w.k, w.E, w.H, w.I)
            y = torch.empty_like(b["x"])
            with torch.cuda.stream(s):
                for _ in range(4):  # back-to-back steps keep the launches of the threads overlapping
                    p = moe.plan(b["topk_idx"], b["topk_w"], w.E, w.H, w.I, workspace=ws, stream=s)
                    moe.forward(b["x"], W1, W2, p, y, stream=s)
            st = moe.plan_check(p, stream=s)
            results[i] = (st, gh.bits(y))
        except Exception as e:  # reported in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(batches))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (st, y) in enumerate(results):
        assert st == moe.OK, (i, moe.error_string(st))
        np.testing.assert_array_equal(y, alone[i])
