"""Forward parity on a spread of small shapes: hidden and intermediate sizes of
1 to 11 multiples of 128 (odd counts leave a half-empty last L2 output tile),
expert counts from 1 to 300, top-k from 1 to 12, uniform and Zipf-skewed
routing, and some entries not routed (-1).  Every token against the oracle."""
import numpy as np
import pytest

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu

# (T, H, I, E, k, router, fraction of entries set to -1)
SHAPES = [
    (40, 128, 128, 1, 1, "uniform", 0.0),
    (77, 384, 640, 5, 3, "zipf", 0.0),
    (130, 640, 384, 16, 4, "uniform", 0.2),
    (200, 1408, 256, 300, 12, "uniform", 0.0),
    (300, 256, 1152, 24, 2, "zipf", 0.5),
    (513, 896, 128, 7, 7, "zipf", 0.1),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s[0]}H{s[1]}I{s[2]}E{s[3]}k{s[4]}{s[5]}" for s in SHAPES])
def test_forward_shape(moe, oracle, shape):
    T, H, I, E, k, router, drop = shape
    w = inputs.Workload("shape", T, H, I, E, k, router)
    idx, tw = inputs.make_routing(w, seed=7)
    idx = idx.numpy().copy()
    if drop:
        rng = np.random.default_rng(3)
        idx[rng.random(idx.shape) < drop] = -1
    d, W1, W2 = gh.setup(moe, w, idx=idx, tw=tw.numpy())
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    y = moe.forward(d["x"], W1, W2, p)
    assert moe.plan_check(p) == 0
    gh.check_forward(oracle, p, y, gh.host(d), w.E, what=f"shape {shape}")
