"""The seeded input generators produce the workloads' shapes and statistics."""
import numpy as np
import torch

from moe_expert_layer_counts_gb300 import inputs


def test_weights_distribution(oracle):
    K = 2048
    q, sf = inputs.make_weights(2, 64, K, seed=0)
    assert q.shape == (2, 64, K // 2) and sf.shape == (2, 64, K // 32)
    tab = np.array([oracle.e2m1_decode(c) for c in range(16)])
    qn = q.numpy()
    nib = np.stack([qn & 15, qn >> 4], -1).reshape(2, 64, K)
    scale = np.exp2(sf.numpy().astype(np.float64) - 127).repeat(32, -1)
    w = tab[nib] * scale
    assert abs(w.std() * np.sqrt(K) - 1.0) < 0.05, w.std() * np.sqrt(K)
    assert abs(w.mean()) < 0.05 / np.sqrt(K)
    s0, p_up = inputs.weight_exponent_recipe(K)
    assert set(np.unique(sf.numpy())) <= {127 + s0, 128 + s0}
    # same seed, same bytes
    q2, sf2 = inputs.make_weights(2, 64, K, seed=0)
    assert torch.equal(q, q2) and torch.equal(sf, sf2)


def test_routing_workloads():
    for name in ("tiny", "mid", "full", "decode", "share"):
        w = inputs.WORKLOADS[name]
        idx, tw = inputs.make_routing(w)
        assert idx.shape == (w.T, w.k) and tw.shape == (w.T, w.k)
        if name == "share":
            assert idx.min() >= -1 and idx.max() < w.E
            frac = (idx >= 0).float().mean().item()
            assert 0.08 < frac < 0.17, frac
        else:
            assert idx.min() >= 0 and idx.max() < w.E
            assert torch.all(torch.sort(idx, dim=1).values.diff(dim=1) > 0)  # distinct per token
            assert torch.allclose(tw.sum(1), torch.ones(w.T), atol=1e-5)
    full = inputs.WORKLOADS["full"]
    idx, _ = inputs.make_routing(full)
    counts = torch.bincount(idx.reshape(-1), minlength=full.E)
    assert counts.max() > 0.9 * full.T  # Zipf bias: one expert takes nearly every token
    assert (counts > 0).sum() < full.E
