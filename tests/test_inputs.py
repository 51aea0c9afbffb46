"""The seeded input generators produce the workloads' shapes and statistics."""
import numpy as np
import torch

from moe_expert_layer_counts_gb300 import inputs


def test_weights_distribution(oracle):
    """Gaussian weights N(0, 1/sqrt(K)) quantised to MXFP4: the bytes equal the
    oracle's own MX E2M1 quantiser (an independent implementation) applied to
    the same Gaussian draw, the dequantised weights have the configured
    spread, and every 32-block's largest magnitude maps to code 5, 6 or 7 (a
    value in (3, 6] after the ceil scale rule)."""
    K, N, E = 2048, 64, 2
    q, sf = inputs.make_weights(E, N, K, seed=0)
    assert q.shape == (E, N, K // 2) and sf.shape == (E, N, K // 32)
    g = torch.Generator().manual_seed(0)
    for e in range(E):
        w = torch.randn(N, K, generator=g, dtype=torch.float32) / np.sqrt(K)
        nib, osf = oracle.quant_mx_e2m1(w.numpy())
        packed = nib.reshape(N, K)[:, 0::2] | (nib.reshape(N, K)[:, 1::2] << 4)
        np.testing.assert_array_equal(q[e].numpy(), packed)
        np.testing.assert_array_equal(sf[e].numpy().ravel(), osf)
    tab = np.array([oracle.e2m1_decode(c) for c in range(16)])
    qn = q.numpy()
    nib = np.stack([qn & 15, qn >> 4], -1).reshape(E, N, K)
    scale = np.exp2(sf.numpy().astype(np.float64) - 127).repeat(32, -1)
    wq = tab[nib] * scale
    assert abs(wq.std() * np.sqrt(K) - 1.0) < 0.05, wq.std() * np.sqrt(K)
    assert abs(wq.mean()) < 0.05 / np.sqrt(K)
    top = (nib & 7).reshape(E, N, K // 32, 32).max(-1)
    assert top.min() >= 5
    # same seed, same bytes
    q2, sf2 = inputs.make_weights(E, N, K, seed=0)
    assert torch.equal(q, q2) and torch.equal(sf, sf2)


def test_quantize_mxfp4_ties_and_signs(oracle):
    """Rounding ties go to the even E2M1 code, negative values (and a value
    that rounds to zero from below) carry the sign bit, an all-zero block has
    scale byte 127: the same bytes as the oracle's codec."""
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    row = np.concatenate([ties, -ties, np.array([-0.1, 0.1, 0.0, -0.0] + [0.0] * 12, np.float32)])
    w = torch.from_numpy(np.stack([row, np.zeros(32, np.float32)]))
    q, sf = inputs.quantize_mxfp4(w)
    nib, osf = oracle.quant_mx_e2m1(w.numpy())
    np.testing.assert_array_equal(q.numpy(), (nib.reshape(2, 32)[:, 0::2] | (nib.reshape(2, 32)[:, 1::2] << 4)))
    np.testing.assert_array_equal(sf.numpy().ravel(), osf)
    assert sf[1, 0] == 127


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
