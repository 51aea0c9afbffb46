"""Pins of the oracle's layer options: the OCP MX "floor" scale rule (closed
forms, saturation, torch's E4M3 cast for the in-range codes), the activation
clamp (dense special case rebuilt with torch ops), and the brute-force
restatement with both options on."""
import math

import numpy as np
import pytest
import torch

from test_oracle_ffn import _bits, _deq_w, _golden_e2m1, _small


def test_floor_rule_closed_forms(oracle):
    # 448 = 1.75 * 2^8: floor(log2(448 * 2^n)) - 8 = n
    for n in range(-30, 31):
        assert oracle.ue8m0_floor(448.0 * 2.0 ** n, 8) == 127 + n
        # 6 = 1.5 * 2^2 for E2M1
        assert oracle.ue8m0_floor(6.0 * 2.0 ** n, 2) == 127 + n
    for m in range(-40, 41):
        assert oracle.ue8m0_floor(2.0 ** m, 8) == 127 + m - 8
        assert oracle.ue8m0_floor(math.nextafter(2.0 ** m, 0.0), 8) == 127 + m - 9
    assert oracle.ue8m0_floor(0.0, 8) == 127
    assert oracle.ue8m0_floor(2.0 ** -140, 8) == 1      # clamped at 2^-126
    assert oracle.ue8m0_floor(2.0 ** 200, 8) == 254     # clamped at 2^127


def test_floor_rule_differs_from_ceil_and_saturates(oracle):
    v = np.zeros(32, np.float32)
    v[0] = 500.0          # floor(log2 500) = 8 -> scale 2^0; 500 saturates to 448
    v[1] = -3.0
    v[2] = 0.3
    codes, sf = oracle.quant_mx_e4m3(v, scale_rule=oracle.SCALE_RULE_OCP_FLOOR)
    assert sf[0] == 127
    assert codes[0] == 0x7E                   # +448
    ref = torch.from_numpy(v[1:]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes[1:], ref)
    # the ceil rule takes 2^1 instead, nothing saturates
    codes_c, sf_c = oracle.quant_mx_e4m3(v, scale_rule=oracle.SCALE_RULE_CEIL)
    assert sf_c[0] == 128
    ref_c = torch.from_numpy(v / 2.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes_c, ref_c)


def test_floor_rule_random_blocks_against_torch(oracle):
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(32 * 64) * np.exp2(rng.integers(-20, 20, size=32 * 64))).astype(np.float32)
    codes, sf = oracle.quant_mx_e4m3(v, scale_rule=oracle.SCALE_RULE_OCP_FLOOR)
    for b in range(64):
        blk = v[32 * b:32 * b + 32].astype(np.float64)
        amax = np.abs(blk).max()
        e = math.floor(math.log2(amax)) - 8
        assert sf[b] == 127 + e
        scaled = blk * 2.0 ** -e
        sat = np.abs(scaled) > 448.0
        ref = torch.from_numpy(np.where(sat, 0.0, scaled).astype(np.float32)).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy().copy()
        ref[sat] = np.where(scaled[sat] > 0, 0x7E, 0xFE)
        np.testing.assert_array_equal(codes[32 * b:32 * b + 32], ref)


def _mx8_floor_torch(v64: torch.Tensor):
    rows = v64.reshape(-1, 32)
    out = torch.empty_like(rows)
    for i in range(rows.shape[0]):
        a = float(rows[i].abs().max())
        e = 0 if a == 0 else max(-126, min(127, math.floor(math.log2(a)) - 8))
        scaled = (rows[i] * 2.0 ** -e).clamp(-448.0, 448.0)
        out[i] = scaled.to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64) * 2.0 ** e
    return out.reshape(v64.shape)


@pytest.mark.parametrize("clamp", [0.0, 0.75])
def test_dense_special_case_with_options_against_torch(oracle, clamp):
    """E=1, k=1, w=1 with the floor rule (and a clamp): a dense quantised FFN,
    rebuilt from torch matmuls, torch.clamp and torch's E4M3/bf16 casts."""
    T, H, I = 16, 128, 64
    w, d = _small(T, H, I, 1, 1, seed=13)
    idx = np.zeros((T, 1), np.int64)
    tw = np.ones((T, 1), np.float32)
    args = [a.numpy() for a in (d["w1q"], d["w1sf"], d["w2q"], d["w2sf"])]
    y = oracle.forward(_bits(d["x"]), idx, tw, 1, *args, activation_clamp=clamp,
                       scale_rule=oracle.SCALE_RULE_OCP_FLOOR)["y"]
    tab = _golden_e2m1()
    W1 = _deq_w(d["w1q"][0], d["w1sf"][0], tab)
    W2 = _deq_w(d["w2q"][0], d["w2sf"][0], tab)
    xq = _mx8_floor_torch(d["x"].to(torch.float64))
    acc = (xq @ W1.T).to(torch.float32).to(torch.bfloat16).to(torch.float32)
    g, u = acc[:, :I], acc[:, I:]
    if clamp > 0:
        g, u = g.clamp(-clamp, clamp), u.clamp(-clamp, clamp)
    g64 = g.to(torch.float64)
    silu = (g64 / (1.0 + torch.exp(-g64))).to(torch.float32)
    h = silu * u
    hq = _mx8_floor_torch(h.to(torch.float64))
    o = (hq @ W2.T).to(torch.float32).to(torch.bfloat16)
    ref = o.view(torch.int16).numpy().astype(np.uint16)
    assert np.mean(ref != y) <= 1e-3
    if clamp > 0:
        # the clamp bites: some gate/up values lie outside [-c, c]
        assert float((acc.abs() > clamp).float().mean()) > 0.05


@pytest.mark.parametrize("clamp,rule", [(0.5, 1), (0.5, 0), (0.0, 1)])
def test_bruteforce_matches_pool_oracle_with_options(oracle, clamp, rule):
    T, H, I, E, k = 24, 128, 64, 4, 2
    w, d = _small(T, H, I, E, k, seed=17)
    x = _bits(d["x"])
    idx, tw = d["topk_idx"].numpy(), d["topk_w"].numpy()
    args = [a.numpy() for a in (d["w1q"], d["w1sf"], d["w2q"], d["w2sf"])]
    res = oracle.forward(x, idx, tw, E, *args, activation_clamp=clamp, scale_rule=rule)
    base = oracle.forward(x, idx, tw, E, *args)
    assert not np.array_equal(res["y"], base["y"])     # the options change the result
    for t in range(T):
        yb, st = oracle.bruteforce_token(x[t], idx[t], tw[t], E, *args, activation_clamp=clamp, scale_rule=rule)
        assert st == 0
        np.testing.assert_array_equal(yb, res["y"][t])
