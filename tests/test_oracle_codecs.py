"""Pins of the oracle's number formats against the format definitions (golden
tables from the OCP specifications) and library casts (torch CPU)."""
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e4m3_golden_points(oracle):
    for code, val in _table("e4m3_points.txt"):
        got = oracle.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_decode_matches_torch_all_codes(oracle):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], c


def test_e4m3_roundtrip_and_ties(oracle):
    vals = [oracle.e4m3_decode(c) for c in range(127)]  # positive finite, monotone
    assert all(a < b for a, b in zip(vals, vals[1:]))
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, c
    # midpoints between neighbours go to the even code
    for c in range(126):
        mid = (vals[c] + vals[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, (c, mid)
        assert oracle.e4m3_encode(-mid) == 0x80 | want
    # saturation
    assert oracle.e4m3_encode(448.0001) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE


def test_e4m3_encode_matches_torch_cast(oracle):
    g = torch.Generator().manual_seed(0)
    v = torch.randn(4000, generator=g, dtype=torch.float32) * torch.exp2(torch.randint(-12, 9, (4000,), generator=g)).float()
    v = v.clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v.numpy()], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e2m1_golden_and_ties(oracle):
    for code, val in _table("e2m1_values.txt"):
        c = int(code, 16)
        got = oracle.e2m1_decode(c)
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))
        assert oracle.e2m1_encode(got) == c
    # ties to the even code; saturation
    for v, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (7.0, 7), (100.0, 7),
                 (-0.75, 0xA), (-5.0, 0xE), (0.2, 0), (0.3, 1), (2.6, 5), (4.9, 6), (5.1, 7)]:
        assert oracle.e2m1_encode(v) == c, v


def test_ue8m0_closed_forms(oracle):
    for maxnorm, amax, byte in _table("ue8m0_points.txt"):
        assert oracle.ue8m0_ceil(float(amax), float(maxnorm)) == int(byte), (maxnorm, amax)
    for n in range(-120, 120):
        for m in (448.0, 6.0):
            a = m * 2.0 ** n
            assert oracle.ue8m0_ceil(a, m) == n + 127
            assert oracle.ue8m0_ceil(np.nextafter(a, np.inf), m) == n + 128
    rng = np.random.default_rng(0)
    for a in np.exp(rng.uniform(-60, 60, 2000)):
        b = oracle.ue8m0_ceil(a, 448.0)
        e = b - 127
        assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)
        assert oracle.ue8m0_value(b) == 2.0 ** e


def test_bf16_matches_torch(oracle):
    g = torch.Generator().manual_seed(1)
    v = torch.randn(3000, generator=g) * torch.exp2(torch.randint(-30, 30, (3000,), generator=g)).float()
    v = torch.cat([v, torch.tensor([0.0, -0.0, 1.0, 3.0e38, -3.0e38, 1e-40])])
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_encode(float(x)) for x in v.numpy()], np.uint16)
    np.testing.assert_array_equal(got, ref)
    for b in ref[:50]:
        assert oracle.bf16_decode(int(b)) == float(torch.from_numpy(np.array([b], np.uint16).view(np.int16)).view(torch.bfloat16).float())


def test_mx_quant_block(oracle):
    # one block: amax 3.0 -> scale byte for E4M3 = smallest e with 3 <= 448*2^e -> e = -7
    v = np.zeros(32, np.float32)
    v[0], v[5], v[31] = 3.0, -1.5, 0.001
    q, sf = oracle.quant_mx_e4m3(v)
    assert sf[0] == 127 - 7
    assert oracle.e4m3_decode(int(q[0])) * 2.0 ** -7 == 3.0
    assert oracle.e4m3_decode(int(q[5])) * 2.0 ** -7 == -1.5
    # all-zero block: scale 1, codes 0
    q0, sf0 = oracle.quant_mx_e4m3(np.zeros(32, np.float32))
    assert sf0[0] == 127 and not q0.any()
    # E2M1 block
    w = np.linspace(-1, 1, 32).astype(np.float32)
    nib, sfw = oracle.quant_mx_e2m1(w)
    assert sfw[0] == oracle.ue8m0_ceil(1.0, 6.0)
    deq = np.array([oracle.e2m1_decode(int(n)) for n in nib]) * 2.0 ** (int(sfw[0]) - 127)
    assert np.max(np.abs(deq - w)) <= 0.25 * 2.0 ** (int(sfw[0]) - 127) * 2 + 1e-9
