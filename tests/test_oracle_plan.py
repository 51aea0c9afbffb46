"""Pins of the oracle's dispatch plan: the invariants the method fixes and a
brute-force stable counting sort written independently in Python."""
import numpy as np
import pytest

BM = 128


def brute_plan(idx, E):
    """Independent restatement: sort the valid entries by (expert, flat index)."""
    T, k = idx.shape
    flat = idx.reshape(-1)
    entries = sorted((int(e), i) for i, e in enumerate(flat) if 0 <= e < E)
    count = np.bincount([e for e, _ in entries], minlength=E).astype(np.int64)
    padded = (count + BM - 1) // BM * BM
    poff = np.concatenate([[0], np.cumsum(padded)])
    slot = -np.ones(T * k, np.int64)
    seen = {}
    for e, i in entries:
        slot[i] = poff[e] + seen.get(e, 0)
        seen[e] = seen.get(e, 0) + 1
    return count, poff, slot


def check_invariants(p, idx, w, E):
    T, k = idx.shape
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    # counts sum to the number of non-negative entries
    assert p["count"].sum() == valid.sum()
    # offsets are exclusive scans
    np.testing.assert_array_equal(p["off"], np.concatenate([[0], np.cumsum(p["count"])]))
    padded = (p["count"] + BM - 1) // BM * BM
    np.testing.assert_array_equal(p["poff"], np.concatenate([[0], np.cumsum(padded)]))
    assert np.all(p["poff"] % BM == 0)
    # the pool mapping is a bijection between valid entries and rows with row_token >= 0
    s = p["slot_of"]
    assert np.all(s[~valid] == -1)
    sv = s[valid]
    assert len(np.unique(sv)) == len(sv)
    used = np.nonzero(p["row_token"] >= 0)[0]
    np.testing.assert_array_equal(np.sort(sv), used)
    fi = np.nonzero(valid)[0]
    np.testing.assert_array_equal(p["row_token"][sv], fi // k)
    np.testing.assert_array_equal(p["row_topk"][sv], fi % k)
    np.testing.assert_array_equal(p["row_weight"][sv], w.reshape(-1)[fi])
    # each row lies in its expert's segment; slots increase with flat index inside an expert
    e_of = flat[fi]
    assert np.all(sv >= p["poff"][e_of]) and np.all(sv < p["poff"][e_of] + p["count"][e_of])
    for e in range(E):
        se = sv[e_of == e]
        assert np.all(np.diff(se) == 1)


@pytest.mark.parametrize("T,k,E,seed", [(64, 2, 8, 0), (300, 6, 64, 1), (1000, 8, 256, 2), (5, 1, 3, 3)])
def test_plan_random(oracle, T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = rng.integers(-1, E, size=(T, k)).astype(np.int64)
    w = rng.random((T, k)).astype(np.float32)
    p = oracle.plan(idx, w, E)
    assert p["status"] == 0
    check_invariants(p, idx, w, E)
    count, poff, slot = brute_plan(idx, E)
    np.testing.assert_array_equal(p["count"], count)
    np.testing.assert_array_equal(p["poff"], poff)
    np.testing.assert_array_equal(p["slot_of"], slot)


def test_plan_edge_cases(oracle):
    E = 16
    # every entry skipped
    idx = -np.ones((10, 4), np.int64)
    p = oracle.plan(idx, np.ones((10, 4), np.float32), E)
    assert p["count"].sum() == 0 and p["poff"][-1] == 0 and np.all(p["slot_of"] == -1)
    # all tokens to one expert, with duplicates inside a token's top-k
    idx = np.full((300, 2), 5, np.int64)
    w = np.full((300, 2), 0.5, np.float32)
    p = oracle.plan(idx, w, E)
    assert p["count"][5] == 600 and p["poff"][-1] == 640
    np.testing.assert_array_equal(p["slot_of"], np.arange(600))
    check_invariants(p, idx, w, E)
    # experts with 0, 1, BM-1, BM, BM+1 rows
    sizes = {0: 0, 1: 1, 2: BM - 1, 3: BM, 4: BM + 1}
    flat = np.concatenate([np.full(n, e) for e, n in sizes.items()])
    flat = np.random.default_rng(0).permutation(flat).astype(np.int64)
    idx = flat.reshape(-1, 1)
    w = np.ones_like(idx, np.float32)
    p = oracle.plan(idx, w, 5)
    np.testing.assert_array_equal(p["count"], [0, 1, BM - 1, BM, BM + 1])
    np.testing.assert_array_equal(p["poff"], [0, 0, BM, 2 * BM, 3 * BM, 5 * BM])
    check_invariants(p, idx, w, 5)
    # empty batch
    p = oracle.plan(np.zeros((0, 3), np.int64), np.zeros((0, 3), np.float32), E)
    assert p["count"].sum() == 0 and p["slot_of"].size == 0


def test_plan_bad_ids_flagged_and_skipped(oracle):
    idx = np.array([[0, 7], [9, -1], [-2, 3]], np.int64)
    w = np.ones((3, 2), np.float32)
    p = oracle.plan(idx, w, 8)
    assert p["status"] == 1
    np.testing.assert_array_equal(p["slot_of"][[2, 4]], [-1, -1])
    assert p["count"].sum() == 3
