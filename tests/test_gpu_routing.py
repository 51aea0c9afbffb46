"""GPU dispatch plan against the oracle plan, bit-exact, on every workload and
on edge cases: the one-launch plan (route_fused, E <= 256: one chunk per CTA,
or several when the chunks outnumber its 512 CTAs), the one-CTA plan for more
experts and at most 2048 entries (route_small), and the chunked count / scan /
slot kernels beyond."""
import numpy as np
import pytest
import torch

from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu


def run_plan(moe, idx, tw, E, H=256, I=128):
    p = moe.plan(torch.as_tensor(idx, device="cuda"), torch.as_tensor(tw, device="cuda"), E, H, I)
    st = moe.plan_check(p)
    return p, st


def compare_plan(moe, oracle, idx, tw, E, H=256, I=128):
    idx = np.ascontiguousarray(idx, np.int64)
    tw = np.ascontiguousarray(tw, np.float32)
    p, st = run_plan(moe, idx, tw, E, H, I)
    ref = oracle.plan(idx, tw, E, p_cap=p.export("pool_rows"))
    assert st == (moe.ERR_BAD_EXPERT_ID if ref["status"] == 1 else 0)
    g = lambda n: p.export(n).cpu().numpy()
    np.testing.assert_array_equal(g("count"), ref["count"])
    np.testing.assert_array_equal(g("off"), ref["off"])
    np.testing.assert_array_equal(g("poff"), ref["poff"])
    np.testing.assert_array_equal(g("slot_of"), ref["slot_of"])
    P = int(ref["poff"][-1])
    assert int(g("n_blocks")[0]) == P // 128
    assert int(g("max_count")[0]) == int(ref["count"].max(initial=0))
    np.testing.assert_array_equal(g("row_token")[:P], ref["row_token"][:P])
    np.testing.assert_array_equal(g("row_topk")[:P], ref["row_topk"][:P])
    np.testing.assert_array_equal(g("row_weight")[:P].view(np.uint32), ref["row_weight"][:P].view(np.uint32))
    be = g("block_expert")[: P // 128]
    want = np.repeat(np.arange(E), (np.diff(ref["poff"]) // 128))
    np.testing.assert_array_equal(be, want)
    return p


@pytest.mark.parametrize("name", ["tiny", "mid", "share", "full", "decode"])
def test_plan_workloads(moe, oracle, name):
    w = inputs.WORKLOADS[name]
    idx, tw = inputs.make_routing(w)
    compare_plan(moe, oracle, idx.numpy(), tw.numpy(), w.E)


def test_plan_edge_cases(moe, oracle):
    rng = np.random.default_rng(0)
    E = 16
    # every entry skipped
    compare_plan(moe, oracle, -np.ones((50, 4)), np.ones((50, 4)), E)
    # all tokens to one expert, duplicates inside each token
    compare_plan(moe, oracle, np.full((3000, 2), 5), rng.random((3000, 2)), E)
    # experts with 0, 1, 127, 128, 129 rows spread over several routing chunks
    flat = np.concatenate([np.full(n, e) for e, n in {0: 0, 1: 1, 2: 127, 3: 128, 4: 129, 5: 4000}.items()])
    flat = rng.permutation(flat)
    compare_plan(moe, oracle, flat.reshape(-1, 1), np.ones((flat.size, 1)), 6)
    # many chunks, k = 32, E = 1024
    compare_plan(moe, oracle, rng.integers(-1, 1024, size=(700, 32)), rng.random((700, 32)), 1024)
    # bad ids are skipped and reported
    idx = rng.integers(-1, 8, size=(100, 4))
    idx[3, 1] = 8
    idx[50, 0] = -7
    idx[77, 3] = 1 << 40
    compare_plan(moe, oracle, idx, rng.random((100, 4)), 8)


@pytest.mark.parametrize("n", [1, 2047, 2048, 2049, 4096])
@pytest.mark.parametrize("E", [8, 300, 512, 1024])
def test_plan_one_kernel_and_chunked_paths(moe, oracle, n, E):
    """Both sides of the 2048-entry switch, with skipped and bad ids: E = 8
    runs the one-launch plan on either side (one chunk on 16 CTAs, or two);
    more experts run the one-CTA kernel up to 2048 entries and the chunked
    count / scan / slot kernels above it, with 1024, 640 and 256 threads."""
    rng = np.random.default_rng(n + E)
    idx = rng.integers(-1, E, size=(n, 1))
    if n > 3:
        idx[n // 2, 0] = E
    compare_plan(moe, oracle, idx, rng.random((n, 1)), E)


@pytest.mark.parametrize("n", [512 * 2048, 512 * 2048 + 1, 1_100_000])
def test_plan_more_chunks_than_ctas(moe, oracle, n):
    """The one-launch plan has at most 512 CTAs: at 512 chunks each still
    counts and slots one chunk from registers; beyond it the CTAs take
    further chunks from the work counters."""
    rng = np.random.default_rng(n)
    E = 64
    # skewed ids: a few hot experts, every expert present, some skipped entries
    idx = np.minimum(rng.zipf(1.3, size=n) - 1, E - 1)
    idx[rng.random(n) < 0.05] = -1
    compare_plan(moe, oracle, idx.reshape(-1, 8 if n % 8 == 0 else 1), rng.random(n).reshape(-1, 8 if n % 8 == 0 else 1), E)


def test_empty_batch(moe):
    p, st = run_plan(moe, np.zeros((0, 4), np.int64), np.zeros((0, 4), np.float32), 8)
    assert st == 0
    assert int(p.export("n_blocks").cpu()[0]) == 0
    assert int(p.export("max_count").cpu()[0]) == 0
    assert p.export("count").sum().item() == 0


def test_plan_is_deterministic(moe):
    w = inputs.WORKLOADS["full"]
    idx, tw = inputs.make_routing(w)
    a, _ = run_plan(moe, idx, tw, w.E)
    b, _ = run_plan(moe, idx, tw, w.E)
    assert torch.equal(a.export("slot_of"), b.export("slot_of"))
