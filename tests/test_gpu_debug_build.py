"""The debug build of the library (-DMOE_DEBUG: device bounds checks on the
plan tables that dispatch, the expert kernel and combine consume; the
stand-in for a memory checker, which is not available on this GPU pool).

On valid plans it gives exactly the release build's bytes.  A corrupted plan
table (a slot one past the pool, an expert id one past the last expert) is
reported as MOE_ERR_DEBUG_BOUNDS with the place of the first failure, the
access is skipped or clamped (the corrupted values are chosen so that even an
unchecked access would stay inside the caller's buffers), and the context
stays usable.  The debug library runs in a child process, since a process
loads one libmoe."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
import numpy as np, torch
root = sys.argv[1]
sys.path.insert(0, root); sys.path.insert(0, os.path.join(root, "tests"))
from moe_expert_layer_counts_gb300 import build as b
import moe_expert_layer_counts_gb300 as moe
moe.LIB_PATH = b.build(debug=True)
import gpu_helpers as gh
from moe_expert_layer_counts_gb300 import inputs
mode, out = sys.argv[2], sys.argv[3]
res = {}
if mode == "valid":
    for name in ("tiny", "mid", "decode"):
        w = inputs.WORKLOADS[name]
        d, W1, W2 = gh.setup(moe, w)
        p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
        y = moe.forward(d["x"], W1, W2, p)
        res[name] = moe.plan_check(p)
        np.save(os.path.join(out, name + ".npy"), y.view(torch.int16).cpu().numpy())
else:
    w = inputs.WORKLOADS["tiny"]
    d, W1, W2 = gh.setup(moe, w)
    for what in ("slot_of", "block_expert"):
        p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
        assert moe.plan_check(p) == moe.OK
        if what == "slot_of":
            p.export("slot_of")[0] = p.export("pool_rows")      # one past the pool
        else:
            p.export("block_expert")[0] = w.E                   # one past the experts
        moe.forward(d["x"], W1, W2, p)
        res[what] = [moe.plan_check(p), int(p.export("error").cpu()[1])]
    # the context is still good: a fresh plan runs clean
    p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
    moe.forward(d["x"], W1, W2, p)
    res["after"] = moe.plan_check(p)
json.dump(res, open(os.path.join(out, "res.json"), "w"))
"""


def run_child(mode, tmp_path):
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, mode, str(tmp_path)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.load(open(os.path.join(tmp_path, "res.json")))


def test_debug_build_matches_release_bytes(moe, tmp_path):
    res = run_child("valid", tmp_path)
    for name in ("tiny", "mid", "decode"):
        assert res[name] == moe.OK, (name, res[name])
        w = inputs.WORKLOADS[name]
        d, W1, W2 = gh.setup(moe, w)
        p = moe.plan(d["topk_idx"], d["topk_w"], w.E, w.H, w.I)
        y = moe.forward(d["x"], W1, W2, p)
        assert moe.plan_check(p) == moe.OK
        np.testing.assert_array_equal(y.view(torch.int16).cpu().numpy(), np.load(os.path.join(tmp_path, name + ".npy")))


def test_debug_build_reports_corrupted_plan_tables(moe, tmp_path):
    res = run_child("corrupt", tmp_path)
    # dispatch meets the bad slot first (place 1), the expert kernel the bad expert id (place 3)
    assert res["slot_of"] == [moe.ERR_DEBUG_BOUNDS, 201], res
    assert res["block_expert"] == [moe.ERR_DEBUG_BOUNDS, 203], res
    assert res["after"] == moe.OK
