"""The checked build (-DQ4MM_CHECKED, q4_build_flags() bit 0): the decode
mat-vec checks its shared-memory layout against the launch, every weight
record it copies against the layer and every slot row it reads or writes,
and reports a failed check as Q4_ERR_DEVICE_CHECK in the device status word
instead of touching memory out of range. Valid calls report nothing and give
the ordinary build's bits; a negative slot row is reported and skipped (that
case runs on the checked build only: the ordinary build takes slot rows as
given)."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT
from q4_quantized_linear_gb300 import synth
from q4_testlib import pack_dev, run_matmul

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SHAPES = [(1, 9728, 2560), (4, 2560, 9728), (8, 1000, 2080), (16, 14336, 4096), (13, 130, 640)]

CHILD = r"""
import json, os, sys
import numpy as np
ROOT, OUT = sys.argv[1], sys.argv[2]
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))
import torch
from q4_quantized_linear_gb300 import binding as q4, synth
from q4_testlib import pack_dev, run_matmul
res = {"flags": q4.q4_build_flags(), "status": {}}
assert res["flags"] & 1, "not the checked build"
q4.q4_last_device_status(clear=True)
for (m, n, k) in json.loads(sys.argv[3]):
    blocks = synth.q4_0_blocks(n, k, seed=n + m)
    X = synth.activations(m, k, seed=m)
    Y = run_matmul(q4, pack_dev(q4, blocks, n, k), X, n)
    res["status"][f"{m}x{n}x{k}"] = q4.q4_last_device_status(clear=True)
    np.save(os.path.join(OUT, f"{m}x{n}x{k}.npy"), Y)
# a slot row out of range: reported, its row skipped, the others written
n, k = 130, 640
blocks = synth.q4_0_blocks(n, k, seed=5)
W = pack_dev(q4, blocks, n, k)
Xs = torch.from_numpy(synth.activations(4, k, seed=6)).cuda()
Ys = torch.full((4, n), 7.0, dtype=torch.float32, device="cuda")
slots = torch.tensor([0, -5, 3], dtype=torch.int32, device="cuda")
q4.q4_set_decode_kernel(q4.Q4_DECODE_MATVEC)
try:
    q4.q4_0_matmul_batched_slots(W, Xs, k, slots, 3, Ys, n, k, n)
    res["bad_slot_status"] = q4.q4_last_device_status(clear=True)
finally:
    q4.q4_set_decode_kernel(q4.Q4_DECODE_AUTO)
np.save(os.path.join(OUT, "slots.npy"), Ys.cpu().numpy())
res["after_status"] = q4.q4_last_device_status(clear=True)
json.dump(res, open(os.path.join(OUT, "res.json"), "w"))
"""


@pytest.fixture(scope="module")
def checked_run(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q4_quantized_linear_gb300 import build
    lib = build.build(checked=True)
    out = str(tmp_path_factory.mktemp("checked"))
    env = dict(os.environ, Q4MM_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, out, json.dumps(SHAPES)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    with open(os.path.join(out, "res.json")) as f:
        return out, json.load(f)


def test_checked_build_reports_nothing_and_matches_the_ordinary_build(q4lib, checked_run):
    out, res = checked_run
    for (m, n, k) in SHAPES:
        key = f"{m}x{n}x{k}"
        assert res["status"][key] == 0, key
        blocks = synth.q4_0_blocks(n, k, seed=n + m)
        X = synth.activations(m, k, seed=m)
        Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
        assert np.array_equal(np.load(os.path.join(out, key + ".npy")), Y), key


def test_checked_build_reports_a_slot_row_out_of_range(q4lib, oracle_mod, checked_run):
    out, res = checked_run
    assert res["bad_slot_status"] == q4lib.Q4_ERR_DEVICE_CHECK
    assert res["after_status"] == 0
    n, k = 130, 640
    blocks = synth.q4_0_blocks(n, k, seed=5)
    Xs = synth.activations(4, k, seed=6)
    Ys = np.load(os.path.join(out, "slots.npy"))
    Yr, _ = oracle_mod.matmul(blocks, Xs, n, k)
    # slots 0 and 3 written (the decode bound), 1 and 2 untouched
    from q4_testlib import tol_for
    rtol, atol = tol_for(3)
    _, B = oracle_mod.matmul(blocks, Xs, n, k)
    for r in (0, 3):
        assert np.all(np.abs(Ys[r] - Yr[r]) <= rtol * B[r] + atol)
    assert np.all(Ys[1] == 7.0) and np.all(Ys[2] == 7.0)
