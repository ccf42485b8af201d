"""The W4A8 entry point (q4_0_matmul_w4a8) against the oracle's W4A8 variant.

X is coded per 32-element block to int8 on the GPU with the same fp32
operations as the oracle (codes are integers decided in the same precision
on both sides), each block's dot product is an exact integer, and d * s and
the sum over blocks are fp32. Tolerance per element, B8 from the oracle:
  |y - y_ref| <= 4e-5 * B8 + 1e-6
(fp32 rounding of d * s, of each block term and of the running sum over at
most 304 blocks: (304 + 2) * 2^-24 < 2e-5). The integer case (codes equal to
X, power-of-two d) is compared bit-exactly; so are the hand-derived ties.
"""

import json
import os

import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth
from q4_testlib import pack_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RTOL, ATOL = 4e-5, 1e-6
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_w4a8(q4lib, W, X, n):
    m, k = X.shape
    Xd = to_dev(np.ascontiguousarray(X, dtype=np.float32))
    Y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    q4lib.q4_0_matmul_w4a8(W, Xd, Y, m, k, n)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    return Y.cpu().numpy().astype(np.float64)


def assert_w4a8(Y, Yr, B8, what):
    nan_ref = np.isnan(Yr)
    assert np.array_equal(np.isnan(Y), nan_ref), f"{what}: NaN pattern differs"
    ok = ~nan_ref
    err = np.abs(Y[ok] - Yr[ok])
    ratio = float((err / (RTOL * B8[ok] + ATOL)).max()) if err.size else 0.0
    assert ratio <= 1.0, f"{what}: max err / tol = {ratio:.3g}"


SHAPES = [(1, 32), (64, 64), (65, 96), (200, 1056), (1000, 2080), (333, 4096), (130, 8192 + 64)]


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("n,k", SHAPES)
def test_w4a8_parity(q4lib, oracle_mod, m, n, k):
    blocks = synth.q4_0_blocks(n, k, seed=3000 + n)
    X = synth.activations(m, k, seed=4000 + m)
    Y = run_w4a8(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B8 = oracle_mod.matmul_w4a8(blocks, X, n, k)
    assert_w4a8(Y, Yr, B8, f"w4a8 m={m} n={n} k={k}")


@pytest.mark.parametrize("m,n,k", [(1, 9728, 2560), (4, 9728, 2560), (4, 2560, 9728),
                                   (8, 14336, 4096), (16, 14336, 4096)])
def test_w4a8_workload_sizes(q4lib, oracle_mod, m, n, k):
    blocks = synth.q4_0_blocks(n, k, seed=0)
    X = synth.activations(m, k, seed=0)
    Y = run_w4a8(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B8 = oracle_mod.matmul_w4a8(blocks, X, n, k)
    assert_w4a8(Y, Yr, B8, f"w4a8 m={m} n={n} k={k}")


@pytest.mark.parametrize("m", [1, 4, 7, 8, 9, 16])
def test_w4a8_integer_case_is_bit_exact(q4lib, oracle_mod, m):
    """Integer X with |x| <= 127 and a +-127 in every block (codes = X, scale
    1) and power-of-two d: every block term and sum is exact in fp32."""
    n, k = 200, 1024
    blocks = synth.q4_0_blocks(n, k, seed=51)
    nb = k // 32
    e = (synth.draw_u64(51, 9, n * nb) % np.uint64(6)).astype(np.int64) - 8
    d = np.ldexp(1.0, e).astype(np.float16).reshape(n, nb)
    blocks[:, :, 0:2] = d.astype("<f2").view(np.uint8).reshape(n, nb, 2)
    xi = (synth.draw_u64(52, 9, m * k) % np.uint64(255)).astype(np.int64) - 127
    X = xi.astype(np.float32).reshape(m, k)
    X[:, ::32] = 127.0
    Y = run_w4a8(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, _ = oracle_mod.matmul_w4a8(blocks, X, n, k)
    assert np.array_equal(Y, Yr)


def test_w4a8_golden_codes(q4lib):
    """The hand-derived cases of tests/golden/w4a8_blocks.json: round-half-even
    ties and one scale per block, through the GPU."""
    with open(os.path.join(GOLDEN, "w4a8_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        k = case["k"]
        nb = k // 32
        blocks = np.zeros((1, nb, 18), dtype=np.uint8)
        for b in range(nb):
            blocks[0, b, 0] = case["d_bits"][b] & 0xFF
            blocks[0, b, 1] = case["d_bits"][b] >> 8
            blocks[0, b, 2:] = 0x99
        X = np.zeros((1, k), dtype=np.float32)
        for i, v in case["x_nonzero"].items():
            X[0, int(i)] = v
        Y = run_w4a8(q4lib, pack_dev(q4lib, blocks, 1, k), X, 1)
        assert abs(Y[0, 0] - case["y"]) <= 1e-6 * abs(case["y"]), f"{case['name']}: {Y[0, 0]} != {case['y']}"


@pytest.mark.parametrize("m", [1, 3, 9])
def test_w4a8_nonfinite_rows_and_zero_rows(q4lib, oracle_mod, m):
    n, k = 100, 256
    blocks = synth.q4_0_blocks(n, k, seed=53)
    X = synth.activations(m, k, seed=54)
    X[0, 5] = np.nan
    if m > 1:
        X[m - 1, 77] = np.inf
        X[1] = 0.0
    Y = run_w4a8(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B8 = oracle_mod.matmul_w4a8(blocks, X, n, k)
    assert_w4a8(Y, Yr, B8, "non-finite rows")
    if m > 1:
        assert np.all(Y[1] == 0.0)


def test_w4a8_is_bitwise_deterministic_and_m0_is_a_no_op(q4lib):
    n, k, m = 1000, 2080, 5
    blocks = synth.q4_0_blocks(n, k, seed=55)
    X = synth.activations(m, k, seed=56)
    W = pack_dev(q4lib, blocks, n, k)
    Y1 = run_w4a8(q4lib, W, X, n)
    Y2 = run_w4a8(q4lib, W, X, n)
    assert np.array_equal(Y1, Y2)
    Y = torch.full((1, n), 7.0, dtype=torch.float32, device="cuda")
    Xd = to_dev(X)
    assert q4lib.q4_0_matmul_w4a8(W, Xd, Y, 0, k, n) == 0
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)
