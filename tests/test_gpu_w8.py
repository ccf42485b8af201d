"""Per-output-channel int8 weights through the C ABI (rembed "Architecture",
"int8 quantization", the weight-only form): the GPU quantiser against the
oracle's codes and scales (bit-exact: both take every decision in fp32), and
q4_w8_matmul against the oracle's fp64 product of those codes, element by
element at the decode tolerance |y - y_ref| <= 1e-3 * B + 1e-5."""

import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth
from q4_testlib import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RTOL, ATOL = 1e-3, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def weights(n, k, seed):
    W = synth.activations(n, k, seed=seed)      # fp32 N(0, 1)
    W[::7] *= 0.02                              # rows of other magnitudes
    return W


def quantize_dev(q4lib, W):
    n, k = W.shape
    Wd = to_dev(W)
    P = torch.empty(q4lib.q4_w8_packed_size(n, k), dtype=torch.uint8, device="cuda")
    q4lib.q4_w8_quantize(P, Wd, n, k)
    return P


def unpack_dev(q4lib, P, n, k):
    codes = torch.empty((n, k), dtype=torch.int8, device="cuda")
    scales = torch.empty(n, dtype=torch.float32, device="cuda")
    q4lib.q4_w8_unpack(codes, scales, P, n, k)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def run_w8(q4lib, P, X, n):
    m, k = X.shape
    Y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    q4lib.q4_w8_matmul(P, to_dev(X), Y, m, k, n)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    return Y.cpu().numpy().astype(np.float64)


def check(Y, Yr, B, what):
    nan_ref = np.isnan(Yr)
    assert np.array_equal(np.isnan(Y), nan_ref), f"{what}: NaN pattern differs"
    ok = ~nan_ref & ~np.isinf(Yr)
    assert np.array_equal(Y[np.isinf(Yr)], Yr[np.isinf(Yr)]), f"{what}: infinities differ"
    err = np.abs(Y[ok] - Yr[ok])
    ratio = float((err / (RTOL * B[ok] + ATOL)).max()) if err.size else 0.0
    assert ratio <= 1.0, f"{what}: max err/tol {ratio:.3g}"


@pytest.mark.parametrize("n,k", [(1, 32), (130, 96), (200, 1056), (9728, 2560)])
def test_quantizer_matches_the_oracle_bit_for_bit(q4lib, oracle_mod, n, k):
    W = weights(n, k, seed=n + k)
    W[n // 2] = 0.0                              # a zero row: codes 0, scale 0
    codes, scales = unpack_dev(q4lib, quantize_dev(q4lib, W), n, k)
    c_ref, s_ref = oracle_mod.quantize_w_int8(W)
    assert np.array_equal(codes, c_ref), "codes differ from the oracle's"
    assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32)), "scales differ from the oracle's"


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 13, 16, 17, 40])
@pytest.mark.parametrize("n,k", [(1, 32), (65, 96), (200, 1056), (333, 4096), (130, 8192 + 64)])
def test_w8_matmul_parity(q4lib, oracle_mod, m, n, k):
    W = weights(n, k, seed=500 + n)
    X = synth.activations(m, k, seed=600 + m)
    P = quantize_dev(q4lib, W)
    Y = run_w8(q4lib, P, X, n)
    c, s = oracle_mod.quantize_w_int8(W)
    Yr, B = oracle_mod.matmul_w8(c, s, X)
    check(Y, Yr, B, f"w8 m={m} n={n} k={k}")


@pytest.mark.parametrize("m,n,k", [(1, 9728, 2560), (4, 9728, 2560), (4, 2560, 9728), (16, 14336, 4096)])
def test_w8_workload_sizes(q4lib, oracle_mod, m, n, k):
    W = weights(n, k, seed=0)
    X = synth.activations(m, k, seed=0)
    Y = run_w8(q4lib, quantize_dev(q4lib, W), X, n)
    c, s = oracle_mod.quantize_w_int8(W)
    Yr, B = oracle_mod.matmul_w8(c, s, X)
    check(Y, Yr, B, f"w8 workload m={m} n={n} k={k}")


def test_w8_nonfinite_x_and_zero_rows(q4lib, oracle_mod):
    m, n, k = 3, 100, 256
    W = weights(n, k, seed=41)
    W[5] = 0.0
    X = synth.activations(m, k, seed=42)
    X[0, 5] = np.nan
    X[2, 77] = np.inf
    Y = run_w8(q4lib, quantize_dev(q4lib, W), X, n)
    c, s = oracle_mod.quantize_w_int8(W)
    Yr, B = oracle_mod.matmul_w8(c, s, X)
    check(Y, Yr, B, "w8 non-finite X")


def test_w8_m_zero_and_determinism(q4lib):
    m, n, k = 4, 2560, 9728
    W = weights(n, k, seed=7)
    P = quantize_dev(q4lib, W)
    Y0 = torch.full((1, n), 3.0, dtype=torch.float32, device="cuda")
    q4lib.q4_w8_matmul(P, to_dev(np.zeros((1, k), np.float32)), Y0, 0, k, n)
    torch.cuda.synchronize()
    assert bool((Y0 == 3.0).all())
    X = synth.activations(m, k, seed=8)
    Y1, Y2 = run_w8(q4lib, P, X, n), run_w8(q4lib, P, X, n)
    assert np.array_equal(Y1.view(np.uint64), Y2.view(np.uint64))
