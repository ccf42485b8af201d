"""q4_0_matmul_static_scratch, the form of q4_0_matmul that allocates nothing
(its scratch is a fixed device array of the library), for callers that may
not allocate device memory. Checked through the C ABI on two calls in a row:
against the CPU oracle at the decode or prefill tolerance, and against the
existing entry point q4_0_matmul (the same kernels, so the same bits); and
its refusal of shapes whose scratch does not fit. Collected last, it must
pass on its own and after every other test."""
import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth
from q4_testlib import pack_dev, to_dev, tol_for

pytestmark = pytest.mark.gpu


def _run(q4lib, fn, W, Xd, m, k, n):
    import torch
    Y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    fn(W, Xd, Y, m, k, n)
    return Y


@pytest.mark.parametrize("m,n,k", [(64, 200, 1056), (540, 9728, 2560), (4, 9728, 2560)])
def test_static_scratch_matches_matmul_on_two_calls(q4lib, oracle_mod, m, n, k):
    import torch
    blocks = synth.q4_0_blocks(n, k, seed=7000 + n)
    W = pack_dev(q4lib, blocks, n, k)
    rtol, atol = tol_for(m)
    rng = np.random.default_rng(17)
    for call in range(2):
        X = synth.activations(m, k, seed=8000 + 10 * m + call)   # a new X each call
        Xd = to_dev(X)
        Ys = _run(q4lib, q4lib.q4_0_matmul_static_scratch, W, Xd, m, k, n)
        Yr = _run(q4lib, q4lib.q4_0_matmul, W, Xd, m, k, n)
        torch.cuda.synchronize()
        assert q4lib.q4_last_device_status(clear=True) == 0
        ys = Ys.cpu().numpy().astype(np.float64)
        yr = Yr.cpu().numpy().astype(np.float64)
        assert np.isfinite(ys).all() and np.isfinite(yr).all(), f"call {call}: unwritten outputs"
        # the same kernels as the existing entry point: the same bits
        assert np.array_equal(ys.view(np.uint64), yr.view(np.uint64)), f"call {call}: differs from q4_0_matmul"
        # and the oracle's Y, element by element on a sample, at the tolerance of m
        cnt = 4000
        t = np.concatenate([rng.integers(0, m, cnt), [0, m - 1]])
        j = np.concatenate([rng.integers(0, n, cnt), [0, n - 1]])
        Yo, B = oracle_mod.matmul_sampled(blocks, X, n, k, t, j)
        err = np.abs(ys[t, j] - Yo)
        assert np.all(err <= rtol * B + atol), f"call {call}: max err/tol {float((err / (rtol * B + atol)).max())}"


def test_static_scratch_refuses_oversize_shapes(q4lib):
    import torch
    m, n, k = 4096, 128, 4096
    need = q4lib.q4_0_matmul_workspace_size(m, k, n)
    assert need > q4lib.Q4_STATIC_SCRATCH_BYTES
    W = torch.zeros(q4lib.q4_0_packed_size(n, k), dtype=torch.uint8, device="cuda")
    X = torch.zeros((m, k), dtype=torch.float32, device="cuda")
    Y = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    rc = q4lib.q4_0_matmul_static_scratch(W, X, Y, m, k, n, check=False)
    torch.cuda.synchronize()
    assert rc == q4lib.Q4_ERR_WORKSPACE
    assert bool((Y == 7.0).all()), "nothing may run for a refused shape"
