"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, and compare with the CPU oracle element by element.

Tolerances (per output element, B = sum_i |x_i w_i| from the oracle in fp64):
  m <= 16 (decode, fp32 X):        |y - y_ref| <= 1e-3 * B + 1e-5
  m >  16 (prefill, X cast bf16):  |y - y_ref| <= 1e-2 * B + 1e-4
"""

from __future__ import annotations

import numpy as np

DECODE_TOL = (1e-3, 1e-5)
PREFILL_TOL = (1e-2, 1e-4)


def tol_for(m: int):
    return DECODE_TOL if m <= 16 else PREFILL_TOL


def to_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack_dev(q4lib, blocks: np.ndarray, n: int, k: int):
    import torch
    b = to_dev(blocks.reshape(-1))
    W = torch.empty(q4lib.q4_0_packed_size(n, k), dtype=torch.uint8, device="cuda")
    q4lib.q4_0_pack(W, b, n, k)
    return W


def run_matmul(q4lib, W, X: np.ndarray, n: int, use_library_ws: bool = False):
    import torch
    m, k = X.shape
    Xd = to_dev(X)
    Y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    if use_library_ws:
        q4lib.q4_0_matmul(W, Xd, Y, m, k, n)
    else:
        ws, wsb = q4lib.workspace_for(m, k, n)
        q4lib.q4_0_matmul_ws(W, Xd, Y, m, k, n, ws, wsb)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    return Y.cpu().numpy()


def assert_parity(Y: np.ndarray, Yref: np.ndarray, B: np.ndarray, m: int, what: str = "") -> float:
    """Element-wise tolerance check; returns max err / tol."""
    rtol, atol = tol_for(m)
    Y = Y.astype(np.float64)
    assert Y.shape == Yref.shape
    nan_ref = np.isnan(Yref)
    assert np.array_equal(np.isnan(Y), nan_ref), f"{what}: NaN pattern differs"
    fin = ~nan_ref
    inf_ref = np.isinf(Yref) & fin
    assert np.array_equal(Y[inf_ref], Yref[inf_ref]), f"{what}: infinities differ"
    ok = fin & ~inf_ref
    err = np.abs(Y[ok] - Yref[ok])
    tol = rtol * B[ok] + atol
    ratio = float((err / tol).max()) if err.size else 0.0
    if ratio > 1.0:
        i = int(np.argmax(err / tol))
        raise AssertionError(f"{what}: max err/tol {ratio:.3g} (err {err[i]:.3g}, tol {tol[i]:.3g})")
    return ratio
