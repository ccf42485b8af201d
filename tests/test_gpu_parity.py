"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Covers the repacker (byte-exact), decode m = 1..16 and prefill m > 16 on
ragged shapes spanning several tiles, the workload sizes (full compare
where the oracle finishes in seconds, sampled elements otherwise),
continuous batching through slot indices, and the degenerate cases: m = 0,
all-zero weights, exact integer inputs (bit-exact), NaN/Inf propagation,
zero and negative scales, run-to-run bitwise determinism, and the bounded
device wait.
"""

import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth
from q4_testlib import assert_parity, pack_dev, run_matmul, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# ------------------------------------------------------------- repacker ----

@pytest.mark.parametrize("n,k", [(1, 32), (16, 64), (64, 64), (70, 96), (333, 1056), (9728, 2560)])
def test_pack_matches_oracle_layout_and_unpack_inverts(q4lib, oracle_mod, n, k):
    blocks = synth.q4_0_blocks(n, k, seed=n + k)
    W = pack_dev(q4lib, blocks, n, k)
    torch.cuda.synchronize()
    ref = oracle_mod.pack_reference(blocks, n, k)
    assert np.array_equal(W.cpu().numpy(), ref), "packed bytes differ from the layout reference"
    back = torch.empty(blocks.size, dtype=torch.uint8, device="cuda")
    q4lib.q4_0_unpack(back, W, n, k)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), blocks.reshape(-1)), "unpack(pack(W)) != W"


# --------------------------------------------------------- small shapes ----

SHAPES = [(1, 32), (64, 64), (65, 96), (200, 1056), (1000, 2080), (333, 4096), (130, 8192 + 64)]

# The decode kernels (m <= 16) selectable through q4_set_decode_kernel.
DECODE_KERNELS = {"warp_mma": 1, "cuda_core": 2, "tcgen05": 3, "record_mma": 4, "matvec": 5}


@pytest.fixture(params=sorted(DECODE_KERNELS))
def decode_kernel(request, q4lib):
    """Run the test once per decode kernel; the library's own choice again after."""
    q4lib.q4_set_decode_kernel(DECODE_KERNELS[request.param])
    yield request.param
    q4lib.q4_set_decode_kernel(q4lib.Q4_DECODE_AUTO)


def once_for_prefill(decode_kernel, m):
    """m > 16 takes the GEMM under an explicitly chosen decode kernel (the
    default dispatch may serve 17..32 rows with mat-vec pieces instead, which
    test_pieces_dispatch covers): run such a case under one of them."""
    if m > 16 and decode_kernel != "warp_mma":
        pytest.skip("prefill case: decode kernel irrelevant")
    if decode_kernel == "cuda_core" and m > 4:
        pytest.skip("this kernel serves m <= 4")



@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("n,k", SHAPES)
def test_decode_parity(q4lib, oracle_mod, decode_kernel, m, n, k):
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=1000 + n)
    X = synth.activations(m, k, seed=2000 + m)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, f"{decode_kernel} m={m} n={n} k={k}")


@pytest.mark.parametrize("kind,m,n,k,rtol", [
    ("cuda_core", 1, 9728, 2560, 2e-5), ("cuda_core", 2, 14336, 4096, 2e-5),
    ("cuda_core", 3, 2560, 9728, 2e-5), ("cuda_core", 4, 151936, 256, 2e-5),
    ("warp_mma", 1, 9728, 2560, 1e-4), ("warp_mma", 4, 2560, 9728, 1e-4),
    ("record_mma", 1, 9728, 2560, 1e-4), ("record_mma", 3, 14336, 4096, 1e-4),
    ("record_mma", 6, 2560, 9728, 1e-4), ("record_mma", 8, 14336, 4096, 1e-4),
    ("record_mma", 13, 9728, 2560, 1e-4), ("record_mma", 16, 1000, 2080, 1e-4),
    ("warp_mma", 9, 14336, 4096, 1e-4), ("warp_mma", 16, 1000, 2080, 1e-4),
    ("matvec", 1, 9728, 2560, 1e-4), ("matvec", 2, 2560, 9728, 1e-4), ("matvec", 3, 14336, 4096, 1e-4),
    ("matvec", 6, 2560, 9728, 1e-4), ("matvec", 8, 14336, 4096, 1e-4), ("matvec", 13, 9728, 2560, 1e-4),
    ("matvec", 16, 1000, 2080, 1e-4)])
def test_decode_kernel_accuracy_margin(q4lib, oracle_mod, kind, m, n, k, rtol):
    """The CUDA-core kernel forms (q - 8) exactly and multiplies fp32 X
    unrounded; the warp-MMA kernels form (q - 8) exactly and keep 22 bits of
    X per block (16 in the mat-vec's fixed-point split, with exact block dot
    products): all stay far inside the decode bound (checked at rtol)."""
    blocks = synth.q4_0_blocks(n, k, seed=91)
    X = synth.activations(m, k, seed=92)
    W = pack_dev(q4lib, blocks, n, k)
    q4lib.q4_set_decode_kernel(DECODE_KERNELS[kind])
    try:
        Y = run_matmul(q4lib, W, X, n).astype(np.float64)
    finally:
        q4lib.q4_set_decode_kernel(q4lib.Q4_DECODE_AUTO)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    ratio = float((np.abs(Y - Yr) / (rtol * B + 1e-7)).max())
    assert ratio <= 1.0, f"{kind} m={m}: max err / ({rtol} B + 1e-7) = {ratio:.3g}"


@pytest.mark.parametrize("m", [17, 31, 64, 100, 257, 300])
@pytest.mark.parametrize("n,k", [(64, 64), (65, 96), (200, 1056), (513, 2080), (260, 640)])
def test_prefill_parity(q4lib, oracle_mod, m, n, k):
    blocks = synth.q4_0_blocks(n, k, seed=3000 + n)
    X = synth.activations(m, k, seed=4000 + m)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, f"prefill m={m} n={n} k={k}")


# m = 896 over 76 row tiles plans 448-token tiles, too wide for the epilogue
# to stage in shared memory: those CTAs store Y directly.
@pytest.mark.parametrize("m,n,k", [(896, 9728, 256)])
def test_prefill_wide_token_tile_sampled(q4lib, oracle_mod, m, n, k):
    blocks = synth.q4_0_blocks(n, k, seed=31)
    X = synth.activations(m, k, seed=32)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    r = np.random.default_rng(33)
    t = np.concatenate([r.integers(0, m, 4000), [0, m - 1, 447, 448, m - 1]])
    j = np.concatenate([r.integers(0, n, 4000), [0, n - 1, 127, 128, 0]])
    Yr, B = oracle_mod.matmul_sampled(blocks, X, n, k, t, j)
    assert_parity(Y[t, j], Yr, B, m, f"wide token tile m={m} n={n} k={k}")


# 17..32 rows under the default dispatch, which runs either the GEMM (with a
# K split on layers of few 128-row groups) or two mat-vec calls (16 rows,
# then the rest), whichever the planners estimate faster; plain rows and
# slot rows with padded strides, against the oracle element by element.
@pytest.mark.parametrize("m,n,k", [(17, 2560, 9728), (32, 2560, 9728), (24, 4096, 4096), (31, 260, 1024)])
def test_pieces_dispatch(q4lib, oracle_mod, m, n, k):
    q4lib.q4_set_decode_kernel(q4lib.Q4_DECODE_AUTO)
    blocks = synth.q4_0_blocks(n, k, seed=41)
    X = synth.activations(m, k, seed=42)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, f"pieces m={m} n={n} k={k}")
    slots = m + 9
    ldx, ldy = k + 8, n + 4
    Xs = np.zeros((slots, ldx), dtype=np.float32)
    Xs[:, :k] = synth.activations(slots, k, seed=43)
    ids = synth.slot_ids(m, slots, seed=44)
    sentinel = np.float32(-12345.5)
    Yd = torch.full((slots, ldy), float(sentinel), dtype=torch.float32, device="cuda")
    ws, wsb = q4lib.workspace_for(m, k, n)
    q4lib.q4_0_matmul_batched_slots_ws(W, to_dev(Xs), ldx, to_dev(ids), m, Yd, ldy, k, n, ws, wsb)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status() == 0
    Ys = Yd.cpu().numpy()
    Yr2, B2 = oracle_mod.matmul(blocks, Xs[ids, :k], n, k)
    assert_parity(Ys[ids, :n], Yr2, B2, m, f"pieces slots m={m}")
    untouched = np.ones(slots, dtype=bool)
    untouched[ids] = False
    assert np.all(Ys[untouched] == sentinel), "rows of inactive slots were written"
    assert np.all(Ys[ids, n:] == sentinel), "padding columns of active rows were written"


def test_library_workspace_forms(q4lib, oracle_mod):
    for (m, n, k) in [(4, 2560, 9728), (40, 300, 1024), (1, 500, 256)]:
        blocks = synth.q4_0_blocks(n, k, seed=5)
        X = synth.activations(m, k, seed=6)
        W = pack_dev(q4lib, blocks, n, k)
        Y = run_matmul(q4lib, W, X, n, use_library_ws=True)
        Yr, B = oracle_mod.matmul(blocks, X, n, k)
        assert_parity(Y, Yr, B, m, f"library workspace m={m}")


# ----------------------------------------------------- workload sizes ----

FULL = [  # (m, n, k): oracle compares every element
    (1, 1024, 1024),     # single GEMV
    (1, 9728, 2560),     # decode up-projection
    (4, 9728, 2560),     # 4 slots, up-projection
    (4, 2560, 9728),     # 4 slots, down-projection (K split)
    (1, 14336, 4096), (2, 14336, 4096), (4, 14336, 4096), (8, 14336, 4096), (16, 14336, 4096),
]


@pytest.mark.parametrize("m,n,k", FULL)
def test_workload_sizes_full_compare(q4lib, oracle_mod, decode_kernel, m, n, k):
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=0)
    X = synth.activations(m, k, seed=0)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, f"m={m} n={n} k={k}")


@pytest.mark.parametrize("m,n,k", [(4, 151936, 2560), (16, 151936, 2560), (540, 9728, 2560)])
def test_workload_sizes_sampled(q4lib, oracle_mod, decode_kernel, m, n, k):
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=0)
    X = synth.activations(m, k, seed=0)
    W = pack_dev(q4lib, blocks, n, k)
    Y = run_matmul(q4lib, W, X, n)
    r = np.random.default_rng(7)
    cnt = 6000
    t = r.integers(0, m, cnt)
    j = r.integers(0, n, cnt)
    # always include the corners and the last row/column
    t = np.concatenate([t, [0, m - 1, 0, m - 1]])
    j = np.concatenate([j, [0, 0, n - 1, n - 1]])
    Yr, B = oracle_mod.matmul_sampled(blocks, X, n, k, t, j)
    assert_parity(Y[t, j], Yr, B, m, f"sampled m={m} n={n} k={k}")


# ------------------------------------------------- continuous batching ----

# pad = ldy - n. With ldy a multiple of 4 and n not, the prefill epilogue's
# 16-byte row-quad stores meet a last quad that is only partly inside Y's
# n columns (130 = 4 * 32 + 2, 514 = 4 * 128 + 2).
@pytest.mark.parametrize("m,slots,n,k,pad", [(1, 8, 300, 512, 5), (4, 40, 9728, 2560, 5), (16, 20, 200, 4096, 5),
                                             (4, 12, 2560, 9728, 5), (20, 64, 260, 1024, 5), (37, 40, 130, 640, 5),
                                             (37, 40, 130, 640, 2), (300, 320, 514, 1056, 2), (64, 64, 256, 512, 4)])
def test_batched_slots(q4lib, oracle_mod, decode_kernel, m, slots, n, k, pad):
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=11)
    ldx, ldy = k + 8, n + pad
    Xs = np.zeros((slots, ldx), dtype=np.float32)
    Xs[:, :k] = synth.activations(slots, k, seed=12)
    ids = synth.slot_ids(m, slots, seed=13)
    W = pack_dev(q4lib, blocks, n, k)
    Xd = to_dev(Xs)
    sentinel = np.float32(-12345.5)
    Yd = torch.full((slots, ldy), float(sentinel), dtype=torch.float32, device="cuda")
    idd = to_dev(ids)
    ws, wsb = q4lib.workspace_for(m, k, n)
    q4lib.q4_0_matmul_batched_slots_ws(W, Xd, ldx, idd, m, Yd, ldy, k, n, ws, wsb)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status() == 0
    Y = Yd.cpu().numpy()
    Yr, B = oracle_mod.matmul(blocks, Xs[ids, :k], n, k)
    assert_parity(Y[ids, :n], Yr, B, m, f"slots m={m}")
    untouched = np.ones(slots, dtype=bool)
    untouched[ids] = False
    assert np.all(Y[untouched] == sentinel), "rows of inactive slots were written"
    assert np.all(Y[ids, n:] == sentinel), "padding columns of active rows were written"


# ------------------------------------------------------ degenerate cases ----

def test_m_zero_is_a_no_op(q4lib):
    n, k = 64, 64
    W = pack_dev(q4lib, synth.q4_0_blocks(n, k), n, k)
    X = torch.zeros((1, k), dtype=torch.float32, device="cuda")
    Y = torch.full((1, n), 3.0, dtype=torch.float32, device="cuda")
    q4lib.q4_0_matmul(W, X, Y, 0, k, n)
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0)


@pytest.mark.parametrize("m", [1, 2, 4, 7, 16, 17, 100])
def test_all_eights_give_exact_zero(q4lib, decode_kernel, m):
    once_for_prefill(decode_kernel, m)
    n, k = 130, 640
    blocks = synth.q4_0_blocks(n, k, seed=21)
    blocks[:, :, 2:] = 0x88
    X = synth.activations(m, k, seed=22)
    Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    assert np.all(Y == 0.0)


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 16, 17, 64, 300])
def test_exact_integer_case_is_bit_exact(q4lib, oracle_mod, decode_kernel, m):
    """Power-of-two scales and small integer X: every partial sum is an exact
    integer times a power of two, on every path, so the results are equal."""
    once_for_prefill(decode_kernel, m)
    n, k = 200, 1024
    blocks = synth.q4_0_blocks(n, k, seed=31)
    nb = k // 32
    e = (synth.draw_u64(31, 9, n * nb) % np.uint64(6)).astype(np.int64) - 8
    d = np.ldexp(1.0, e).astype(np.float16).reshape(n, nb)
    blocks[:, :, 0:2] = d.astype("<f2").view(np.uint8).reshape(n, nb, 2)
    xi = (synth.draw_u64(32, 9, m * k) % np.uint64(33)).astype(np.int64) - 16
    X = xi.astype(np.float32).reshape(m, k)
    Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, _ = oracle_mod.matmul(blocks, X, n, k)
    assert np.array_equal(Y.astype(np.float64), Yr)


@pytest.mark.parametrize("m", [1, 3, 5, 16, 17, 64])
def test_nonfinite_x_propagates(q4lib, oracle_mod, decode_kernel, m):
    once_for_prefill(decode_kernel, m)
    n, k = 100, 256
    blocks = synth.q4_0_blocks(n, k, seed=41)
    X = synth.activations(m, k, seed=42)
    X[0, 5] = np.nan
    if m > 1:
        X[m - 1, 77] = np.inf
    Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, "non-finite X")


@pytest.mark.parametrize("m", [3, 6, 33])
def test_zero_and_negative_scales(q4lib, oracle_mod, decode_kernel, m):
    once_for_prefill(decode_kernel, m)
    n, k = 96, 512
    blocks = synth.q4_0_blocks(n, k, seed=51)
    blocks[::3, ::2, 0:2] = 0                       # d = +0
    blocks[1::3, :, 1] |= 0x80                      # d negative
    X = synth.activations(m, k, seed=52)
    Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, "zero/negative scales")


@pytest.mark.parametrize("m,n,k", [(1, 9728, 2560), (2, 2560, 9728), (4, 2560, 9728), (8, 2560, 9728),
                                   (16, 14336, 4096), (540, 9728, 2560)])
def test_bitwise_deterministic(q4lib, decode_kernel, m, n, k):
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=61)
    X = synth.activations(m, k, seed=62)
    W = pack_dev(q4lib, blocks, n, k)
    Y1 = run_matmul(q4lib, W, X, n)
    Y2 = run_matmul(q4lib, W, X, n)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))


@pytest.mark.parametrize("m,n,k", [(1, 9728, 2560), (4, 2560, 9728), (8, 2560, 9728), (16, 1000, 2080),
                                   (100, 1000, 2080)])
def test_weight_prefetch_mode_gives_identical_results(q4lib, oracle_mod, decode_kernel, m, n, k):
    """Streaming W before the preceding kernel finishes changes timing only."""
    once_for_prefill(decode_kernel, m)
    blocks = synth.q4_0_blocks(n, k, seed=81)
    X = synth.activations(m, k, seed=82)
    W = pack_dev(q4lib, blocks, n, k)
    torch.cuda.synchronize()
    Y0 = run_matmul(q4lib, W, X, n)
    try:
        q4lib.q4_set_weight_prefetch(True)
        Y1 = run_matmul(q4lib, W, X, n)
        Y2 = run_matmul(q4lib, W, X, n)
    finally:
        q4lib.q4_set_weight_prefetch(False)
    assert np.array_equal(Y0.view(np.uint32), Y1.view(np.uint32))
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y1, Yr, B, m, "prefetch mode")


def test_bounded_wait_reports_timeout_and_context_survives(q4lib, oracle_mod):
    import time
    q4lib.q4_last_device_status(clear=True)
    t0 = time.time()
    q4lib.q4_selftest_wait_timeout(5_000_000)       # 5 ms
    assert q4lib.q4_last_device_status(clear=True) == q4lib.Q4_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 5.0
    # the context still works
    n, k, m = 64, 128, 2
    blocks = synth.q4_0_blocks(n, k, seed=71)
    X = synth.activations(m, k, seed=72)
    Y = run_matmul(q4lib, pack_dev(q4lib, blocks, n, k), X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, "after timeout")


@pytest.mark.parametrize("m,n,k", [(1, 14336, 4096), (4, 2560, 9728), (16, 1000, 2080)])
def test_matvec_wait_limit_reports_timeout_and_context_survives(q4lib, oracle_mod, m, n, k):
    """The decode mat-vec's own bounded waits (ring slots, the warps' partial
    rows, the K slices' exchange) give up at a 1 ns limit: the call reports
    Q4_ERR_DEVICE_TIMEOUT through the status word instead of hanging, still
    lets every copy already in flight land, and the next call with the
    default limit is correct."""
    blocks = synth.q4_0_blocks(n, k, seed=81)
    X = synth.activations(m, k, seed=82)
    W = pack_dev(q4lib, blocks, n, k)
    q4lib.q4_last_device_status(clear=True)
    q4lib.q4_set_decode_kernel(q4lib.Q4_DECODE_MATVEC)
    Xd = to_dev(X)
    Yd = torch.empty((m, n), dtype=torch.float32, device="cuda")
    q4lib.q4_set_wait_limit_ns(1)
    try:
        q4lib.q4_0_matmul(W, Xd, Yd, m, k, n)
        status = q4lib.q4_last_device_status(clear=True)
    finally:
        q4lib.q4_set_wait_limit_ns(2_000_000_000)
        q4lib.q4_set_decode_kernel(q4lib.Q4_DECODE_AUTO)
    assert status == q4lib.Q4_ERR_DEVICE_TIMEOUT
    Y = run_matmul(q4lib, W, X, n)
    assert q4lib.q4_last_device_status(clear=True) == 0
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, "after a wait gave up")


# -------------------------------------------------------- expert groups ----

def test_expert_groups_match_the_oracle(q4lib, oracle_mod):
    """Rows grouped by expert, groups of 0 to 40 rows (decode and prefill
    sizes, empty experts), each checked at its size's tolerance."""
    n, k = 200, 1056
    sizes = [0, 1, 3, 16, 17, 40, 0, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    rows = int(offsets[-1])
    experts = [synth.q4_0_blocks(n, k, seed=700 + e) for e in range(len(sizes))]
    W = [pack_dev(q4lib, b, n, k) if s else None for b, s in zip(experts, sizes)]
    X = synth.activations(rows, k, seed=701)
    Xd = to_dev(X)
    Y = torch.full((rows, n), float("nan"), dtype=torch.float32, device="cuda")
    q4lib.q4_0_matmul_experts(W, offsets, Xd, Y, k, n)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    Y = Y.cpu().numpy()
    Yr, B = oracle_mod.matmul_experts(experts, X, offsets, n, k)
    for e, s in enumerate(sizes):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if s:
            assert_parity(Y[a:b], Yr[a:b], B[a:b], s, f"expert {e} ({s} rows)")


@pytest.mark.parametrize("n,k,sizes", [
    (130, 640, [1, 0, 2, 3, 4, 5, 8, 16, 1, 9]),                           # one launch for all
    (200, 1056, [(e * 7) % 17 for e in range(40)]),                         # two sets of <= 32
    (9728, 2560, [1, 3, 0, 16, 5, 2, 8, 4]),                                # the layer's size
    (96, 2080, [20, 1, 33, 2]),                                             # with GEMM-sized groups
    (130, 640, [17, 32, 33, 1, 23, 40]),                                    # both sides of the 32-row switch
])
def test_expert_sets_match_the_oracle(q4lib, oracle_mod, n, k, sizes):
    """Experts of up to 32 rows run the mat-vec in pieces of at most 16 rows,
    pieces of one instance sharing a launch per set of up to 32 (a cluster
    per group of a piece); larger ones the GEMM. Each group is checked at its
    size's tolerance, and rows of other groups are not touched."""
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    rows = int(offsets[-1])
    experts = [synth.q4_0_blocks(n, k, seed=900 + e) if s_ else None for e, s_ in enumerate(sizes)]
    W = [pack_dev(q4lib, b, n, k) if b is not None else None for b in experts]
    X = synth.activations(rows, k, seed=901)
    Y = torch.full((rows, n), float("nan"), dtype=torch.float32, device="cuda")
    q4lib.q4_0_matmul_experts(W, offsets, to_dev(X), Y, k, n)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    Y = Y.cpu().numpy()
    for e, s_ in enumerate(sizes):
        if s_:
            a, b = int(offsets[e]), int(offsets[e + 1])
            Yr, B = oracle_mod.matmul(experts[e], X[a:b], n, k)
            assert_parity(Y[a:b], Yr, B, s_, f"expert {e} ({s_} rows)")
