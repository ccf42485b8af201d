"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin is a plain function that raises AssertionError on a mismatch, so
the last test can re-run all of them with one deliberate mistake switched
into the oracle and check that every mistake is caught by some pin.

Pins used:
  * hand-derived goldens (tests/golden/): a split-half block and its dot
    products, fixed facts of the nibble offset and of binary16;
  * the nibble order, exhaustively over every byte position and value;
  * binary16 decode, exhaustively over all 65,536 bit patterns, against
    numpy's float16 (a library routine);
  * an exact integer closed form (power-of-two scales, small integer X),
    evaluated with Python integers;
  * a brute-force special case: the product reduces to numpy's matmul of
    the dequantised matrix, which numpy builds from the bytes by itself;
  * invariants: exact power-of-two homogeneity, oddness in X and in d,
    linearity in X, B >= |Y| with equality for same-sign terms;
  * for the W4A8 variant: hand-derived codes and products (round-half-even
    ties, a scale per block), all-eights gives zero, integer-coded X reduces
    it to the exact product above, power-of-two homogeneity, NaN rows, and
    the coding error bound against the exact product.
"""

import json
import os

import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _numpy_dequant(blocks, n, k):
    """Dense W[n x k] built from the bytes with numpy alone (library fp16)."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(n, k // 32, 18)
    d = b[:, :, 0:2].copy().view("<f2").astype(np.float64)[:, :, 0]
    qs = b[:, :, 2:].astype(np.int64)
    q = np.concatenate([qs & 0xF, qs >> 4], axis=2)  # elements 0..15, then 16..31
    return ((q - 8).astype(np.float64) * d[:, :, None]).reshape(n, k)


# ---------------------------------------------------------------- pins ----

def pin_golden_block(orc):
    g = _golden("split_half_block.json")
    blocks = synth.blocks_from_parts(np.array([[g["d_bits"]]]), np.array([[g["qs"]]]))
    W = orc.dequant_matrix(blocks, 1, 32)
    assert np.array_equal(W[0], np.array(g["w"])), "split-half golden block"
    X = np.stack([np.ones(32), np.arange(32)]).astype(np.float32)
    Y, B = orc.matmul(blocks, X, 1, 32)
    assert Y[0, 0] == g["dot_ones"] and Y[1, 0] == g["dot_index"], "golden dot products"
    assert B[0, 0] == g["bound_ones"], "golden magnitude sum"


def pin_format_facts(orc):
    g = _golden("format_facts.json")
    for nib, w in g["nibble_weight_d1"].items():
        qs = np.full((1, 1, 16), 0x88, dtype=np.uint8)
        qs[0, 0, 3] = (0x80 | int(nib))          # element 3 carries the nibble
        blocks = synth.blocks_from_parts(np.array([[0x3C00]]), qs)
        X = np.zeros((1, 32), dtype=np.float32)
        X[0, 3] = 1.0
        Y, _ = orc.matmul(blocks, X, 1, 32)
        assert Y[0, 0] == w, f"nibble {nib} with d = 1"
    for bits, val in g["fp16"].items():
        got = orc.fp16_to_double(int(bits, 16))
        if val == "nan":
            assert np.isnan(got), bits
        else:
            want = float(val)
            assert got == want and np.signbit(got) == np.signbit(want), bits


def pin_all_eights_is_zero(orc):
    n, k, m = 7, 96, 3
    rng_blocks = synth.q4_0_blocks(n, k, seed=11)
    rng_blocks[:, :, 2:] = 0x88
    X = synth.activations(m, k, seed=12)
    Y, B = orc.matmul(rng_blocks, X, n, k)
    assert np.all(Y == 0.0) and np.all(B == 0.0), "all nibbles 8 must give exactly 0"


def pin_nibble_order(orc):
    """Every byte position j, both nibbles, every value v: with d = 1 and the
    other nibbles 8, element j (low) or j+16 (high) is v - 8, all else 0.
    X = identity, so Y is the dense W transposed."""
    rows = []
    expect = []
    for high in (0, 1):
        for j in range(16):
            for v in range(16):
                qs = np.full(16, 0x88, dtype=np.uint8)
                qs[j] = ((v << 4) | 0x8) if high else (0x80 | v)
                rows.append(qs)
                e = np.zeros(32)
                e[j + 16 * high] = v - 8
                expect.append(e)
    n = len(rows)
    blocks = synth.blocks_from_parts(np.full((n, 1), 0x3C00), np.array(rows)[:, None, :])
    X = np.eye(32, dtype=np.float32)
    Y, _ = orc.matmul(blocks, X, n, 32)
    assert np.array_equal(Y.T, np.array(expect)), "split-half nibble order"


def pin_fp16_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "binary16 NaN set"
    assert np.array_equal(got[~nan], ref[~nan]), "binary16 values"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "binary16 signs"


def pin_exact_integer(orc):
    """d = 2^e, X small integers: Y = 2^e * sum (q-8) x exactly (Python ints)."""
    n, k, m = 9, 160, 4
    blocks = synth.q4_0_blocks(n, k, seed=21)
    nb = k // 32
    exps = (synth.draw_u64(21, 9, n * nb) % np.uint64(16)).astype(np.int64) - 10
    d = np.ldexp(1.0, exps).astype(np.float16).reshape(n, nb)
    blocks[:, :, 0:2] = d.astype("<f2").view(np.uint8).reshape(n, nb, 2)
    xi = (synth.draw_u64(22, 9, m * k) % np.uint64(17)).astype(np.int64) - 8
    X = xi.astype(np.float32).reshape(m, k)
    Y, _ = orc.matmul(blocks, X, n, k)
    qs = blocks[:, :, 2:].astype(np.int64)
    for j in range(n):
        for t in range(m):
            total = 0
            for b in range(nb):
                acc = 0
                for i in range(32):
                    q = int(qs[j, b, i] & 0xF) if i < 16 else int(qs[j, b, i - 16] >> 4)
                    acc += (q - 8) * int(xi[t * k + 32 * b + i])
                e = int(exps[j * nb + b])
                total += acc * 2 ** e if e >= 0 else acc / 2 ** (-e)
            assert Y[t, j] == total, f"exact integer case ({t}, {j})"


def pin_numpy_special_case(orc):
    for (m, n, k) in [(1, 1, 32), (2, 3, 64), (3, 5, 96), (5, 2, 32), (4, 7, 128)]:
        blocks = synth.q4_0_blocks(n, k, seed=31 + n)
        X = synth.activations(m, k, seed=41 + m)
        Y, B = orc.matmul(blocks, X, n, k)
        W = _numpy_dequant(blocks, n, k)
        X64 = X.astype(np.float64)
        Yr = X64 @ W.T
        Br = np.abs(X64) @ np.abs(W).T
        assert np.allclose(Y, Yr, rtol=1e-12, atol=1e-15), f"numpy matmul ({m},{n},{k})"
        assert np.allclose(B, Br, rtol=1e-12, atol=1e-15), f"numpy bound ({m},{n},{k})"


def pin_invariants(orc):
    n, k, m = 13, 192, 3
    blocks = synth.q4_0_blocks(n, k, seed=51)
    X = synth.activations(m, k, seed=52)
    Y, B = orc.matmul(blocks, X, n, k)
    for p in (-3, 5):
        Yp, Bp = orc.matmul(blocks, np.ldexp(X, p), n, k)
        assert np.array_equal(Yp, np.ldexp(Y, p)), "power-of-two homogeneity in X"
        assert np.array_equal(Bp, np.ldexp(B, p)), "power-of-two homogeneity of B"
    Yn, Bn = orc.matmul(blocks, -X, n, k)
    assert np.array_equal(Yn, -Y) and np.array_equal(Bn, B), "odd in X"
    neg = blocks.copy()
    neg[:, :, 1] ^= 0x80                             # flip the sign bit of every d
    Yd, Bd = orc.matmul(neg, X, n, k)
    assert np.array_equal(Yd, -Y) and np.array_equal(Bd, B), "odd in d"
    X2 = synth.activations(m, k, seed=53)
    Y2, B2 = orc.matmul(blocks, X2, n, k)
    Ys, _ = orc.matmul(blocks, X + X2, n, k)
    # X + X2 is rounded to fp32, so linearity holds to that rounding
    Yx, _ = orc.matmul(blocks, (X + X2).astype(np.float32), n, k)
    assert np.allclose(Ys, Yx) and np.allclose(Ys, Y + Y2, rtol=1e-6, atol=1e-6 * B.max()), \
        "linearity in X"
    assert np.all(B >= np.abs(Y)) and np.all(B >= 0), "B bounds |Y|"
    # same-sign terms: |X| against weights with q >= 8 and d >= 0 makes B == Y
    pos = blocks.copy()
    pos[:, :, 2:] |= 0x88
    pos[:, :, 1] &= 0x7F
    Yq, Bq = orc.matmul(pos, np.abs(X), n, k)
    assert np.allclose(Yq, Bq, rtol=1e-15, atol=0), "B equals Y for same-sign terms"


def pin_sampled_matches_full(orc):
    n, k, m = 70, 320, 5
    blocks = synth.q4_0_blocks(n, k, seed=61)
    X = synth.activations(m, k, seed=62)
    Y, B = orc.matmul(blocks, X, n, k)
    t = np.array([0, 4, 2, 3, 1]); j = np.array([0, 69, 33, 64, 5])
    Ys, Bs = orc.matmul_sampled(blocks, X, n, k, t, j)
    assert np.array_equal(Ys, Y[t, j]) and np.array_equal(Bs, B[t, j]), "sampled == full"


# ---------------------------------------------------------------- W4A8 --

def _w4a8_blocks(k, d_bits, nibble=9):
    """One row of blocks: the given fp16 scale bits, every nibble the same."""
    nb = k // 32
    blocks = np.zeros((1, nb, 18), dtype=np.uint8)
    for b in range(nb):
        blocks[0, b, 0] = d_bits[b] & 0xFF
        blocks[0, b, 1] = d_bits[b] >> 8
        blocks[0, b, 2:] = nibble | (nibble << 4)
    return blocks


def pin_w4a8_golden(orc):
    """Hand-derived codes and products (tests/golden/w4a8_blocks.json)."""
    g = _golden("w4a8_blocks.json")
    for case in g["cases"]:
        k = case["k"]
        X = np.zeros((1, k), dtype=np.float32)
        for i, v in case["x_nonzero"].items():
            X[0, int(i)] = v
        codes, scales, bad = orc.quantize_x_w4a8(X, k)
        want = np.zeros(k, dtype=np.int8)
        for i, v in case["codes_nonzero"].items():
            want[int(i)] = v
        assert np.array_equal(codes[0], want), f"{case['name']}: codes {codes[0][codes[0] != 0]}"
        if "scale_block1" in case:
            assert float(scales[0, 1]) == case["scale_block1"], f"{case['name']}: scale"
        Y, B = orc.matmul_w4a8(_w4a8_blocks(k, case["d_bits"]), X, 1, k)
        assert abs(Y[0, 0] - case["y"]) <= 1e-12 * abs(case["y"]), f"{case['name']}: y {Y[0, 0]} != {case['y']}"


def pin_w4a8_all_eights_is_zero(orc):
    """Every nibble 8 means every weight 0, whatever X and d."""
    k = 96
    X = synth.activations(3, k, seed=81)
    Y, B = orc.matmul_w4a8(_w4a8_blocks(k, [0x3C00, 0x4400, 0xB800], nibble=8), X, 1, k)
    assert np.all(Y == 0.0) and np.all(B == 0.0), "all-eights W4A8 product is zero"


def pin_w4a8_integer_case_is_the_exact_product(orc):
    """Integer X with |x| <= 127 and some |x| = 127 in every block: the codes
    are X itself and every scale 1, so the W4A8 product is the exact product
    (pinned above); power-of-two d keeps every sum exact in fp64."""
    rng = np.random.default_rng(83)
    n, k, m = 9, 160, 4
    blocks = synth.q4_0_blocks(n, k, seed=84).reshape(n, k // 32, 18).copy()
    e = rng.integers(-6, 3, size=(n, k // 32))
    dbits = (2.0 ** e).astype(np.float16) * np.where(rng.random((n, k // 32)) < 0.5, -1, 1).astype(np.float16)
    raw = dbits.view(np.uint16)
    blocks[:, :, 0] = raw & 0xFF
    blocks[:, :, 1] = raw >> 8
    X = rng.integers(-126, 127, size=(m, k)).astype(np.float32)
    X[:, ::32] = np.where(rng.random((m, k // 32)) < 0.5, -127.0, 127.0)
    Y8, B8 = orc.matmul_w4a8(blocks, X, n, k)
    Y, B = orc.matmul(blocks, X, n, k)
    assert np.array_equal(Y8, Y), "integer-coded X: W4A8 equals the exact product"


def pin_w4a8_homogeneity_and_nan(orc):
    """X * 2^p scales every code's scale by 2^p and leaves the codes: Y * 2^p
    exactly. A row holding a NaN gives NaN outputs; other rows are unchanged."""
    n, k, m = 11, 128, 3
    blocks = synth.q4_0_blocks(n, k, seed=85)
    X = synth.activations(m, k, seed=86)
    Y, _ = orc.matmul_w4a8(blocks, X, n, k)
    Y2, _ = orc.matmul_w4a8(blocks, X * np.float32(8.0), n, k)
    assert np.array_equal(Y2, Y * 8.0), "W4A8 homogeneity"
    Xn = X.copy()
    Xn[1, 70] = np.nan
    Yn, _ = orc.matmul_w4a8(blocks, Xn, n, k)
    assert np.all(np.isnan(Yn[1])) and np.array_equal(Yn[[0, 2]], Y[[0, 2]]), "W4A8 NaN row"


def pin_w4a8_quantization_bound(orc):
    """|Y8 - Y| <= sum_b |d| * s_b / 2 * sum_i |q - 8| (each code within half a
    step of x / s), with a little slack for fp64 rounding."""
    n, k, m = 13, 256, 3
    blocks = synth.q4_0_blocks(n, k, seed=87)
    X = synth.activations(m, k, seed=88)
    Y8, _ = orc.matmul_w4a8(blocks, X, n, k)
    Y, _ = orc.matmul(blocks, X, n, k)
    codes, scales, bad = orc.quantize_x_w4a8(X, k)
    W = orc.dequant_matrix(blocks, n, k)                       # (q - 8) * d, [n x k]
    bound = np.zeros((m, n))
    for b in range(k // 32):
        Wb = np.abs(W[:, 32 * b:32 * b + 32]).sum(axis=1)     # |d| * sum |q - 8|
        bound += np.outer(scales[:, b].astype(np.float64) / 2, Wb)
    assert np.all(np.abs(Y8 - Y) <= bound * (1 + 1e-9) + 1e-12), "W4A8 within the coding bound"


def pin_experts_offsets(orc):
    """Expert grouping: with every expert holding the same weights the grouped
    product is the plain one; changing one expert's weights changes exactly
    its own rows; empty groups are allowed."""
    n, k = 23, 96
    X = synth.activations(9, k, seed=91)
    W = synth.q4_0_blocks(n, k, seed=92)
    offsets = [0, 2, 2, 7, 9]
    Y, _ = orc.matmul(W, X, n, k)
    Ye, _ = orc.matmul_experts([W, W, W, W], X, offsets, n, k)
    assert np.array_equal(Ye, Y), "same weights: grouped == plain"
    W2 = synth.q4_0_blocks(n, k, seed=93)
    Ye2, _ = orc.matmul_experts([W, W, W2, W], X, offsets, n, k)
    changed = np.any(Ye2 != Ye, axis=1)
    assert np.array_equal(changed, np.array([r in range(2, 7) for r in range(9)])), "one expert's rows only"
    Y2, _ = orc.matmul(W2, X, n, k)
    assert np.array_equal(Ye2[2:7], Y2[2:7]), "those rows are the plain product with that expert"


def pin_w8_codes_and_product(orc):
    """Per-channel int8 weights: a row whose largest |w| is 127 keeps integer
    weights as they are (scale 1), so the product is X . W^T exactly;
    hand-derived ties (amax 127: 2.5 -> 2, 3.5 -> 4, -0.5 -> 0, -1.5 -> -2)
    and one scale per row (a row with amax 1 gets scale fp32(1/127) and codes
    127, 64 for 1, 0.5); a zero row gives zeros; the coding bound holds."""
    W = np.array([[127.0, 2.5, 3.5, -0.5, -1.5] + [0.0] * 27,
                  [1.0, 0.5] + [0.0] * 30,
                  [0.0] * 32], dtype=np.float32)
    codes, scales = orc.quantize_w_int8(W)
    assert list(codes[0, :5]) == [127, 2, 4, 0, -2], "round half to even"
    assert list(codes[1, :2]) == [127, 64] and scales[1] == np.float32(1) / np.float32(127), "per-row scale"
    assert scales[0] == 1.0 and scales[2] == 0.0 and not codes[2].any(), "scale 1 and the zero row"
    rng = np.random.default_rng(95)
    Wi = rng.integers(-126, 127, size=(7, 64)).astype(np.float32)
    Wi[:, 0] = 127.0
    Xi = rng.integers(-20, 21, size=(3, 64)).astype(np.float32)
    c, s = orc.quantize_w_int8(Wi)
    Y, B = orc.matmul_w8(c, s, Xi)
    exact = (Xi.astype(np.int64) @ Wi.astype(np.int64).T).astype(np.float64)
    assert np.array_equal(Y, exact) and np.all(B >= np.abs(Y)), "integer rows are exact"
    Wf = synth.activations(9, 128, seed=96)
    X = synth.activations(4, 128, seed=97)
    c, s = orc.quantize_w_int8(Wf)
    Y8, _ = orc.matmul_w8(c, s, X)
    bound = (np.abs(X.astype(np.float64)) @ np.ones((128, 9))) * (s.astype(np.float64) / 2)[None, :]
    assert np.all(np.abs(Y8 - X.astype(np.float64) @ Wf.astype(np.float64).T) <= bound * (1 + 1e-9) + 1e-12), \
        "within half a step per weight"


PINS = [pin_golden_block, pin_format_facts, pin_all_eights_is_zero, pin_nibble_order,
        pin_fp16_exhaustive, pin_exact_integer, pin_numpy_special_case, pin_invariants,
        pin_sampled_matches_full, pin_w4a8_golden, pin_w4a8_all_eights_is_zero,
        pin_w4a8_integer_case_is_the_exact_product, pin_w4a8_homogeneity_and_nan, pin_w4a8_quantization_bound,
        pin_experts_offsets, pin_w8_codes_and_product]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle_mod, pin):
    oracle_mod.set_mutation(0)
    pin(oracle_mod)


def test_thread_count_does_not_change_bits(oracle_mod):
    n, k, m = 90, 256, 3
    blocks = synth.q4_0_blocks(n, k, seed=71)
    X = synth.activations(m, k, seed=72)
    Y1, B1 = oracle_mod.matmul(blocks, X, n, k, nthreads=1)
    Y4, B4 = oracle_mod.matmul(blocks, X, n, k, nthreads=4)
    assert np.array_equal(Y1, Y4) and np.array_equal(B1, B4)


def test_every_planted_mistake_is_caught(oracle_mod):
    """Switch in each deliberate mistake; at least one pin must fail."""
    cheap = [p for p in PINS if p is not pin_fp16_exhaustive] + [pin_fp16_exhaustive]
    uncaught = []
    try:
        for mut in range(1, oracle_mod.mutation_count()):
            oracle_mod.set_mutation(mut)
            caught = False
            for pin in cheap:
                try:
                    pin(oracle_mod)
                except AssertionError:
                    caught = True
                    break
            if not caught:
                uncaught.append(mut)
    finally:
        oracle_mod.set_mutation(0)
    assert not uncaught, f"mutations not caught by any pin: {uncaught}"
