"""Seeded input generators, and the oracle's packed-layout reference checked
element by element against the layout's written specification."""

import numpy as np

from q4_quantized_linear_gb300 import synth


def test_generators_are_deterministic_and_seeded():
    a = synth.q4_0_blocks(33, 96, seed=0)
    b = synth.q4_0_blocks(33, 96, seed=0)
    c = synth.q4_0_blocks(33, 96, seed=1)
    assert a.shape == (33, 3, 18) and np.array_equal(a, b) and not np.array_equal(a, c)
    x = synth.activations(3, 64, seed=0)
    assert x.dtype == np.float32 and np.array_equal(x, synth.activations(3, 64, seed=0))


def test_generator_distributions():
    blocks = synth.q4_0_blocks(256, 1024, seed=0)
    qs = blocks[:, :, 2:]
    nib = np.concatenate([(qs & 0xF).ravel(), (qs >> 4).ravel()])
    counts = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(counts - 1 / 16) < 0.003)
    d = blocks[:, :, 0:2].copy().view("<f2").astype(np.float64).ravel()
    assert np.all(d >= 0)
    # E|N(0,1)| = sqrt(2/pi)
    assert abs(d.mean() / 0.02 - np.sqrt(2 / np.pi)) < 0.02
    x = synth.activations(64, 4096, seed=0).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_slot_ids_distinct():
    s = synth.slot_ids(16, 40, seed=0)
    assert s.dtype == np.int32 and len(set(s.tolist())) == 16 and s.min() >= 0 and s.max() < 40


def _locate(row, blk, elem):
    """Record, byte offset and nibble shift of weight (row, blk, elem) in the
    packed layout, from its specification (128-row groups, 64-k pairs,
    4608-byte records: 512 bytes of scale pairs, then 16 bytes per row for the
    pair's first block, then 16 bytes per row for its second)."""
    G, r = divmod(row, 128)
    p, b2 = divmod(blk, 2)
    shift = 0 if elem < 16 else 4
    return (G, p), 512 + 2048 * b2 + 16 * r + elem % 16, shift


def test_pack_reference_matches_specification(oracle_mod):
    n, k = 140, 96           # ragged rows (140 = 128 + 12) and an odd block count (3)
    blocks = synth.q4_0_blocks(n, k, seed=5)
    packed = oracle_mod.pack_reference(blocks, n, k)
    groups, pairs = 2, 2
    assert packed.size == oracle_mod.packed_size(n, k) == groups * pairs * 4608
    rec = packed.reshape(groups, pairs, 4608)
    nb = k // 32
    seen = np.zeros(packed.size, dtype=np.int32)
    for row in range(groups * 128):
        for blk in range(pairs * 2):
            (G, p), _, _ = _locate(row, blk, 0)
            r = row % 128
            off = 4 * r + 2 * (blk % 2)
            dbits = rec[G, p, off] | (rec[G, p, off + 1].astype(np.int64) << 8)
            real = row < n and blk < nb
            want_d = (blocks[row, blk, 0] | (blocks[row, blk, 1].astype(np.int64) << 8)) if real else 0
            assert dbits == want_d
            for elem in range(32):
                (G, p), off, shift = _locate(row, blk, elem)
                q = (rec[G, p, off] >> shift) & 0xF
                if real:
                    src = blocks[row, blk, 2 + elem % 16]
                    want = (src & 0xF) if elem < 16 else (src >> 4)
                else:
                    want = 8
                assert q == want, (row, blk, elem)
                seen[(G * pairs + p) * 4608 + off] += 1
    # every nibble byte is hit exactly twice (low and high nibble)
    nib_bytes = np.concatenate([np.arange(512, 4608) + r * 4608 for r in range(groups * pairs)])
    assert np.all(seen[nib_bytes] == 2)
