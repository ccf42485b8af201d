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
    """Byte offset and nibble shift of weight (row, blk, elem) in the packed
    layout, from its specification (64-row groups, 64-k pairs, 16-row tiles,
    576-byte records: 64 bytes of scales then 32 lanes x 16 bytes)."""
    G, r = divmod(row, 64)
    t, r16 = divmod(r, 16)
    h, g = divmod(r16, 8)
    p, b2 = divmod(blk, 2)
    byte_in_qs = elem % 16
    shift = 0 if elem < 16 else 4
    c, byte_in_word = divmod(byte_in_qs, 4)
    lane = 4 * g + c
    word = b2 * 2 + h
    return ((G, p, t), 64 + lane * 16 + word * 4 + byte_in_word, shift)


def test_pack_reference_matches_specification(oracle_mod):
    n, k = 70, 96            # ragged rows (70 = 64 + 6) and an odd block count (3)
    blocks = synth.q4_0_blocks(n, k, seed=5)
    packed = oracle_mod.pack_reference(blocks, n, k)
    groups, pairs = 2, 2
    assert packed.size == oracle_mod.packed_size(n, k) == groups * pairs * 4 * 576
    rec = packed.reshape(groups, pairs, 4, 576)
    nb = k // 32
    seen = np.zeros(packed.size, dtype=np.int32)
    for row in range(groups * 64):
        for blk in range(pairs * 2):
            (G, p, t), _, _ = _locate(row, blk, 0)
            r16 = row % 16
            s = (r16 % 8) * 4 + (blk % 2) * 2 + r16 // 8
            dbits = rec[G, p, t, 2 * s] | (rec[G, p, t, 2 * s + 1].astype(np.int64) << 8)
            real = row < n and blk < nb
            want_d = (blocks[row, blk, 0] | (blocks[row, blk, 1].astype(np.int64) << 8)) if real else 0
            assert dbits == want_d
            for elem in range(32):
                (G, p, t), off, shift = _locate(row, blk, elem)
                q = (rec[G, p, t, off] >> shift) & 0xF
                if real:
                    src = blocks[row, blk, 2 + elem % 16]
                    want = (src & 0xF) if elem < 16 else (src >> 4)
                else:
                    want = 8
                assert q == want, (row, blk, elem)
                seen[((G * pairs + p) * 4 + t) * 576 + off] += 1
    # every nibble byte is hit exactly twice (low and high nibble)
    nib_bytes = np.concatenate([np.arange(64, 576) + r * 576 for r in range(groups * pairs * 4)])
    assert np.all(seen[nib_bytes] == 2)
