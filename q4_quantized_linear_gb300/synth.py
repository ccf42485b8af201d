"""Seeded synthetic inputs for the Q4_0 linear layer.

This module draws random bits and random reals and lays them out as GGUF
Q4_0 weight blocks and fp32 activation rows. It holds none of the layer's
own arithmetic (no dequantisation, no dot products): both the CPU oracle
and the CUDA path receive the very same bytes from here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: element i of a stream is mix64(key + (i + 1) * GAMMA), where the
stream key is itself mix64 of (seed, stream id). That makes every draw a
pure function of (seed, stream, index), so numpy can produce millions of
them at once and any subset can be recomputed on its own.

Normal variates use the Box-Muller transform in float64 on two uniforms in
(0, 1] built from the top 53 bits of a draw.

Workload recipe (the configurations the layer is measured on):
  nibbles  uniform over 0..15 (4 random bits each)
  scale d  fp16(|N(0,1)| * 0.02), rounded to nearest even by numpy
  X        fp32(N(0,1)), rounded to nearest even by numpy
"""

from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_NIBBLES = 0
STREAM_SCALES = 1
STREAM_X = 2

BLOCK_K = 32          # weights per Q4_0 block
BLOCK_BYTES = 18      # 2-byte fp16 scale + 16 bytes of nibbles


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) & 0xFFFFFFFF) << 32 | (int(stream) & 0xFFFFFFFF)],
                    dtype=np.uint64)
    return mix64(mix64(base) + GAMMA)[0]


def draw_u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """Draws offset .. offset+count-1 of stream (seed, stream) as uint64."""
    key = stream_key(seed, stream)
    idx = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + idx * GAMMA)


def uniform01(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """Uniform float64 in (0, 1] from the top 53 bits of each draw."""
    r = draw_u64(seed, stream, count, offset)
    return ((r >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """count standard normal float64 values (Box-Muller, both branches)."""
    pairs = (count + 1) // 2
    u = uniform01(seed, stream, 2 * pairs)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = rad * np.cos(ang)
    z[1::2] = rad * np.sin(ang)
    return z[:count]


def q4_0_blocks(n: int, k: int, seed: int = 0, scale_sigma: float = 0.02) -> np.ndarray:
    """GGUF Q4_0 weight matrix W[n x k] as uint8 array of shape (n, k/32, 18).

    Per block: bytes 0..1 = d as little-endian fp16, bytes 2..17 = qs[16].
    """
    if k % BLOCK_K:
        raise ValueError("k must be a multiple of 32")
    nb = k // BLOCK_K
    nblk = n * nb
    qs = draw_u64(seed, STREAM_NIBBLES, 2 * nblk).astype("<u8").view(np.uint8)
    qs = qs.reshape(n, nb, 16)
    d = (np.abs(normal(seed, STREAM_SCALES, nblk)) * scale_sigma).astype(np.float16)
    dbytes = d.astype("<f2").view(np.uint8).reshape(n, nb, 2)
    out = np.empty((n, nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = dbytes
    out[:, :, 2:] = qs
    return out


def activations(m: int, k: int, seed: int = 0) -> np.ndarray:
    """X[m x k] fp32 standard normal, row-major."""
    return normal(seed, STREAM_X, m * k).astype(np.float32).reshape(m, k)


def slot_ids(m: int, num_slots: int, seed: int = 0) -> np.ndarray:
    """m distinct slot indices in [0, num_slots), int32, in a seeded order."""
    if m > num_slots:
        raise ValueError("more active rows than slots")
    keys = draw_u64(seed, 3, num_slots)
    return np.argsort(keys, kind="stable")[:m].astype(np.int32)


def blocks_from_parts(d_bits: np.ndarray, qs: np.ndarray) -> np.ndarray:
    """Assemble blocks from raw fp16 scale bits (uint16, shape (n, nb)) and
    nibble bytes (uint8, shape (n, nb, 16)). Used for hand-built cases."""
    d_bits = np.asarray(d_bits, dtype=np.uint16)
    qs = np.asarray(qs, dtype=np.uint8)
    n, nb = d_bits.shape
    out = np.empty((n, nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d_bits.astype("<u2").view(np.uint8).reshape(n, nb, 2)
    out[:, :, 2:] = qs
    return out
