"""CPU oracle of the Q4_0 quantized linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it. The arithmetic lives in ``q4_oracle.c`` (plain C,
fp64, fixed summation order); this module compiles it with gcc and wraps it
with ctypes.

Functions and the passages they follow:
  matmul / matmul_sampled -- Y = X . W^T with W stored [n x k] (rembed
      "Architecture", "The pluggable kernel interface"), W in GGUF Q4_0
      blocks, nibble order from goinfer ch. 10 "Layout, concretely".
      Also returns B = sum |x_i w_i|, the magnitude the tolerances scale by.
  fp16_to_double -- IEEE 754 binary16 decode of the block scale.
  dequant_matrix -- the dense fp64 weight matrix (tiny shapes).
  matmul_w4a8 / quantize_x_w4a8 -- the activation-quantised variant: X
      coded per 32-element block to int8 (round-half-even of x * 127 / amax,
      scale amax / 127), integer dot products, fp64 outer sums (goinfer ch.
      10 "Which kernel runs is a runtime decision"; rembed "Architecture",
      "int8 quantization"; the coding rule is this oracle's reading).
  matmul_experts -- the expert-grouped product (golem-server, "Several
      conversations, in one pass"): rows grouped by expert, each group the
      plain product against its expert's weights.
  quantize_w_int8 / matmul_w8 -- per-output-channel symmetric int8 weights
      and their product with fp32 X (rembed "Architecture", "int8
      quantization"; the rounding rule is this oracle's reading).
  pack_reference -- byte-exact reference of the CUDA library's packed layout
      (goinfer ch. 10 "Making Go fast enough": weights repacked for the
      kernel's access order), written from the layout's specification.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_q4.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile q4_oracle.c into a shared library (gcc, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.q4o_set_mutation.argtypes = [ctypes.c_int]
        lib.q4o_set_mutation.restype = ctypes.c_int
        lib.q4o_mutation_count.restype = ctypes.c_int
        lib.q4o_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.q4o_fp16_to_double.restype = ctypes.c_double
        lib.q4o_matmul.argtypes = [P, P, I64, I64, I64, P, P, ctypes.c_int]
        lib.q4o_matmul.restype = ctypes.c_int
        lib.q4o_matmul_sampled.argtypes = [P, P, I64, I64, I64, P, P, I64, P, P, ctypes.c_int]
        lib.q4o_matmul_sampled.restype = ctypes.c_int
        lib.q4o_dequant_matrix.argtypes = [P, I64, I64, P]
        lib.q4o_dequant_matrix.restype = ctypes.c_int
        lib.q4o_packed_size.argtypes = [I64, I64]
        lib.q4o_packed_size.restype = ctypes.c_size_t
        lib.q4o_pack_reference.argtypes = [P, I64, I64, P]
        lib.q4o_pack_reference.restype = ctypes.c_int
        lib.q4o_num_threads.restype = ctypes.c_int
        lib.q4o_quantize_x_w4a8.argtypes = [P, I64, I64, P, P, P]
        lib.q4o_quantize_x_w4a8.restype = ctypes.c_int
        lib.q4o_matmul_w4a8.argtypes = [P, P, I64, I64, I64, P, P, ctypes.c_int]
        lib.q4o_matmul_w4a8.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_blocks(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.size != n * (k // 32) * 18:
        raise ValueError("blocks do not hold n x k/32 18-byte blocks")
    return blocks


def num_threads() -> int:
    return int(_load().q4o_num_threads())


def set_mutation(mutation: int) -> None:
    """Test-only: switch in one deliberate mistake (0 = none)."""
    if _load().q4o_set_mutation(int(mutation)) != 0:
        raise ValueError(f"unknown mutation {mutation}")


def mutation_count() -> int:
    return int(_load().q4o_mutation_count())


def fp16_to_double(bits: int) -> float:
    return float(_load().q4o_fp16_to_double(int(bits) & 0xFFFF))


def matmul(blocks: np.ndarray, X: np.ndarray, n: int, k: int, nthreads: int = 0):
    """(Y, B) in float64, both [m x n]."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    m = X.shape[0] if X.ndim == 2 else 0
    if X.ndim != 2 or X.shape[1] != k:
        raise ValueError("X must be [m x k]")
    blocks = _check_blocks(blocks, n, k)
    Y = np.empty((m, n), dtype=np.float64)
    B = np.empty((m, n), dtype=np.float64)
    rc = _load().q4o_matmul(_ptr(blocks), _ptr(X), m, k, n, _ptr(Y), _ptr(B), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"q4o_matmul failed ({rc})")
    return Y, B


def matmul_sampled(blocks: np.ndarray, X: np.ndarray, n: int, k: int,
                   t_idx: np.ndarray, j_idx: np.ndarray, nthreads: int = 0):
    """(Y, B) at the listed (t, j) elements, float64 vectors."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    m = X.shape[0]
    blocks = _check_blocks(blocks, n, k)
    t_idx = np.ascontiguousarray(t_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    Y = np.empty(t_idx.size, dtype=np.float64)
    B = np.empty(t_idx.size, dtype=np.float64)
    rc = _load().q4o_matmul_sampled(_ptr(blocks), _ptr(X), m, k, n, _ptr(t_idx), _ptr(j_idx),
                                    t_idx.size, _ptr(Y), _ptr(B), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"q4o_matmul_sampled failed ({rc})")
    return Y, B


def dequant_matrix(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = _check_blocks(blocks, n, k)
    W = np.empty((n, k), dtype=np.float64)
    if _load().q4o_dequant_matrix(_ptr(blocks), n, k, _ptr(W)) != 0:
        raise RuntimeError("q4o_dequant_matrix failed")
    return W


def packed_size(n: int, k: int) -> int:
    return int(_load().q4o_packed_size(n, k))


def pack_reference(blocks: np.ndarray, n: int, k: int) -> np.ndarray:
    blocks = _check_blocks(blocks, n, k)
    out = np.empty(packed_size(n, k), dtype=np.uint8)
    if _load().q4o_pack_reference(_ptr(blocks), n, k, _ptr(out)) != 0:
        raise RuntimeError("q4o_pack_reference failed")
    return out


def quantize_x_w4a8(X: np.ndarray, k: int):
    """int8 codes [m x k], fp32 scales [m x k/32] and per-row non-finite flags."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    m = X.shape[0]
    codes = np.zeros((m, k), dtype=np.int8)
    scales = np.zeros((m, k // 32), dtype=np.float32)
    bad = np.zeros(m, dtype=np.int32)
    rc = _load().q4o_quantize_x_w4a8(_ptr(X), m, k, _ptr(codes), _ptr(scales), _ptr(bad))
    if rc != 0:
        raise ValueError("bad sizes")
    return codes, scales, bad.astype(bool)


def matmul_w4a8(blocks: np.ndarray, X: np.ndarray, n: int, k: int, nthreads: int = 0):
    """(Y, B8): the W4A8 product and the per-element magnitude sum of its block terms."""
    blocks = _check_blocks(blocks, n, k)
    X = np.ascontiguousarray(X, dtype=np.float32)
    m = X.shape[0]
    Y = np.zeros((m, n), dtype=np.float64)
    B = np.zeros((m, n), dtype=np.float64)
    rc = _load().q4o_matmul_w4a8(_ptr(blocks), _ptr(X), m, k, n, _ptr(Y), _ptr(B), nthreads)
    if rc != 0:
        raise ValueError("bad sizes")
    return Y, B


def matmul_experts(expert_blocks, X: np.ndarray, offsets, n: int, k: int):
    """Expert-grouped product (golem-server, "Several conversations, in one
    pass": a mixture reads each expert once for the columns that chose it):
    X's rows are grouped by expert, rows offsets[e] .. offsets[e+1]-1 going to
    expert e, and Y[r] = X[r] . W_e^T for those rows. Each group is the plain
    product above on its rows. Returns (Y, B)."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    offsets = [int(o) for o in offsets]
    if offsets[0] != 0 or offsets[-1] != X.shape[0] or any(a > b for a, b in zip(offsets, offsets[1:])):
        raise ValueError("offsets must rise from 0 to the row count")
    if len(offsets) != len(expert_blocks) + 1:
        raise ValueError("one offset per expert, plus the end")
    Y = np.zeros((X.shape[0], n), dtype=np.float64)
    B = np.zeros((X.shape[0], n), dtype=np.float64)
    for e, blocks in enumerate(expert_blocks):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            Y[a:b], B[a:b] = matmul(blocks, X[a:b], n, k)
    return Y, B


def quantize_w_int8(W: np.ndarray):
    """Per-output-channel symmetric int8 weights (rembed "Architecture",
    "int8 quantization": dense weights quantised at load to per-output-channel
    symmetric int8, one per-channel multiply in the epilogue). The pages print
    no rounding rule; the reading taken, per row j of W [n x k], in fp32:
    amax = max |w|, scale s = amax / 127, code c = round-half-even(w * (127 /
    amax)); a row with amax = 0 has codes 0 and scale 0. Returns (codes int8
    [n x k], scales fp32 [n])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    amax = np.abs(W).max(axis=1).astype(np.float32)
    inv = np.zeros_like(amax)
    nz = amax > 0
    inv[nz] = np.float32(127.0) / amax[nz]
    codes = np.rint(W * inv[:, None]).astype(np.int8)
    scales = (amax / np.float32(127.0)).astype(np.float32)
    return codes, scales


def matmul_w8(codes: np.ndarray, scales: np.ndarray, X: np.ndarray):
    """Y[t][j] = s_j * sum_c X[t][c] * code[j][c], fp64, with B = sum |terms|."""
    Xd = np.asarray(X, dtype=np.float64)
    Cd = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scales, dtype=np.float64)
    return (Xd @ Cd.T) * s[None, :], (np.abs(Xd) @ np.abs(Cd).T) * np.abs(s)[None, :]
