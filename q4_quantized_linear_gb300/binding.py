"""Thin Python binding of libq4mm's C ABI (include/q4mm.h).

Every function here has the name of the C entry point it calls and only
marshals arguments (torch CUDA tensors or raw device addresses, the current
torch stream by default); all arithmetic runs in libq4mm's CUDA kernels.
There is no CPU path: if the library has not been built, importing this
module raises.

Build the library with ``python -m q4_quantized_linear_gb300.build`` (or
``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB as _DEFAULT_LIB

# Q4MM_LIBRARY selects another build of the same ABI (e.g. a profiling build).
LIB = os.environ.get("Q4MM_LIBRARY", _DEFAULT_LIB)
if not os.path.exists(LIB):
    raise ImportError(
        f"libq4mm is not built ({LIB} missing); run `python -m q4_quantized_linear_gb300.build`")

_lib = ctypes.CDLL(LIB)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_INT = ctypes.c_int

_SIGS = {
    "q4_0_packed_size": (_SZ, [_I64, _I64]),
    "q4_0_pack": (_INT, [_P, _P, _I64, _I64, _P]),
    "q4_0_unpack": (_INT, [_P, _P, _I64, _I64, _P]),
    "q4_0_matmul_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "q4_0_matmul": (_INT, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "q4_0_matmul_ws": (_INT, [_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "q4_0_matmul_w4a8": (_INT, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "q4_w8_packed_size": (_SZ, [_I64, _I64]),
    "q4_w8_quantize": (_INT, [_P, _P, _I64, _I64, _P]),
    "q4_w8_unpack": (_INT, [_P, _P, _P, _I64, _I64, _P]),
    "q4_w8_matmul": (_INT, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "q4_0_matmul_experts": (_INT, [ctypes.POINTER(_P), _I64, ctypes.POINTER(_I64), _P, _P, _I64, _I64, _P]),
    "q4_0_matmul_static_scratch": (_INT, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "q4_0_matmul_batched_slots": (_INT, [_P, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _P]),
    "q4_0_matmul_batched_slots_ws": (_INT, [_P, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "q4_status_string": (ctypes.c_char_p, [_INT]),
    "q4_last_device_status": (_INT, [_INT]),
    "q4_build_flags": (_INT, []),
    "q4_set_wait_limit_ns": (_INT, [ctypes.c_uint64]),
    "q4_set_weight_prefetch": (_INT, [_INT]),
    "q4_set_decode_kernel": (_INT, [_INT]),
    "q4_selftest_wait_timeout": (_INT, [ctypes.c_uint64, _P]),
    "q4_debug_set_trace": (_INT, [_P, _SZ, ctypes.c_uint32]),
    "q4_gguf_open": (_INT, [ctypes.c_char_p, ctypes.POINTER(_P)]),
    "q4_gguf_close": (None, [_P]),
    "q4_gguf_tensor_count": (_I64, [_P]),
    "q4_gguf_find_tensor": (_I64, [_P, ctypes.c_char_p]),
    "q4_gguf_tensor_info": (_INT, [_P, _I64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_INT),
                                   ctypes.POINTER(_INT), ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_uint64),
                                   ctypes.POINTER(ctypes.c_uint64)]),
    "q4_gguf_read_tensor": (_INT, [_P, _I64, _P, ctypes.c_uint64]),
    "q4_gguf_get_int": (_INT, [_P, ctypes.c_char_p, ctypes.POINTER(_I64)]),
    "q4_gguf_get_string": (_INT, [_P, ctypes.c_char_p, ctypes.POINTER(ctypes.c_char_p)]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

Q4_OK = 0
Q4_ERR_INVALID_ARG = 1
Q4_ERR_ALIGNMENT = 2
Q4_ERR_UNSUPPORTED_DEVICE = 3
Q4_ERR_CUDA = 4
Q4_ERR_DEVICE_TIMEOUT = 5
Q4_ERR_WORKSPACE = 6
Q4_ERR_NO_MEMORY = 7
Q4_ERR_IO = 8
Q4_ERR_FORMAT = 9
Q4_ERR_DEVICE_CHECK = 10
GGUF_TYPE_Q4_0 = 2


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {q4_status_string(status)} ({status})")


def library_path() -> str:
    return LIB


def exported_symbols() -> list[str]:
    return sorted(_SIGS)


def _addr(x) -> int | None:
    """Device address of a torch tensor, or an int address as is (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != Q4_OK:
        raise Q4Error(rc, where)
    return rc


# ------------------------------------------------------------- C ABI calls --

def q4_status_string(status: int) -> str:
    return _lib.q4_status_string(int(status)).decode()


def q4_0_packed_size(n: int, k: int) -> int:
    return int(_lib.q4_0_packed_size(n, k))


def q4_0_matmul_workspace_size(m: int, k: int, n: int) -> int:
    return int(_lib.q4_0_matmul_workspace_size(m, k, n))


def q4_0_pack(W_packed, blocks, n: int, k: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_pack(_addr(W_packed), _addr(blocks), n, k, _stream(stream))
    return _check(rc, "q4_0_pack") if check else rc


def q4_0_unpack(blocks, W_packed, n: int, k: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_unpack(_addr(blocks), _addr(W_packed), n, k, _stream(stream))
    return _check(rc, "q4_0_unpack") if check else rc


def q4_0_matmul(W_packed, X, Y, m: int, k: int, n: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_matmul(_addr(W_packed), _addr(X), _addr(Y), m, k, n, _stream(stream))
    return _check(rc, "q4_0_matmul") if check else rc


def q4_0_matmul_experts(W_list, offsets, X, Y, k: int, n: int, stream=None, check: bool = True) -> int:
    """W_list: one packed weight buffer per expert (None for an expert with no
    rows); offsets: n_experts + 1 row offsets into X and Y."""
    E = len(W_list)
    ws = (_P * E)(*[_addr(w) for w in W_list])
    offs = (_I64 * len(offsets))(*[int(o) for o in offsets])
    if len(offsets) != E + 1:
        raise ValueError("one offset per expert, plus the end")
    rc = _lib.q4_0_matmul_experts(ws, E, offs, _addr(X), _addr(Y), k, n, _stream(stream))
    return _check(rc, "q4_0_matmul_experts") if check else rc


def q4_0_matmul_w4a8(W_packed, X, Y, m: int, k: int, n: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_matmul_w4a8(_addr(W_packed), _addr(X), _addr(Y), m, k, n, _stream(stream))
    return _check(rc, "q4_0_matmul_w4a8") if check else rc


def q4_w8_packed_size(n: int, k: int) -> int:
    return int(_lib.q4_w8_packed_size(n, k))


def q4_w8_quantize(W8_packed, W, n: int, k: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_w8_quantize(_addr(W8_packed), _addr(W), n, k, _stream(stream))
    return _check(rc, "q4_w8_quantize") if check else rc


def q4_w8_unpack(codes, scales, W8_packed, n: int, k: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_w8_unpack(_addr(codes), _addr(scales), _addr(W8_packed), n, k, _stream(stream))
    return _check(rc, "q4_w8_unpack") if check else rc


def q4_w8_matmul(W8_packed, X, Y, m: int, k: int, n: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_w8_matmul(_addr(W8_packed), _addr(X), _addr(Y), m, k, n, _stream(stream))
    return _check(rc, "q4_w8_matmul") if check else rc


def q4_0_matmul_ws(W_packed, X, Y, m: int, k: int, n: int, workspace, workspace_bytes: int,
                   stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_matmul_ws(_addr(W_packed), _addr(X), _addr(Y), m, k, n, _addr(workspace),
                             workspace_bytes, _stream(stream))
    return _check(rc, "q4_0_matmul_ws") if check else rc


Q4_STATIC_SCRATCH_BYTES = 8 << 20


def q4_0_matmul_static_scratch(W_packed, X, Y, m: int, k: int, n: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_matmul_static_scratch(_addr(W_packed), _addr(X), _addr(Y), m, k, n, _stream(stream))
    return _check(rc, "q4_0_matmul_static_scratch") if check else rc


def q4_0_matmul_batched_slots(W_packed, X_slots, ldx: int, slot_ids, m: int, Y_slots, ldy: int,
                              k: int, n: int, stream=None, check: bool = True) -> int:
    rc = _lib.q4_0_matmul_batched_slots(_addr(W_packed), _addr(X_slots), ldx, _addr(slot_ids), m,
                                        _addr(Y_slots), ldy, k, n, _stream(stream))
    return _check(rc, "q4_0_matmul_batched_slots") if check else rc


def q4_0_matmul_batched_slots_ws(W_packed, X_slots, ldx: int, slot_ids, m: int, Y_slots, ldy: int,
                                 k: int, n: int, workspace, workspace_bytes: int, stream=None,
                                 check: bool = True) -> int:
    rc = _lib.q4_0_matmul_batched_slots_ws(_addr(W_packed), _addr(X_slots), ldx, _addr(slot_ids), m,
                                           _addr(Y_slots), ldy, k, n, _addr(workspace),
                                           workspace_bytes, _stream(stream))
    return _check(rc, "q4_0_matmul_batched_slots_ws") if check else rc


def q4_last_device_status(clear: bool = True) -> int:
    return int(_lib.q4_last_device_status(1 if clear else 0))


def q4_build_flags() -> int:
    """Bit 0: the checked build (-DQ4MM_CHECKED); bit 1: the trace build."""
    return int(_lib.q4_build_flags())


def q4_set_wait_limit_ns(ns: int) -> int:
    return _check(_lib.q4_set_wait_limit_ns(int(ns)), "q4_set_wait_limit_ns")


def q4_set_weight_prefetch(enable: bool) -> int:
    return _check(_lib.q4_set_weight_prefetch(1 if enable else 0), "q4_set_weight_prefetch")


Q4_DECODE_AUTO = 0
Q4_DECODE_WARP_MMA = 1
Q4_DECODE_CUDA_CORE = 2
Q4_DECODE_TCGEN05 = 3
Q4_DECODE_RECORD_MMA = 4
Q4_DECODE_MATVEC = 5


def q4_set_decode_kernel(kind: int) -> int:
    return _check(_lib.q4_set_decode_kernel(int(kind)), "q4_set_decode_kernel")


def q4_debug_set_trace(buffer, nbytes: int, cta: int = 0, check: bool = True) -> int:
    rc = _lib.q4_debug_set_trace(_addr(buffer), nbytes, cta)
    return _check(rc, "q4_debug_set_trace") if check else rc


def q4_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return _check(_lib.q4_selftest_wait_timeout(int(limit_ns), _stream(stream)), "q4_selftest_wait_timeout")


# ------------------------------------------------------ tensor conveniences --

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace_for(m: int, k: int, n: int, device=None, stream=None):
    """A zeroed torch uint8 workspace large enough for (m, k, n), cached per
    (device, stream) and grown on demand (torch's allocator, no cudaMalloc
    per call once warm). Returns (tensor or None, bytes)."""
    import torch
    need = q4_0_matmul_workspace_size(m, k, n)
    if need == 0:
        return None, 0
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = (dev.index, _stream(stream))
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < need:
            buf = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=dev)
            _ws_cache[key] = buf
    return buf, buf.numel()


def pack(blocks, n: int, k: int, stream=None):
    """GGUF Q4_0 blocks (torch uint8 CUDA tensor, n*(k/32)*18 bytes) -> packed tensor."""
    import torch
    out = torch.empty(q4_0_packed_size(n, k), dtype=torch.uint8, device=blocks.device)
    q4_0_pack(out, blocks, n, k, stream)
    return out


def matmul(W_packed, X, n: int, out=None, stream=None):
    """Y = X . W^T for fp32 CUDA X [m x k]; returns Y [m x n] fp32."""
    import torch
    m, k = X.shape
    Y = torch.empty((m, n), dtype=torch.float32, device=X.device) if out is None else out
    ws, wsb = workspace_for(m, k, n, X.device, stream)
    q4_0_matmul_ws(W_packed, X, Y, m, k, n, ws, wsb, stream)
    return Y


# ------------------------------------------------------------------ GGUF --

def q4_gguf_open(path: str) -> int:
    """Parse a GGUF file's header, metadata and descriptors; returns a handle."""
    h = _P()
    _check(_lib.q4_gguf_open(os.fsencode(path), ctypes.byref(h)), "q4_gguf_open")
    return h.value


def q4_gguf_close(handle: int) -> None:
    _lib.q4_gguf_close(handle)


def q4_gguf_tensor_count(handle: int) -> int:
    return _lib.q4_gguf_tensor_count(handle)


def q4_gguf_find_tensor(handle: int, name: str) -> int:
    return _lib.q4_gguf_find_tensor(handle, name.encode())


def q4_gguf_tensor_info(handle: int, index: int) -> dict:
    name = ctypes.c_char_p()
    typ, nd = _INT(), _INT()
    dims = (_I64 * 4)()
    off, nbytes = ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.q4_gguf_tensor_info(handle, index, ctypes.byref(name), ctypes.byref(typ), ctypes.byref(nd), dims,
                                    ctypes.byref(off), ctypes.byref(nbytes)), "q4_gguf_tensor_info")
    return dict(name=name.value.decode(), type=typ.value, dims=list(dims[:nd.value]),
                file_offset=off.value, bytes=nbytes.value)


def q4_gguf_read_tensor(handle: int, index: int, host_dst, dst_bytes: int, check: bool = True) -> int:
    rc = _lib.q4_gguf_read_tensor(handle, index, _addr_host(host_dst), dst_bytes)
    return _check(rc, "q4_gguf_read_tensor") if check else rc


def q4_gguf_get_int(handle: int, key: str) -> int:
    v = _I64()
    _check(_lib.q4_gguf_get_int(handle, key.encode(), ctypes.byref(v)), "q4_gguf_get_int")
    return v.value


def q4_gguf_get_string(handle: int, key: str) -> str:
    v = ctypes.c_char_p()
    _check(_lib.q4_gguf_get_string(handle, key.encode(), ctypes.byref(v)), "q4_gguf_get_string")
    return v.value.decode()


def _addr_host(a) -> int:
    """Host address of a contiguous numpy array."""
    return a.ctypes.data


def gguf_q4_0_blocks(path: str, name: str):
    """(blocks, n, k): a Q4_0 tensor's [n][k/32] 18-byte blocks, read from a
    GGUF file into a host numpy array (uint8, shape (n, k/32, 18))."""
    import numpy as np
    h = q4_gguf_open(path)
    try:
        i = q4_gguf_find_tensor(h, name)
        if i < 0:
            raise KeyError(f"{path}: no tensor {name!r}")
        info = q4_gguf_tensor_info(h, i)
        if info["type"] != GGUF_TYPE_Q4_0 or len(info["dims"]) != 2:
            raise ValueError(f"{name}: not a 2-D Q4_0 tensor (type {info['type']}, dims {info['dims']})")
        k, n = info["dims"]
        blocks = np.empty((n, k // 32, 18), dtype=np.uint8)
        q4_gguf_read_tensor(h, i, blocks, blocks.nbytes)
        return blocks, n, k
    finally:
        q4_gguf_close(h)


def load_q4_0_packed(path: str, name: str, stream=None):
    """(W_packed, n, k): a Q4_0 tensor of a GGUF file, copied to the current
    device and packed once by q4_0_pack (torch holds the device memory)."""
    import torch
    blocks, n, k = gguf_q4_0_blocks(path, name)
    dev_blocks = torch.from_numpy(blocks.reshape(-1)).cuda()
    W = torch.empty(q4_0_packed_size(n, k), dtype=torch.uint8, device="cuda")
    q4_0_pack(W, dev_blocks, n, k, stream)
    return W, n, k
