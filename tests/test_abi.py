"""The C-ABI library loads and exports exactly what include/q4mm.h declares;
host-side argument checks refuse bad calls before any device work. No GPU
is needed (no compute call is made)."""

import re
import subprocess

import pytest

from conftest import ROOT


def _declared():
    with open(f"{ROOT}/include/q4mm.h") as f:
        text = f.read()
    return sorted(set(re.findall(r"Q4MM_API\s+[^;(]*?\b(q4_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ["q4_0_packed_size", "q4_0_pack", "q4_0_unpack", "q4_0_matmul",
                     "q4_0_matmul_batched_slots", "q4_status_string", "q4_last_device_status"]:
        assert required in names


def test_library_exports_every_declared_symbol(q4lib):
    out = subprocess.run(["nm", "-D", "--defined-only", q4lib.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if ln.strip()} - {""})
    q4_exported = [s for s in exported if s.startswith("q4_")]
    assert q4_exported == _declared()
    # the binding wraps every declared entry point under the same name
    assert q4lib.exported_symbols() == _declared()
    for name in _declared():
        assert callable(getattr(q4lib, name))


def test_status_strings(q4lib):
    for code in range(11):
        assert q4lib.q4_status_string(code) not in ("", "unknown status")
    assert q4lib.q4_status_string(99) == "unknown status"


def test_default_build_is_neither_checked_nor_traced(q4lib):
    assert q4lib.q4_build_flags() == 0


def test_int8_weight_packed_size_formula(q4lib):
    # records of 128 rows x 64 int8 codes (8192 bytes), then 4 bytes of scale
    # per padded row
    assert q4lib.q4_w8_packed_size(9728, 2560) == 76 * 40 * 8192 + 76 * 128 * 4
    assert q4lib.q4_w8_packed_size(130, 96) == 2 * 2 * 8192 + 2 * 128 * 4
    assert q4lib.q4_w8_packed_size(0, 64) == 0
    assert q4lib.q4_w8_packed_size(64, 48) == 0


@pytest.mark.parametrize("call,args,code", [
    ("q4_w8_quantize", (0, 0x1000, 64, 64), 1),                       # null packed
    ("q4_w8_quantize", (0x1000, 0, 64, 64), 1),                       # null W
    ("q4_w8_quantize", (0x1000, 0x1000, 64, 48), 1),                  # k % 32 != 0
    ("q4_w8_quantize", (0x1008, 0x1000, 64, 64), 2),                  # packed not 16-byte aligned
    ("q4_w8_quantize", (0x1000, 0x1004, 64, 64), 2),                  # W not 16-byte aligned
    ("q4_w8_unpack", (0, 0x1000, 0x1000, 64, 64), 1),                 # null codes
    ("q4_w8_unpack", (0x1000, 0x1000, 0x1008, 64, 64), 2),            # packed not 16-byte aligned
    ("q4_w8_unpack", (0x1001, 0x1000, 0x1000, 64, 64), 2),            # codes not 4-byte aligned
    ("q4_w8_matmul", (0, 0x1000, 0x1000, 1, 64, 64), 1),              # null packed
    ("q4_w8_matmul", (0x1000, 0x1000, 0x1000, -1, 64, 64), 1),        # m < 0
    ("q4_w8_matmul", (0x1000, 0x1000, 0x1000, 1, 64, 0), 1),          # n == 0
    ("q4_w8_matmul", (0x1000, 0x1004, 0x1000, 1, 64, 64), 2),         # X not 16-byte aligned
    ("q4_w8_matmul", (0x1000, 0x1000, 0x1002, 1, 64, 64), 2),         # Y not 4-byte aligned
])
def test_int8_weight_calls_refuse_bad_arguments_before_device_work(q4lib, call, args, code):
    assert getattr(q4lib, call)(*args, stream=0, check=False) == code


def test_int8_weight_matmul_with_no_rows_is_a_no_op(q4lib):
    assert q4lib.q4_w8_matmul(0x1000, 0x1000, 0x1000, 0, 64, 64, stream=0, check=False) == 0


def test_packed_size_formula(q4lib):
    assert q4lib.q4_0_packed_size(9728, 2560) == 152 * 40 * 2304 == 14008320
    assert q4lib.q4_0_packed_size(70, 96) == 2 * 2 * 2304
    assert q4lib.q4_0_packed_size(0, 64) == 0
    assert q4lib.q4_0_packed_size(64, 48) == 0


@pytest.mark.parametrize("args,code", [
    ((0, 0x1000, 0x1000, 1, 64, 64), 1),        # null W
    ((0x1000, 0, 0x1000, 1, 64, 64), 1),        # null X
    ((0x1000, 0x1000, 0x1000, 1, 48, 64), 1),   # k % 32 != 0
    ((0x1000, 0x1000, 0x1000, 1, 64, 0), 1),    # n == 0
    ((0x1000, 0x1000, 0x1000, -1, 64, 64), 1),  # m < 0
    ((0x1008, 0x1000, 0x1000, 1, 64, 64), 2),   # W not 16-byte aligned
    ((0x1000, 0x1004, 0x1000, 1, 64, 64), 2),   # X not 16-byte aligned
    ((0x1000, 0x1000, 0x1002, 1, 64, 64), 2),   # Y not 4-byte aligned
])
def test_matmul_rejects_bad_arguments_on_the_host(q4lib, args, code):
    assert q4lib.q4_0_matmul(*args, stream=0, check=False) == code


@pytest.mark.parametrize("args,code", [
    ((0, 0x1000, 0x1000, 1, 64, 64), 1),        # null W
    ((0x1000, 0x1000, 0x1000, 17, 64, 64), 1),  # m > 16
    ((0x1000, 0x1000, 0x1000, -1, 64, 64), 1),  # m < 0
    ((0x1000, 0x1000, 0x1000, 1, 48, 64), 1),   # k % 32 != 0
    ((0x1000, 0x1004, 0x1000, 1, 64, 64), 2),   # X not 16-byte aligned
])
def test_w4a8_rejects_bad_arguments_on_the_host(q4lib, args, code):
    assert q4lib.q4_0_matmul_w4a8(*args, stream=0, check=False) == code


@pytest.mark.parametrize("W,offsets,code", [
    ([0x1000, 0x1000], [1, 2, 3], 1),           # offsets do not start at 0
    ([0x1000, 0x1000], [0, 3, 2], 1),           # offsets fall
    ([0x1000, 0], [0, 2, 3], 1),                # an expert with rows has no weights
    ([0x1000, 0x1008], [0, 2, 3], 2),           # weights not 16-byte aligned
])
def test_experts_reject_bad_arguments_on_the_host(q4lib, W, offsets, code):
    assert q4lib.q4_0_matmul_experts(W, offsets, 0x1000, 0x1000, 64, 64, stream=0, check=False) == code


def test_batched_slots_rejects_bad_leading_dimensions(q4lib):
    # ldx < k, ldx % 4 != 0, ldy < n, null slot ids
    assert q4lib.q4_0_matmul_batched_slots(0x1000, 0x1000, 32, 0x1000, 2, 0x1000, 64, 64, 64,
                                           stream=0, check=False) == 1
    assert q4lib.q4_0_matmul_batched_slots(0x1000, 0x1000, 66, 0x1000, 2, 0x1000, 64, 64, 64,
                                           stream=0, check=False) == 2
    assert q4lib.q4_0_matmul_batched_slots(0x1000, 0x1000, 64, 0x1000, 2, 0x1000, 32, 64, 64,
                                           stream=0, check=False) == 1
    assert q4lib.q4_0_matmul_batched_slots(0x1000, 0x1000, 64, 0, 2, 0x1000, 64, 64, 64,
                                           stream=0, check=False) == 1


def test_pack_rejects_bad_arguments_on_the_host(q4lib):
    assert q4lib.q4_0_pack(0, 0x1000, 64, 64, stream=0, check=False) == 1
    assert q4lib.q4_0_pack(0x1000, 0x1000, 64, 40, stream=0, check=False) == 1
    assert q4lib.q4_0_pack(0x1004, 0x1000, 64, 64, stream=0, check=False) == 2
    assert q4lib.q4_0_unpack(0x1001, 0x1000, 64, 64, stream=0, check=False) == 2


def test_decode_kernel_setting_is_checked(q4lib):
    # 0..5 accepted (host-only setting), anything else refused; default restored
    for bad in (-1, 6, 16):
        assert q4lib._lib.q4_set_decode_kernel(bad) == 1
    for good in (1, 2, 3, 4, 5, 0):
        assert q4lib._lib.q4_set_decode_kernel(good) == 0
