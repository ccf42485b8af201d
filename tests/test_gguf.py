"""The GGUF reader in front of q4_0_pack: descriptors, metadata and tensor
bytes read back from files the test writes, every refusal of a malformed
file, and (on a GPU) a Q4_0 tensor loaded, packed and multiplied."""

import struct

import numpy as np
import pytest

from q4_quantized_linear_gb300 import synth
from gguf_writer import gguf_bytes, write_gguf

Q4_0, F32, Q4_K = 2, 0, 12


def _model(alignment=32, n=3, k=64):
    blocks = synth.q4_0_blocks(n, k, seed=5)
    emb = np.arange(16, dtype=np.float32)
    kvs = [("general.architecture", "str", "llama"),
           ("llama.block_count", "u32", 2),
           ("llama.context_length", "u64", 4096),
           ("llama.rope_shift", "i64", -3),
           ("general.quantized", "bool", 1),
           ("llama.rope.freq_base", "f32", 10000.0),
           ("tokenizer.ggml.tokens", "arr", ("str", ["<s>", "a", "bc"])),
           ("tokenizer.ggml.token_type", "arr", ("i32", [1, 2, 3]))]
    if alignment != 32:
        kvs.append(("general.alignment", "u32", alignment))
    tensors = [("token_embd.weight", F32, [8, 2], emb.tobytes()),
               ("blk.0.ffn_up.weight", Q4_0, [k, n], blocks.tobytes()),
               ("blk.0.attn_q.weight", Q4_K, [256, 1], bytes(range(144)))]
    return kvs, tensors, blocks


@pytest.mark.parametrize("alignment", [32, 64])
def test_descriptors_metadata_and_bytes_round_trip(q4lib, tmp_path, alignment):
    kvs, tensors, blocks = _model(alignment)
    path = tmp_path / "m.gguf"
    write_gguf(path, kvs, tensors, alignment)
    h = q4lib.q4_gguf_open(str(path))
    try:
        assert q4lib.q4_gguf_tensor_count(h) == 3
        assert q4lib.q4_gguf_get_string(h, "general.architecture") == "llama"
        assert q4lib.q4_gguf_get_int(h, "llama.block_count") == 2
        assert q4lib.q4_gguf_get_int(h, "llama.context_length") == 4096
        assert q4lib.q4_gguf_get_int(h, "llama.rope_shift") == -3
        assert q4lib.q4_gguf_get_int(h, "general.quantized") == 1
        raw = path.read_bytes()
        for i, (name, typ, dims, data) in enumerate(tensors):
            assert q4lib.q4_gguf_find_tensor(h, name) == i
            info = q4lib.q4_gguf_tensor_info(h, i)
            assert (info["name"], info["type"], info["dims"]) == (name, typ, dims)
            assert info["file_offset"] % alignment == 0
            assert raw[info["file_offset"]:info["file_offset"] + len(data)] == data
            if typ == Q4_K:
                assert info["bytes"] == 0          # size not known to the reader
            else:
                assert info["bytes"] == len(data)
                out = np.zeros(len(data), dtype=np.uint8)
                q4lib.q4_gguf_read_tensor(h, i, out, out.nbytes)
                assert out.tobytes() == data
        assert q4lib.q4_gguf_find_tensor(h, "missing") == -1
        small = np.zeros(8, dtype=np.uint8)
        assert q4lib.q4_gguf_read_tensor(h, 1, small, small.nbytes, check=False) == q4lib.Q4_ERR_INVALID_ARG
        for bad_key, getter in [("missing", q4lib.q4_gguf_get_int), ("general.architecture", q4lib.q4_gguf_get_int),
                                ("llama.block_count", q4lib.q4_gguf_get_string),
                                ("llama.rope.freq_base", q4lib.q4_gguf_get_int)]:
            with pytest.raises(q4lib.Q4Error):
                getter(h, bad_key)
    finally:
        q4lib.q4_gguf_close(h)
    got, n, k = q4lib.gguf_q4_0_blocks(str(path), "blk.0.ffn_up.weight")
    assert (n, k) == (3, 64) and np.array_equal(got, blocks)


def _refused(q4lib, tmp_path, data, code):
    path = tmp_path / "bad.gguf"
    path.write_bytes(data)
    with pytest.raises(q4lib.Q4Error) as e:
        q4lib.q4_gguf_open(str(path))
    assert e.value.status == code


def test_malformed_files_are_refused(q4lib, tmp_path):
    kvs, tensors, _ = _model()
    good = gguf_bytes(kvs, tensors)
    F = q4lib.Q4_ERR_FORMAT
    _refused(q4lib, tmp_path, b"GGUX" + good[4:], F)                       # magic
    _refused(q4lib, tmp_path, gguf_bytes(kvs, tensors, version=1), F)      # version 1 (u32 counts)
    _refused(q4lib, tmp_path, gguf_bytes(kvs, tensors, version=4), F)      # unknown version
    _refused(q4lib, tmp_path, good[:40], F)                                # cut inside the metadata
    _refused(q4lib, tmp_path, good[:-200], F)                              # blob cut short
    _refused(q4lib, tmp_path, b"GGUF", F)                                  # header cut short
    # a string length reaching past the end
    huge = b"GGUF" + struct.pack("<IQQ", 3, 0, 1) + struct.pack("<Q", 1 << 40) + b"key"
    _refused(q4lib, tmp_path, huge, F)
    # alignment that is not a power of two
    _refused(q4lib, tmp_path, gguf_bytes(kvs + [("general.alignment", "u32", 48)], tensors), F)
    # a descriptor offset that is not a multiple of the alignment
    one = [("t", Q4_0, [32, 1], bytes(18))]
    blob = bytearray(gguf_bytes([], one))
    at = blob.index(b"t") + 1 + 4 + 8 + 4       # name, dim count, one dim, type: then the offset
    blob[at:at + 8] = struct.pack("<Q", 8)
    _refused(q4lib, tmp_path, bytes(blob), F)
    # a file that is not there
    with pytest.raises(q4lib.Q4Error) as e:
        q4lib.q4_gguf_open(str(tmp_path / "none.gguf"))
    assert e.value.status == q4lib.Q4_ERR_IO


@pytest.mark.gpu
def test_q4_0_tensor_loads_packs_and_multiplies(q4lib, oracle_mod, tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q4_testlib import assert_parity, run_matmul
    n, k, m = 200, 1056, 3
    blocks = synth.q4_0_blocks(n, k, seed=9)
    path = tmp_path / "w.gguf"
    write_gguf(path, [("general.architecture", "str", "llama")],
               [("blk.0.ffn_down.weight", Q4_0, [k, n], blocks.tobytes())])
    W, n2, k2 = q4lib.load_q4_0_packed(str(path), "blk.0.ffn_down.weight")
    assert (n2, k2) == (n, k)
    X = synth.activations(m, k, seed=10)
    Y = run_matmul(q4lib, W, X, n)
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y, Yr, B, m, "gguf-loaded weights")


def _golden_bytes():
    import os
    import re
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "golden", "gguf_min_q4_0.hex")) as f:
        txt = f.read()
    return bytes(int(x, 16) for line in txt.splitlines() for x in re.sub(r"#.*", "", line).split())


def test_hand_typed_gguf_golden_is_read_as_the_layout_says(q4lib, oracle_mod, tmp_path):
    """A file typed byte by byte from the container's layout (not written by
    the test writer): the reader finds the alignment, the one Q4_0 tensor's
    name, type, dims (innermost first) and the blob offset (128: 98 bytes of
    header rounded up to 32), and its 36 bytes; the oracle reads them as the
    weights the file's comments state."""
    data = _golden_bytes()
    assert len(data) == 164
    path = tmp_path / "golden.gguf"
    path.write_bytes(data)
    h = q4lib.q4_gguf_open(str(path))
    try:
        assert q4lib.q4_gguf_tensor_count(h) == 1
        assert q4lib.q4_gguf_get_int(h, "general.alignment") == 32
        assert q4lib.q4_gguf_find_tensor(h, "w") == 0
        info = q4lib.q4_gguf_tensor_info(h, 0)
        assert (info["name"], info["type"], info["dims"]) == ("w", Q4_0, [32, 2])
        assert (info["file_offset"], info["bytes"]) == (128, 36)
        out = np.zeros(36, dtype=np.uint8)
        q4lib.q4_gguf_read_tensor(h, 0, out, out.nbytes)
    finally:
        q4lib.q4_gguf_close(h)
    assert out.tobytes() == data[128:]
    # W^T through the oracle's product with the identity
    Y, _ = oracle_mod.matmul(out.reshape(2, 1, 18), np.eye(32, dtype=np.float32), 2, 32)
    low = [-8, -6, -4, -2, 0, 2, 4, 6] * 2        # elements 0..15: the bytes' low nibbles - 8
    high = [-7, -5, -3, -1, 1, 3, 5, 7] * 2       # elements 16..31: the high nibbles - 8
    assert np.array_equal(Y[:, 0], np.array(low + high, dtype=np.float64))
    assert np.array_equal(Y[:, 1], np.zeros(32))
