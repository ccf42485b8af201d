"""Row sharding over G GPUs with no exchange (each GPU packs whole 128-row
groups of W and writes its columns of Y): the shard map on the host, the
reassembled Y of two gloo ranks against the oracle's whole Y on the CPU,
and (on a GPU) the shards' kernels writing their columns of one Y in place.
No multi-GPU run happens here: the multi-GPU path is unmeasured on
hardware."""

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from q4_quantized_linear_gb300 import synth  # noqa: E402
from q4_quantized_linear_gb300.shard import row_shards  # noqa: E402


@pytest.mark.parametrize("n", [0, 1, 127, 128, 129, 1000, 9728, 14336, 151936])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_row_shards_cover_the_rows_in_whole_groups(n, world):
    s = row_shards(n, world)
    assert len(s) == world
    pos = 0
    for row0, rows in s:
        assert row0 == pos and rows >= 0
        if row0 + rows < n:
            assert rows % 128 == 0                  # only the last shard ends mid-group
        pos += rows
    assert pos == n
    groups = [-(-rows // 128) for _, rows in s]
    assert max(groups) - min(groups) <= 1


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    n, k, m = 1000, 320, 3
    blocks = synth.q4_0_blocks(n, k, seed=11)
    X = synth.activations(m, k, seed=12)
    row0, rows = row_shards(n, world)[rank]
    Ys, _ = oracle.matmul(blocks[row0:row0 + rows], X, rows, k)      # this rank's columns
    pad = max(r for _, r in row_shards(n, world))   # the widest shard
    buf = torch.zeros((m, pad), dtype=torch.float64)
    buf[:, :rows] = torch.from_numpy(Ys)
    got = [torch.zeros_like(buf) for _ in range(world)]
    dist.all_gather(got, buf)
    Y = np.concatenate([g.numpy()[:, :r] for g, (_, r) in zip(got, row_shards(n, world))], axis=1)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, Y))


def test_two_gloo_ranks_reassemble_the_oracles_y():
    import torch.multiprocessing as mp
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    n, k, m = 1000, 320, 3
    Yr, _ = oracle.matmul(synth.q4_0_blocks(n, k, seed=11), synth.activations(m, k, seed=12), n, k)
    for r in (0, 1):
        assert np.array_equal(got[r], Yr)


@pytest.mark.gpu
@pytest.mark.parametrize("m,world", [(1, 2), (4, 3), (16, 2), (40, 2)])
def test_shards_write_their_columns_of_one_y_in_place(q4lib, oracle_mod, m, world):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q4_testlib import assert_parity, pack_dev, to_dev
    from q4_quantized_linear_gb300.shard import matmul_row_shard
    n, k = 1000, 640
    blocks = synth.q4_0_blocks(n, k, seed=21)
    X = synth.activations(m, k, seed=22)
    Xd = to_dev(X)
    Y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    for row0, rows in row_shards(n, world):
        W = pack_dev(q4lib, np.ascontiguousarray(blocks[row0:row0 + rows]), rows, k)
        matmul_row_shard(q4lib, W, Xd, Y, m, k, n, row0, rows)
    torch.cuda.synchronize()
    assert q4lib.q4_last_device_status(clear=True) == 0
    Yr, B = oracle_mod.matmul(blocks, X, n, k)
    assert_parity(Y.cpu().numpy(), Yr, B, m, f"{world} row shards, m={m}")
