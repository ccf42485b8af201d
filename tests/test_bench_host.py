"""Host-side logic of bench.py: the max-over-ranks timing and whole-job rate
of a torchrun launch (two gloo ranks on the CPU) and the bounded sample of
the reference arm."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank "took" a different time; every rank must see the slowest
    slowest = bench.reduce_max(1.0 + rank)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, slowest))


def test_reduce_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.0, 1: 2.0}


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.25) == 3.25


def test_whole_job_rate_counts_every_rank():
    import bench
    # 2 ranks x 100 steps x 0.014 GB in 0.5 s (the slowest rank)
    assert bench.whole_job_rate(2, 100, 0.014, 0.5) == pytest.approx(5.6)


@pytest.mark.parametrize("steps,warmup,t", [(20, 3, 0.004), (300000, 1000, 0.004), (10, 3, 10.0)])
def test_reference_sample_is_bounded(steps, warmup, t):
    import bench
    rows = bench.reference_sample_rows(9728, steps, warmup, t)
    assert 64 <= rows <= 9728 and (rows % 64 == 0 or rows == 9728)
    est = (steps + warmup) * t * rows / 2048
    assert est <= 130 or rows == 64


def test_kernel_hash_ignores_comments_and_blank_space_only():
    import bench
    code = "__global__ void k(float *y) {\n    y[0] = 1.0f;   // one\n}\n"
    commented = "/* a kernel */\n__global__ void k(float *y)\n{\n  y[0] = 1.0f; // the value one\n}\n"
    changed = "__global__ void k(float *y) {\n    y[0] = 2.0f;\n}\n"
    h = bench.source_code_hash([("a.cu", code)])
    assert bench.source_code_hash([("a.cu", commented)]) == h
    assert bench.source_code_hash([("a.cu", changed)]) != h
    assert bench.source_code_hash([("b.cu", code)]) != h
    # host-only sources (the GGUF reader, the expert loop over q4_0_matmul)
    # hold no kernels or plans: they are left out of the hash
    assert {"q4mm_gguf.cu", "q4mm_experts.cu"} <= bench.HOST_ONLY_SOURCES
