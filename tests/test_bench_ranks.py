"""The multi-rank logic of bench.py on CPU: two gloo ranks agree on the
slowest rank's time, and the whole-job value counts every rank's bytes."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    job_ms = bench.max_over_ranks(local_ms, world)
    dist.barrier()
    q.put((rank, job_ms, bench.whole_job_gbs(world, 10 ** 9, job_ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # 2 ranks x 1 GB per step in 5 ms = 400 GB/s
    assert res[0][2] == pytest.approx(400.0)


def test_single_rank_identity():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_gbs(1, 6 * 10 ** 9, 1000.0) == pytest.approx(6.0)


def test_algorithmic_bytes():
    # per token: bf16 K,V read (2*8*128*2) + FP8 K,V written (2*8*128) + int64 slot
    assert bench.write_bytes(1) == 6152
    # one 32768-token layer: 2 * 8 * 128 bytes of FP8 KV per token dominates
    assert bench.decode_bytes(32768) == 32768 * 2048 + 32 * 128 * 4 + 2048 * 4 + 4 + 64
