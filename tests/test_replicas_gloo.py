"""The multi-rank (replica) bookkeeping on CPU: two gloo ranks agree on the
maximum elapsed time, derive distinct replica seeds and the whole-job rate."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from kv_cache_decode_attention_gb300 import replicas


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        info = replicas.rank_info()
        replicas.barrier()
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        mx = replicas.max_over_ranks(local_ms)
        replicas.barrier()
        out[rank] = (info.rank, info.world, info.is_root, mx, replicas.sequence_seed(2, rank),
                     replicas.whole_job_rate(100.0, mx / 1e3, info.world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_rate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    r0, r1 = res[0], res[1]
    assert (r0[0], r0[1], r0[2]) == (0, 2, True) and (r1[0], r1[2]) == (1, False)
    assert r0[3] == r1[3] == 15.0  # both ranks see the slowest rank's time
    assert r0[4] != r1[4]  # distinct replica seeds
    assert r0[5] == pytest.approx(100.0 * 2 / 0.015)


def test_single_rank_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    info = replicas.rank_info()
    assert (info.rank, info.world, info.local_rank, info.is_root) == (0, 1, 0, True)
    assert replicas.max_over_ranks(3.5) == 3.5
    with pytest.raises(ValueError):
        replicas.rank_info({"WORLD_SIZE": "2", "RANK": "2"})
