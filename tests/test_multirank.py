"""The N-GPU bench path is N replicas (weak scaling, no collective on the data path): each
rank builds its own batch (seed offset per rank) and the job's time is the slowest rank's.
Checked here with two gloo processes on the CPU."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w = bench.workload("decode_b256", layers=1, seed_offset=100 * rank)
        local_ms = 1.5 + rank  # rank 1 is slower
        step_ms = bench.max_over_ranks(local_ms, "cpu")
        lens = torch.from_numpy(w.context_lens.astype(np.int64))
        gathered = [torch.zeros_like(lens) for _ in range(world)]
        dist.all_gather(gathered, lens)
        results[rank] = (step_ms, w.seed, w.num_seqs, w.decode_kv_bytes(),
                         bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_their_own_batches():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    (t0, seed0, s0, kv0, same0), (t1, seed1, s1, kv1, _) = res[0], res[1]
    assert t0 == t1 == 2.5  # max over ranks, seen by every rank
    assert seed0 != seed1 and s0 == s1 == 256  # own batch, same shape
    assert not same0  # different context draws
    import bench
    assert bench.whole_job_gbs(kv0, world, t0) == kv0 * 2 / 2.5e-3 / 1e9
