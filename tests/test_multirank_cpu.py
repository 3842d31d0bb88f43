"""The data-parallel host logic of bench.py on 2 CPU ranks (gloo).

The sublayer shards over the batch with no exchange step: every rank runs
whole, independent sequences. This checks, without a GPU, that (1) the
per-rank inputs are distinct seeded batches, (2) outputs computed per rank
(here by the fp64 oracle) equal those of one process doing all ranks' work,
and (3) the job timing is the max over ranks and the job throughput counts
every rank's units.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    import bench
    import oracle
    from transformer_head_scaled_fwd_gb300 import workloads as W
    wl = W.Workload("shard", 1, "bf16", 2, 6, 6, 32, 4, True, True, valid_range=(3, 6))
    inp = bench.rank_inputs(wl, rank)
    w = inp.weights
    out = oracle.mha_forward(inp.query, inp.key, inp.value, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"],
                             w["b_v"], w["w_o"], w["b_o"], wl.h, causal=True, valid_lens=inp.valid_lens)
    gathered = [torch.zeros(out.shape, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(out))
    total, e2e = bench.job_times(10.0 + rank, 20.0 + 3 * rank, world)
    if rank == 0:
        np.save(os.path.join(outdir, "gathered.npy"), torch.stack(gathered).numpy())
        np.save(os.path.join(outdir, "times.npy"), np.array([total, e2e]))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_rank_batch_sharding(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    gathered = np.load(tmp_path / "gathered.npy")
    total, e2e = np.load(tmp_path / "times.npy")
    assert total == 11.0 and e2e == 23.0                      # max over ranks
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from transformer_head_scaled_fwd_gb300 import workloads as W
    wl = W.Workload("shard", 1, "bf16", 2, 6, 6, 32, 4, True, True, valid_range=(3, 6))
    for r in range(world):                                     # one process doing every rank's work
        inp = bench.rank_inputs(wl, r)
        w = inp.weights
        ref = oracle.mha_forward(inp.query, inp.key, inp.value, w["w_q"], w["b_q"], w["w_k"], w["b_k"],
                                 w["w_v"], w["b_v"], w["w_o"], w["b_o"], wl.h, causal=True,
                                 valid_lens=inp.valid_lens)
        np.testing.assert_array_equal(gathered[r], ref)
    assert not np.array_equal(gathered[0], gathered[1])        # ranks hold distinct sequences
    assert bench.job_throughput(2, 1e12, 1000.0) == pytest.approx(2.0)
