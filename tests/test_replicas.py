"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The layer's tokens are independent, so a job on N GPUs is N replicas with no collective on the
data path: each rank draws the same seeded workload, the ranks meet only at barriers, the
slowest rank's step time sets the job time and the job throughput counts every rank's tokens.
These tests run that logic as two gloo processes; no GPU is touched.
"""
import hashlib
import os
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_moe_layer_sigmoid_gb300 import configs, inputs


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _digest(tensors):
    h = hashlib.sha256()
    for name in sorted(tensors):
        t = tensors[name]
        if isinstance(t, torch.Tensor):
            h.update(name.encode())
            h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    assert bench.rank_env() == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # step times differ per rank: the job takes the slowest one
        ms = 2.0 + 1.5 * rank
        job_ms = bench.max_over_ranks(ms, dist, "cpu")
        assert job_ms == 2.0 + 1.5 * (world - 1)
        tokens = 4096
        value = bench.job_tokens_per_s(world, tokens, job_ms)
        assert value == pytest.approx(world * tokens / (job_ms * 1e-3), rel=1e-12)

        # every replica draws the same seeded workload (weak scaling: fixed work per rank)
        cfg = configs.CONFIGS["tiny_f32"]
        digests = [None] * world
        dist.all_gather_object(digests, _digest(inputs.make_inputs(cfg, "cpu")))
        assert len(set(digests)) == 1

        # the reference arm runs on rank 0 alone; the other ranks return at once
        if rank != 0:
            args = types.SimpleNamespace(warmup=3, steps=1, gpus=world, workload=cfg.name)
            assert bench.run_reference(args, cfg, rank, world) is None
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.ok"), "w") as f:
            f.write(f"{job_ms} {value}\n")
    finally:
        dist.destroy_process_group()


def test_replica_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    lines = [(tmp_path / f"rank{r}.ok").read_text().split() for r in range(world)]
    assert lines[0] == lines[1]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.job_tokens_per_s(1, 4096, 4.0) == pytest.approx(1.024e6)
