"""Host logic of the multi-GPU bench on CPU: two `gloo` ranks (world size 2).

bench.py runs one replica of the workload per GPU (frames are independent
and the path has no exchange step).  What the ranks share is host logic:
a barrier, the job's step time as the MAX over ranks, the whole-job
throughput from it, rank 0 alone printing, and the reference arm running on
rank 0 only.  These run here as two CPU processes on the gloo backend."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.5, 0.8][rank]                      # rank 1 is the slow replica
        dist.barrier()
        job_ms = bench.max_over_ranks(local, torch.device("cpu"))
        value = bench.job_tflops(2.0e9, world, job_ms)

        class Args:
            workload, steps, warmup = "layer_list_fp32_n1", 1, 0
        ref = bench.run_reference(Args, rank, world) if rank == 1 else None
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"job_ms": job_ms, "value": value, "ref_is_none": ref is None}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["job_ms"] == r1["job_ms"] == 0.8          # the slowest replica sets the job time
    assert r0["value"] == pytest.approx(2 * 2.0e9 / 0.8e-3 / 1e12)   # both replicas' work in that time
    assert r1["ref_is_none"]                              # the reference arm runs on rank 0 only
