"""The multi-GPU benchmark path on CPU: two gloo ranks (world_size 2).

Several GPUs run independent replicas of the step: each rank drafts (verifies,
or builds the COD lists of) its own seeded batch, nothing crosses ranks on the data path, the job's time is the
slowest rank's and its throughput the units of all ranks over that time.  The
host logic that does this (bench.py: rank_workload, max_over_ranks,
job_throughput) runs here on CPU tensors over gloo.
"""

import hashlib
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from speculative_drafting_gb300 import workloads as W

        # each rank's batch comes from its own seed
        wl = bench.rank_workload(W.get("tiny_fp32"), rank)
        b = W.make_batch(wl)
        digest = hashlib.sha256(b["prev_tok"].tobytes() + b["H_tgt"].tobytes()).hexdigest()
        vwl = bench.rank_workload(W.get_verify("verify_small"), rank)
        vb = W.make_verify_batch(vwl)
        vdigest = hashlib.sha256(vb["logits"].tobytes()).hexdigest()
        cb = W.make_cod_batch(bench.rank_workload(W.get_cod("cod_tiny"), rank))
        cdigest = hashlib.sha256(cb["u_anchor"].tobytes() + cb["loss_mask"].tobytes()).hexdigest()
        digests = [None] * world
        dist.all_gather_object(digests, (digest, vdigest, cdigest))
        # the job's time is the slowest rank's, on every rank
        local_ms = 1.5 + rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_throughput(wl.batch * wl.dims.K, world, job_ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{job_ms} {value} {digests[0][0]} {digests[1][0]} {digests[0][1]} {digests[1][1]} "
                    f"{digests[0][2]} {digests[1][2]}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for job_ms, value, d0, d1, v0, v1, c0, c1 in rows:
        assert float(job_ms) == 2.5                      # the slower rank's time
        assert np.isclose(float(value), 2 * 2 * 4 / 2.5e-3)  # 2 ranks x B=2 x K=4 tokens
        assert d0 != d1 and v0 != v1 and c0 != c1        # distinct batches per rank
    assert rows[0] == rows[1]


def test_one_rank_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_throughput(7, 1, 1.0) == 7000.0
