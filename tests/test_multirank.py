"""The N > 1 path on the host: two gloo ranks on CPU run bench.py's rank plumbing.

The scan shards over batch rows, which are independent recurrences: every rank runs its own shard
with no data-path collective, and the only collectives are the timing barrier and the max over ranks.
Checked here: the shards partition the global batch; the max over ranks and the aggregate rate; the
reference arm prints on rank 0 only; and the oracle run shard by shard (one rank each) equals the
oracle run once over the concatenated global batch, bit for bit, so no exchange is missing."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, out_dir):
    _init(rank, world, port)
    import bench
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(1.5 + rank, world)
        rate = bench.aggregate_rate(1000, world, slowest)
        with open(os.path.join(out_dir, f"timing{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "rate": rate, "env": list(bench.dist_env())}, f)
    finally:
        dist.destroy_process_group()


def _oracle_shard_worker(rank, world, port, out_dir):
    _init(rank, world, port)
    import bench
    import oracle
    try:
        cfg = workloads.SCAN_CONFIGS["tiny"]
        d = bench.rank_inputs(cfg, rank)
        y, h, _ = oracle.scan(d, nthreads=1)
        ys = [torch.zeros_like(torch.from_numpy(y)) for _ in range(world)]
        hs = [torch.zeros_like(torch.from_numpy(h)) for _ in range(world)]
        # the gather is the test's own: the product path never exchanges data between ranks
        dist.all_gather(ys, torch.from_numpy(y))
        dist.all_gather(hs, torch.from_numpy(h))
        if rank == 0:
            np.save(os.path.join(out_dir, "y_shards.npy"), torch.cat(ys).numpy())
            np.save(os.path.join(out_dir, "h_shards.npy"), torch.cat(hs).numpy())
    finally:
        dist.destroy_process_group()


def _reference_worker(rank, world, port, out_dir):
    _init(rank, world, port)
    import bench
    try:
        buf = io.StringIO()
        args = SimpleNamespace(workload="tiny", steps=3, warmup=3)
        with redirect_stdout(buf):
            bench.run_reference(args, rank, world)
        with open(os.path.join(out_dir, f"ref{rank}.txt"), "w") as f:
            f.write(buf.getvalue())
    finally:
        dist.destroy_process_group()


def _spawn(fn, world, tmp_path):
    mp.start_processes(fn, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True, start_method="spawn")


def test_shards_partition_the_global_batch():
    import bench
    for world in (1, 2, 3, 8):
        rows = [r for k in range(world) for r in bench.shard_batches(world, k, 8)]
        assert rows == list(range(8 * world))
    with pytest.raises(ValueError):
        bench.shard_batches(2, 2, 8)


def test_rank_shards_share_parameters_and_differ_in_rows():
    import bench
    cfg = workloads.SCAN_CONFIGS["tiny"]
    a, b = bench.rank_inputs(cfg, 0), bench.rank_inputs(cfg, 1)
    for k in ("A", "Dskip", "delta_bias"):
        assert torch.equal(a[k], b[k]), k
    for k in ("u", "delta", "z", "Bm", "Cm"):
        assert not torch.equal(a[k], b[k]), k


def test_max_over_ranks_and_aggregate_rate_gloo(tmp_path):
    _spawn(_timing_worker, 2, tmp_path)
    got = [json.load(open(tmp_path / f"timing{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert g["slowest"] == 2.5
        assert g["rate"] == pytest.approx(2 * 1000 / 2.5e-3)
        assert g["env"] == [r, 2, r]


def test_sharded_oracle_equals_one_run_over_the_global_batch(tmp_path):
    import bench
    import oracle
    world = 2
    _spawn(_oracle_shard_worker, world, tmp_path)
    cfg = workloads.SCAN_CONFIGS["tiny"]
    shards = [bench.rank_inputs(cfg, r) for r in range(world)]
    glob = dict(shards[0])
    for k in ("u", "delta", "z", "Bm", "Cm"):
        glob[k] = torch.cat([s[k] for s in shards])
    y, h, _ = oracle.scan(glob, nthreads=1)
    assert np.array_equal(np.load(tmp_path / "y_shards.npy"), y)
    assert np.array_equal(np.load(tmp_path / "h_shards.npy"), h)


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    _spawn(_reference_worker, 2, tmp_path)
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": "elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
