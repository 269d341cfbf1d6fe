"""Host-side logic of the multi-GPU benchmark on CPU: two gloo ranks.

The forward shards over (b, head) with no exchange step, so `bench.py --gpus N`
runs one replica of the workload per rank; the only cross-rank steps are the
barrier and the max-over-ranks reduction of the timed region, checked here with
world_size 2 on the gloo backend (no GPU)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_seconds = 1.5 if rank == 0 else 2.5          # rank 1 is the slow one
        bench.barrier()
        worst = bench.reduce_max(local_seconds, "cpu")
        out[rank] = worst
        if rank == 0:
            out[2] = bench.whole_job_tflops(1.0e12, 10, world, worst)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == 2.5 and out[1] == 2.5                 # every rank sees the slowest time
    assert out[2] == pytest.approx(1.0e12 * 10 * 2 / 2.5 / 1e12)   # all ranks' work / max time


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # rank 1 returns 0 at once: no inputs drawn, no oracle run
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0


def test_bench_rejects_short_warmup():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_reference_arm_prints_contract_line(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "3", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
