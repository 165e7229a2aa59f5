"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The decode-step path has no exchange step: N GPUs run N independent replicas.
What needs checking without GPUs is the job-level aggregation (barrier, max of
the per-rank elapsed times, whole-job steps/s) and that the reference arm runs
on rank 0 only.
"""

import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [2.0, 3.0][rank]  # rank 1 is the slow replica
    bench.barrier(world)
    value, el = bench.job_throughput(10, elapsed, world, device="cpu")
    out[rank] = (value, el)
    dist.destroy_process_group()


def test_job_throughput_over_two_gloo_ranks():
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    for rank in (0, 1):
        value, el = res[rank]
        assert el == 3.0  # the slowest rank sets the job time
        assert value == pytest.approx(2 * 10 / 3.0)


def test_reference_arm_is_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(impl="reference", gpus=2, steps=1, warmup=0,
                                    workload="llama2-7b-128k-32layer", layers=None)
    bench.run_reference(args)  # must return without work or output on rank 1
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line(monkeypatch, capsys):
    """Rank 0's reference line carries the keys of the benchmark contract: the
    oracle timed on the host cores, its own e2e with no device copies."""
    import json

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    args = bench.argparse.Namespace(impl="reference", gpus=1, steps=1, warmup=0,
                                    workload="tiny-1layer-mha8-4k", layers=None)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny-1layer-mha8-4k"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["ms_per_step"] == pytest.approx(1e3 / line["value"], rel=1e-3)
