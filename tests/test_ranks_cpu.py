"""The multi-rank path of the benchmark on the CPU: two gloo ranks.

The decode shards with no exchange (every rank decodes its own replicas), so
the only cross-rank steps are the timing reduction (max over ranks) and the
whole-job value; the rank seeds must give independent inputs, and the
reference arm runs on rank 0 only."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    import kvsynth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w = kvsynth.get_workload("tiny-8k")
        seed = bench.rank_seed(w, rank)
        q = kvsynth.queries(w, step=0, seed=seed)
        ms = 10.0 + 3.0 * rank                      # this rank's own time
        ms_job = bench.max_over_ranks(ms, dist, "cpu")
        e2e = bench.max_over_ranks(0.5 + rank, dist, "cpu")
        value = bench.job_value(world, 64, w.batch, w.layers, ms_job / 1e3)
        qs = [torch.zeros(q.size, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(qs, torch.from_numpy(q.reshape(-1).astype(np.int64)))
        out[rank] = (ms_job, e2e, value, [t.numpy().copy() for t in qs], seed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        ms_job, e2e, value, qs, seed = res[r]
        assert ms_job == 13.0 and e2e == 1.5          # every rank sees the slowest rank's time
        assert value == pytest.approx(world * 64 / 0.013)  # the job's steps over the job's time
    assert res[0][4] != res[1][4]
    qs = res[0][3]
    assert not np.array_equal(qs[0], qs[1])            # independent inputs per rank


def test_reference_arm_only_on_rank_zero(capsys):
    import bench
    import kvsynth
    w = kvsynth.get_workload("tiny-8k")

    class A:
        steps, warmup = 1, 0

    bench.run_reference(A(), w, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(capsys):
    """The reference arm (the float64 oracle on the host cores) prints one JSON line with the
    contract's keys, on the workload it is given."""
    import json
    import bench
    import kvsynth
    w = kvsynth.get_workload("tiny-8k")

    class A:
        steps, warmup = 2, 0

    bench.run_reference(A(), w, rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["config"]["workload"] == "tiny-8k"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
