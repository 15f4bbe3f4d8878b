"""The multi-rank host logic of bench.py, as world_size-2 gloo process
groups on the CPU: every rank gets the slowest rank's time, the whole-job
rate counts every rank's units over that time, replicas draw their own
activations, and only rank 0 runs the reference arm."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        times = [0.25, 0.75]            # rank 1 is the slowest
        slowest = bench.max_over_ranks(times[rank], dist, "cpu")
        rate = bench.whole_job_rate(48 * 10, world, slowest)
        out[rank] = (slowest, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, rate = res[rank]
        assert slowest == 0.75
        assert rate == pytest.approx(48 * 10 * 2 / 0.75)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.whole_job_rate(100, 1, 2.0) == 50.0


def test_replicas_draw_their_own_activations():
    import bench
    _, x0, wr0, b0 = bench._gen_layer(("tiny", 3, 0))
    _, x1, wr1, b1 = bench._gen_layer(("tiny", 3, 1))
    assert not np.array_equal(x0, x1)            # each rank its own tokens
    np.testing.assert_array_equal(wr0, wr1)      # the same layer weights
    np.testing.assert_array_equal(b0["gate"], b1["gate"])


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import bench
    class A:  # the fields run_reference reads
        config, steps, warmup, gpus = "tiny", 1, 0, 2
    bench.run_reference(A, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys):
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys, on the same metric and workload as the GPU arm."""
    import json
    import bench

    class A:
        config, steps, warmup, gpus = "tiny", 1, 0, 1
    bench.run_reference(A, rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == "MoE FFN tokens/s (one layer)" and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
