"""bench.py's multi-rank path on CPU with the gloo backend, world size 2:
every rank ends with the slowest rank's timings, the whole-job value counts
the work of all ranks, and the reference arm does nothing on ranks other
than 0.  The ranks are separate processes launched with the environment
variables torchrun sets."""
import json
import os
import socket
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(world):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "multirank_worker.py")],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=240)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return sorted(outs, key=lambda o: o["rank"])


def test_two_ranks_take_the_slowest_timing_and_sum_the_work():
    outs = _launch(2)
    assert [o["rank"] for o in outs] == [0, 1]
    for o in outs:
        # rank 1 was slower in the timed region, rank 0 slower end to end
        assert o["t_ms"] == 107.0 and o["e2e_ms"] == 300.0
        # 2 ranks x 1 TFLOP x 10 steps in 0.107 s
        assert o["value"] == pytest.approx(2 * 10 / 0.107)
    assert outs[1]["reference_stdout"] == "" and outs[1]["reference_ret"] is None


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, [3, 4.5], "cpu") == [3.0, 4.5]
    assert bench.job_throughput(1, 2e12, 5, 1000.0) == pytest.approx(10.0)
    assert bench.job_throughput(4, 2e12, 5, 1000.0) == pytest.approx(40.0)
