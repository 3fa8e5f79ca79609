"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The attention path has no exchange step, so N GPUs run N independent
replicas; what is shared is host logic: the process-group setup, the
barriers around the timed region, the maximum of the step time over ranks and
the whole-job throughput (units of all ranks / slowest rank's time).  These
tests run that logic as two gloo ranks on CPU, and the reference arm of
bench.py under torchrun, where rank 0 alone times the oracle and prints one
line and rank 1 exits 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, REPO)
    import bench
    import torch.distributed as dist

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # Rank r "took" 1.5 + r ms per step; everyone must agree on the slowest.
    ms = bench.max_over_ranks(1.5 + r, w)
    bench.barrier(w)
    rate = bench.whole_job_rate(1000.0, ms, w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ms": ms, "rate": rate}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    slowest = 1.5 + (world - 1)
    for r in res:
        assert r["ms"] == pytest.approx(slowest)
        # 2 ranks x 1000 units in 2.5 ms = 800,000 units/s.
        assert r["rate"] == pytest.approx(world * 1000.0 / (slowest * 1e-3))


def test_whole_job_rate_single_rank():
    sys.path.insert(0, REPO)
    import bench
    assert bench.whole_job_rate(5e12, 10.0, 1) == pytest.approx(5e14)
    assert bench.whole_job_rate(5e12, 10.0, 4) == pytest.approx(2e15)


@pytest.mark.parametrize("extra", [["--workload", "decode", "--decode-tokens", "2"],
                                   ["--workload", "vit_full_d80"]],
                         ids=["decode", "varlen"])
def test_reference_arm_under_torchrun(extra):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--cpu-budget", "0.4"] + extra
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=REPO, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
