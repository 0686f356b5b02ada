"""The multi-GPU path of bench.py is "replicas only": N independent ranks, a
barrier, the max time over ranks and the aggregate.  Its host logic is
checked here with two gloo ranks on the CPU (no GPU, no data-path collective)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, world, local = bench.init_dist()
    import torch.distributed as dist
    assert dist.get_backend() == "gloo" and world == 2 and r == rank
    bench.barrier(world)
    worst = bench.all_reduce_max(10.0 * (rank + 1), world, "cpu")
    # value = all ranks' units / the slowest rank's time
    value = world * 1e12 * 5 / (worst * 1e-3) / 1e12
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"worst_ms": worst, "value": value}, f)
    dist.destroy_process_group()


def test_replica_timing_reduces_to_the_slowest_rank(tmp_path):
    import multiprocessing as mp
    pytest.importorskip("torch")
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0]["worst_ms"] == res[1]["worst_ms"] == 20.0
    assert res[0]["value"] == pytest.approx(2 * 5 / 20e-3)


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-budget", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["value"] > 0 and d["higher_is_better"] is True
