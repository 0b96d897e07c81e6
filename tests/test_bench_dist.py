"""The benchmark's multi-rank path on CPU: world size 2 over gloo.

Each rank runs its own copy of the workload (heads are independent; no data-path
collective); the job's time is the slowest rank's and its work is every rank's."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup(backend="gloo")
    assert (w, r) == (world, rank)
    # rank r took (r + 1) * 10 ms for 5 steps of 1e9 flop each
    ms, tflops = bench.aggregate(10.0 * (rank + 1), 5, 1e9, w)
    bench.barrier(w)
    out.put((rank, ms, tflops))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_sums_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29517
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, tflops in res:
        assert ms == pytest.approx(20.0 / 5)                  # slowest rank: 20 ms / 5 steps
        assert tflops == pytest.approx(2 * 1e9 / 4e-3 / 1e12)  # both ranks' work


def test_single_rank_aggregate_is_local():
    sys.path.insert(0, ROOT)
    import bench
    ms, tflops = bench.aggregate(8.0, 4, 2e9, 1)
    assert ms == 2.0 and tflops == pytest.approx(2e9 / 2e-3 / 1e12)


def test_reference_arm_under_torchrun_prints_one_line(oracle_mod):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29519", "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload",
           "t512_w128_s0"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("args", [
    ["--pass", "bwd", "--workload", "t512_w128_s0"],
    ["--pass", "decode", "--decode-workload", "decode_b8_w4096"],
], ids=["bwd", "decode"])
def test_reference_arms_of_the_other_passes(oracle_mod, args):
    """The oracle arm of the backward and decode passes prints one line with the same
    metric and unit as the GPU arm of that pass."""
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", *args], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    want = bench.BWD_METRIC if args[1] == "bwd" else bench.DECODE_METRIC
    assert line["impl"] == "reference" and line["metric"] == want and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["value"] == line["value"]
