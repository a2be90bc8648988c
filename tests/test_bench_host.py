"""Benchmark host logic on CPU: the algorithmic byte counts, the reference
arm's JSON line, and the multi-process timing reduction (world size 2 over
gloo, as torchrun launches it with one process per GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_of_the_large_layer():
    # rank_size 16, shard 8, N = 855,654,400 bf16 per rank, slices of 106,956,800
    N, W, S = 855_654_400, 16, 8
    sizes = {"W": W, "S": S, "N": N, "shard_total": 2 * N, "slice_ag": N // S, "slice_f32": N // S}
    b = bench.algorithmic_bytes(sizes, "bf16", "bf16", "bf16")
    assert b["ag_copy_out"] == 54_761_881_600
    assert b["rs_ar_reduce"] == 34_226_176_000
    assert b["ag_copy_in"] == 2 * N * 2 + W * S * (N // S) * 2 == 30_803_558_400
    assert b["apply_grads"] == 2 * N * 6 == 10_267_852_800


def test_unfused_bytes_of_the_large_layer():
    # the same layer; every slice is N/S elements (no tail), D = 2 replicas
    N, W, S = 855_654_400, 16, 8
    sl = N // S
    sizes = {"W": W, "S": S, "N": N, "shard_total": 2 * N, "slice_ag": sl, "slice_f32": sl,
             "slice_grad": sl}
    b = bench.unfused_bytes(sizes, "bf16", "bf16", "bf16")
    assert b["ag_copy_in_own_slice"] == 2 * N * 2 + W * sl * 2 == 6_845_235_200
    assert b["ag_gather"] == W * sl * 2 * S == 27_380_940_800   # read once, written to 7 others
    assert b["rs_copy_in"] == W * N * 2 * 2 == 54_761_881_600
    assert b["rs_reduce"] == W * S * sl * 2 + W * sl * 4 == 34_226_176_000
    assert b["ar_reduce"] == 2 * W * sl * 4 == 13_690_470_400
    # one rank per shard group: no gather; one replica: no all-reduce
    one = dict(sizes, S=1, slice_ag=N, slice_f32=N, slice_grad=N, shard_total=W * N)
    assert bench.unfused_bytes(one, "bf16", "bf16", "bf16")["ag_gather"] == 0
    full = dict(sizes, W=S)
    assert bench.unfused_bytes(full, "bf16", "bf16", "bf16")["ar_reduce"] == 0


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fsdp", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"]:
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    bench.dist_init(world, "gloo")
    # the slowest rank sets the time; bytes add up over ranks
    t = bench.dist_max(10.0 + rank, world)
    b = bench.dist_sum(1e9 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, t, b))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_timing_reduction_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 11.0, 3e9), (1, 11.0, 3e9)]


@pytest.mark.timeout(600)
def test_reference_arm_under_two_ranks_prints_once():
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2")
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                                       "--workload", "tiny_fsdp", "--steps", "2", "--warmup", "1",
                                       "--gpus", "2"], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True, env=e, cwd=ROOT))
    outs = [p.communicate(timeout=300) for p in procs]
    assert all(p.returncode == 0 for p in procs), [o[1] for o in outs]
    lines = [[l for l in o[0].splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    assert json.loads(lines[0][0])["n_gpus"] == 2
