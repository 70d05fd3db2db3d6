"""The sharded multi-rank path of bench.py, run as two gloo ranks on the CPU:
disjoint lane blocks, the job time is the slowest rank's, the job's work is
the sum over ranks, and only rank 0 of the reference arm prints."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    lanes = bench.rank_lanes(rank, 3)
    # rank r "took" 10 + r seconds and decoded 100 * (r + 1) frames
    mx, sm = bench.reduce_over_ranks(dist, torch.device("cpu"), [10.0 + rank, 1.0], [100.0 * (rank + 1)])
    gathered = [None] * ws
    dist.all_gather_object(gathered, lanes)
    out[rank] = (mx, sm, gathered, bench.job_rate(sm[0], mx[0]))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_lanes_and_reduce():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    for rank in range(ws):
        mx, sm, gathered, rate = res[rank]
        assert mx == [11.0, 1.0]                     # slowest rank's time
        assert sm == [300.0]                         # every rank's frames
        assert rate == pytest.approx(300.0 / 11.0)
        flat = [b for g in gathered for b in g]
        assert flat == list(range(6))                # disjoint, covering blocks


def test_single_rank_needs_no_process_group():
    mx, sm = bench.reduce_over_ranks(None, None, [2.5], [7.0])
    assert mx == [2.5] and sm == [7.0]
    assert bench.rank_lanes(0, 4) == [0, 1, 2, 3]


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "0"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=280)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.timeout(300)
def test_reference_arm_rank_zero_prints_one_line():
    import json
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "0"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=280)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == "frames/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object as the GPU arm's line (2 ranks x the workload's lanes)
    import synth
    wl = synth.workload(0)
    assert d["config"] == bench.workload_config(wl, synth.make_graph(0), wl.B, 2, 0)
