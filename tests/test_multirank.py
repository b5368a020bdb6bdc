"""The multi-GPU path is replicas only (sequences sharded, no data-path
collective).  Its host logic runs here on CPU with two gloo ranks: the whole-job
figure takes the slowest rank's time and every rank's tokens, replicas draw
different sequences, and the reference arm prints from rank 0 alone."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    # rank r timed 10 + 5 r ms over 100 steps of a batch of 32
    total, value = bench.aggregate_ranks(10.0 + 5.0 * rank, 32, 100, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, total, value))


def test_two_replicas_report_the_slowest_rank_and_every_token():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value in res:
        assert total == 15.0                              # max over ranks
        assert abs(value - 2 * 32 * 100 / 0.015) < 1e-6 * value   # all ranks' tokens / that time


def test_single_rank_needs_no_process_group():
    import bench
    total, value = bench.aggregate_ranks(20.0, 32, 100, 1, "cpu")
    assert total == 20.0 and abs(value - 32 * 100 / 0.020) < 1e-6 * value


def test_replicas_draw_different_sequences():
    import bench
    from fp4_compressed_sparse_gb300 import workloads as wl
    rows = []
    for rank in range(2):
        W = wl.tiny_decode(device="cpu")
        W.seed = bench.replica_seed(W.seed, rank)
        rows.append(W.kv(0, 0, 4))
    assert not torch.equal(rows[0], rows[1])
    assert bench.replica_seed(1, 0) == 1


def test_reference_arm_prints_from_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--workload", "tiny_decode", "--gpus", "2"]
    other = subprocess.run(cmd, env=dict(env, RANK="1", LOCAL_RANK="1"), capture_output=True, text=True,
                           timeout=600)
    assert other.returncode == 0 and other.stdout.strip() == ""
    lead = subprocess.run(cmd, env=dict(env, RANK="0", LOCAL_RANK="0"), capture_output=True, text=True,
                          timeout=600)
    assert lead.returncode == 0, lead.stderr[-2000:]
    lines = [l for l in lead.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_launches_its_own_ranks():
    """`bench.py --gpus 2` without a launcher starts two local ranks itself
    (torch.distributed.run on 127.0.0.1); one line comes back, from rank 0."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                           "MASTER_PORT")}
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "tiny_decode"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "4", "--steps", "1"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
