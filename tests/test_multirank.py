"""The N > 1 host path of bench.py on CPU: world size 2 over gloo.

The (batch x KV head) units are independent, so N GPUs run N replicas with no
data exchange; what crosses ranks is the timing: a barrier around the timed
region and the maximum of the ranks' times.  These tests run that logic as
two CPU processes, and the reference arm under torchrun, where rank 0 alone
runs and prints its one JSON line.  The end-to-end pipeline's piece plan
(host logic of the same script) is checked here too.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's own "time": the job's time is the slowest rank's
    got = bench.max_over_ranks(1.5 + rank, w)
    out.put((rank, got))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--ref-seconds", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_e2e_pieces_cover_every_kv_head_once():
    import bench
    for B, Hkv in [(4, 8), (1, 2), (1, 8), (3, 12), (2, 3), (5, 4)]:
        pieces = bench.e2e_pieces(B, Hkv)
        seen = set()
        for bb, k0, nk in pieces:
            assert nk == Hkv or nk % 4 == 0   # 16-byte-aligned state slices
            for kv in range(k0, k0 + nk):
                assert (bb, kv) not in seen
                seen.add((bb, kv))
        assert seen == {(bb, kv) for bb in range(B) for kv in range(Hkv)}
        # every sequence but the last is one piece
        assert [p for p in pieces if p[0] < B - 1] == [(bb, 0, Hkv) for bb in range(B - 1)]
