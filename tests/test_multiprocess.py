"""The multi-process bench path on CPU: two `gloo` ranks.

Each GPU of a multi-GPU run is an independent replica with its own batch of
requests; the ranks meet only at the timing barrier and the max / sum
reductions of the reported numbers.  These tests run that host logic with
world size 2 on the CPU, and check that the replicas draw disjoint request
ids (so their random streams never coincide).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_pattern):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

    r, wsz, local = bench._dist_init(world)
    bench._barrier(wsz)
    mx = bench._max_over_ranks(1.5 + rank, wsz)
    total = bench._sum_over_ranks(10.0 * (rank + 1), wsz)
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, rank, device="cpu", request_id_base=rank * w.B)
    ids = [None] * wsz
    dist.all_gather_object(ids, inp["request_id"].tolist())
    bench._barrier(wsz)
    with open(out_pattern % rank, "w") as f:
        json.dump(dict(rank=r, world=wsz, local=local, mx=mx, total=total, ids=ids,
                       backend=dist.get_backend()), f)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_shard(tmp_path):
    port = _free_port()
    pattern = str(tmp_path / "rank%d.json")
    mp.start_processes(_worker, args=(2, port, pattern), nprocs=2, start_method="spawn")
    res = [json.load(open(pattern % r)) for r in range(2)]
    for r, d in enumerate(res):
        assert (d["rank"], d["world"], d["local"]) == (r, 2, r)
        assert d["backend"] == "gloo"
        assert d["mx"] == 2.5          # max over ranks of 1.5 + rank
        assert d["total"] == 30.0      # 10 + 20: positions of all replicas add up
    ids0, ids1 = res[0]["ids"]
    assert ids0 == res[1]["ids"][0] and ids1 == res[1]["ids"][1]
    assert not set(ids0) & set(ids1), "replicas must draw disjoint request ids"


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_line_on_rank_zero():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
