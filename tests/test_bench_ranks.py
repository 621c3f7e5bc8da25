"""The bench's multi-rank logic on the CPU: two gloo ranks in separate
processes (the GPU runs use NCCL with one rank per GPU, the same calls).
The path has no exchange step, so the ranks are independent replicas and
only the timing is combined: the job's step time is the slowest rank's, and
the reported rate counts every rank's units."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
local_ms = [12.5, 31.25][rank]           # rank 1 is the slow one
ms = bench.max_over_ranks(local_ms, dist, "cpu")
rate = bench.whole_job_rate(1e9, world, ms)
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "ms": ms, "rate": rate}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(script, world, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), **(extra_env or {}))
        procs.append(subprocess.Popen([sys.executable, *script, *args], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=180)
            assert p.returncode == 0, err
            outs.append(out)
    finally:
        for p in procs:  # a rank left waiting on a failed peer
            if p.poll() is None:
                p.kill()
                p.wait()
    return outs


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    outs = _launch(["-c", RANK_SCRIPT], 2, args=(ROOT,))
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["ms"] == 31.25
        assert r["rate"] == 2 * 1e9 / 31.25e-3


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.whole_job_rate(5.0, 1, 1000.0) == 5.0


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the oracle's arm runs on rank 0 alone; other ranks exit
    0 without work and without output."""
    outs = _launch([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                    "--warmup", "0", "--gpus", "2"], 2)
    assert outs[1].strip() == ""
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
