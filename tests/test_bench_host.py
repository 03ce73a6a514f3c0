"""Host logic of bench.py's replica mode, run as two gloo ranks on the CPU:
the barrier, the max over ranks that sets the job's time, the whole-job value
computed from it, and rank 0 alone printing the reference arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys, time
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
barrier, allmax = bench.dist_helpers("cpu")
barrier()
t0 = time.perf_counter()
if rank == 1:
    time.sleep(0.2)                      # the slow rank sets the job's time
local = time.perf_counter() - t0
barrier()
job = allmax(local)
out = {"rank": rank, "world": world, "local": local, "job": job,
       "max_of_ranks": allmax(float(rank + 1))}
print(json.dumps(out), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code, world=2, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code] if code else [sys.executable, os.path.join(ROOT, "bench.py"), *args]
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_barrier_and_max_over_ranks():
    pytest.importorskip("torch.distributed")
    outs = [json.loads(o.strip().splitlines()[-1]) for o in _run_ranks(WORKER)]
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 for o in outs)
    slow = max(o["local"] for o in outs)
    for o in outs:
        assert o["job"] == pytest.approx(slow)      # both ranks agree on the slowest rank's time
        assert o["max_of_ranks"] == 2.0
    assert slow >= 0.2


def test_reference_arm_prints_on_rank_zero_only():
    outs = _run_ranks(None, args=("--impl", "reference", "--steps", "1", "--warmup", "3"))
    lines = [[ln for ln in o.splitlines() if ln.strip()] for o in outs]
    assert len(lines[1]) == 0                        # rank 1 exits 0 without output
    line = json.loads(lines[0][-1])
    assert line["impl"] == "reference"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_code_hash_ignores_comments_only():
    """The traffic table keys counters by the kernel's code: comment edits keep
    the key, any change to the code changes it."""
    import bench
    src = "// header\n__global__ void k(int* p) {\n    p[0] = 1;   // store\n}\n/* block\n comment */\n"
    same = "__global__ void k(int* p) {\n\n    p[0] = 1;\n}\n// another note\n"
    changed = "__global__ void k(int* p) {\n    p[0] = 2;\n}\n"
    assert bench.code_hash(src) == bench.code_hash(same)
    assert bench.code_hash(src) != bench.code_hash(changed)
