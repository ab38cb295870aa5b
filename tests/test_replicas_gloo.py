"""The N > 1 path of bench.py runs independent replicas: no data-path collective,
only a barrier and a max over ranks of the measured time.  This checks those
helpers with two gloo ranks on the CPU, and that only rank 0 of the reference arm
prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


WORKER = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import torch
import bench
rank, world, dist = bench.dist_init(torch)
assert world == 2 and dist is not None
mine = 1.5 if rank == 0 else 4.25
bench.barrier(dist)
got = bench.max_over_ranks(torch, dist, mine, torch.device("cpu"))
print(json.dumps({"rank": rank, "max": got}))
dist.destroy_process_group()
"""


def _launch(code_or_args, nproc=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(nproc):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(nproc),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, *code_or_args], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_max_over_ranks_gloo_world2():
    outs = _launch(["-c", WORKER, ROOT])
    vals = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(v["rank"] for v in vals) == [0, 1]
    assert all(v["max"] == 4.25 for v in vals)


def test_reference_arm_prints_on_rank0_only():
    outs = _launch([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
                    "--warmup", "0", "--workload", "fp32-256x1024"])
    lines = [[ln for ln in o.splitlines() if ln.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and len(lines[1]) == 0
    d = json.loads(lines[0][0])
    assert d["impl"] == "reference" and d["unit"] == "ms" and d["higher_is_better"] is False
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
