"""The row-sharded step of the design (matrix_aware_optimizer_muon_gb300.shard) on two
gloo ranks on the CPU: every rank holds a row shard of W, G and M; RowNorm steps
normalise wide rows locally and combine tall matrices' column sums of squares in rank
order; refresh steps run each matrix's Newton-Schulz on its owner over the gathered
momentum.  The oracle supplies the arithmetic; the assembled result must equal the
unsharded oracle step.  (The plan is not measured on hardware: one GPU here.)"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from matrix_aware_optimizer_muon_gb300 import shard  # noqa: E402
from test_replicas_gloo import _free_port  # noqa: E402

WORKER = r"""
import json, math, sys
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import torch.distributed as dist
from oracle import muon_ref
from synth import gradient_np, weight_init_np
from matrix_aware_optimizer_muon_gb300 import shard

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
shapes = [(96, 40), (40, 96), (48, 48), (130, 24), (9, 31)]   # tall, wide, square, tall, wide
steps, K = 4, 3
owners = shard.refresh_owners(shapes, world)
err = 0.0
for i, (A, B) in enumerate(shapes):
    r0, r1 = shard.row_shard(A, world, rank)
    W_full = weight_init_np(A, B, 5, i).astype(np.float64)
    W_ref, M_ref = W_full.copy(), np.zeros((A, B))
    W, M = W_full[r0:r1].copy(), np.zeros((r1 - r0, B))
    for t in range(steps):
        G_full = gradient_np(A, B, (1e-2,) * 2, 5, i, t).astype(np.float64)
        W_ref, M_ref, refresh = muon_ref.periodic_step(W_ref, M_ref, G_full, t, K)
        M = muon_ref.momentum(M, G_full[r0:r1], 0.95)
        if refresh:
            # gather the momentum on every rank (gloo all_gather of the row shards); the
            # owner runs NS5 and the rows come back to their ranks (broadcast from the owner)
            per = -(-A // world)
            buf = torch.zeros(per, B, dtype=torch.float64)
            buf[: r1 - r0] = torch.from_numpy(M)
            parts = [torch.zeros(per, B, dtype=torch.float64) for _ in range(world)]
            dist.all_gather(parts, buf)
            full = torch.cat(parts)[:A].numpy()
            O = torch.from_numpy(muon_ref.newton_schulz(full) if rank == owners[i] else np.zeros((A, B)))
            dist.broadcast(O, src=owners[i])
            U = O.numpy()[r0:r1]
            s = muon_ref.update_scale(A, B, True, 0.15)
        elif shard.needs_column_exchange(A, B):
            part = torch.from_numpy(np.sum(M * M, axis=0))
            parts = [torch.zeros(B, dtype=torch.float64) for _ in range(world)]
            dist.all_gather(parts, part)
            ss = parts[0].numpy().copy()
            for q in range(1, world):     # rank order: independent of the topology
                ss = ss + parts[q].numpy()
            nrm = np.sqrt(ss)
            U = np.where(nrm == 0.0, 0.0, M / np.where(nrm == 0.0, 1.0, nrm))
            s = muon_ref.update_scale(A, B, False, 0.15)
        else:
            U = muon_ref.rownorm(M) if M.size else M     # whole rows are local
            s = muon_ref.update_scale(A, B, False, 0.15)
        W = muon_ref.apply_update(W, U, s, 0.02, 0.01)
        err = max(err, float(np.max(np.abs(W - W_ref[r0:r1]))) if W.size else 0.0,
                  float(np.max(np.abs(M - M_ref[r0:r1]))) if M.size else 0.0)
print(json.dumps({"rank": rank, "err": err, "owners": owners}))
dist.destroy_process_group()
"""


def test_row_sharded_step_matches_unsharded_oracle_gloo_world2():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["err"] < 1e-12, o


def test_shard_plan():
    assert shard.row_shard(10, 4, 0) == (0, 3) and shard.row_shard(10, 4, 3) == (9, 10)
    assert [shard.row_shard(5, 8, r) for r in range(8)][-1] == (5, 5)   # empty shards allowed
    assert sum(r1 - r0 for r0, r1 in (shard.row_shard(9216, 3, r) for r in range(3))) == 9216
    assert shard.lines_are_rows(48, 48) and not shard.needs_column_exchange(40, 96)
    assert shard.needs_column_exchange(9216, 3072)
    # 15B set on 8 ranks: owners balanced to within one matrix's cost of each other
    from synth import WORKLOADS
    shapes = [(m.rows, m.cols) for m in WORKLOADS["mmdit-15b"].matrices]
    own = shard.refresh_owners(shapes, 8)
    loads = [0] * 8
    for s, o in zip(shapes, own):
        loads[o] += shard.ns5_cost(*s)
    assert max(loads) - min(loads) <= max(shard.ns5_cost(*s) for s in shapes)
    # RowNorm-step exchange: the column partials of the tall matrices only (qkv, MLP-up, adaLN)
    cb = shard.step_comm_bytes(shapes, 8, refresh=False)["column_partials"]
    assert cb == 4 * 3072 * 88 * 3 * 7
    with pytest.raises(ValueError):
        shard.row_shard(4, 0, 0)
