"""Host-side plan of a row-sharded Periodic Row-wise Muon step (a design for N GPUs).

Nothing here launches work or does the method's arithmetic: it decides which rows of
each matrix a rank holds, which matrices need a collective on RowNorm steps, and
which rank runs each matrix's Newton-Schulz on refresh steps.  It follows the
distributed-implementation paragraph of "Scaling Muon for Diffusion Transformers"
(summary page): W, G and M are sharded by rows (FSDP2 dim 0); on RowNorm steps the
rows of a wide matrix are local and need no communication, and a tall matrix only
combines its per-column sums of squares across ranks; refresh steps need whole
matrices.  The single-GPU library computes every piece (momentum, batched NS5 over
any subset of matrices, RowNorm, apply); only one GPU is available here, so the plan
is exercised on CPU ranks (gloo) in the tests and is not measured on hardware.
"""
from __future__ import annotations

import heapq
from typing import Dict, List, Sequence, Tuple


def row_shard(rows: int, world: int, rank: int) -> Tuple[int, int]:
    """Rows [r0, r1) of an A x B matrix held by `rank` (even split, the last ranks
    taking the remainder's absence: FSDP's dim-0 chunking)."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("bad shard request")
    per = -(-rows // world)
    r0 = min(rows, rank * per)
    return r0, min(rows, r0 + per)


def lines_are_rows(rows: int, cols: int) -> bool:
    """RowNorm lines of the FULL matrix: rows when A <= B (wide or square), columns
    when A > B (tall).  A shard of a tall matrix may itself be wide; the geometry is
    always the full matrix's."""
    return rows <= cols


def needs_column_exchange(rows: int, cols: int) -> bool:
    """Tall matrices: each column spans every rank's rows, so the ranks must combine
    their per-column sums of squares (cols floats each) before normalising."""
    return not lines_are_rows(rows, cols)


def ns5_cost(rows: int, cols: int) -> int:
    """Symmetric-minimum Newton-Schulz work 5*(3 n^2 m + n^3), n = min, m = max."""
    n, m = min(rows, cols), max(rows, cols)
    return 5 * (3 * n * n * m + n ** 3)


def refresh_owners(shapes: Sequence[Tuple[int, int]], world: int) -> List[int]:
    """Owner rank of each matrix's Newton-Schulz: longest processing time first by
    ns5_cost, ties to the lowest rank.  The owner gathers the matrix's shards, runs
    NS5, and returns each rank its rows of the result."""
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(shapes)), key=lambda i: (-ns5_cost(*shapes[i]), i))
    heap = [(0, r) for r in range(world)]
    owner = [0] * len(shapes)
    for i in order:
        load, r = heapq.heappop(heap)
        owner[i] = r
        heapq.heappush(heap, (load + ns5_cost(*shapes[i]), r))
    return owner


def step_comm_bytes(shapes: Sequence[Tuple[int, int]], world: int, refresh: bool, x_bytes: int = 2) -> Dict[str, int]:
    """Bytes a rank sends per step under the plan (for sizing, not measured).
    RowNorm steps: the rank's column partials of every tall matrix, sent to each other
    rank (fp32).  Refresh steps, averaged over the ranks: each matrix's shards held
    outside its owner go to the owner as bf16 X~ (a fraction (world - 1)/world of the
    matrix), and the owner's result rows come back (bf16)."""
    if not refresh:
        cols = sum(c for (r, c) in shapes if needs_column_exchange(r, c))
        return {"column_partials": 4 * cols * (world - 1)}
    total = sum(2 * r * c * x_bytes * (world - 1) // world for (r, c) in shapes)   # gather + scatter
    return {"gather_scatter": total // world}
