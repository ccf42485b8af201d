"""Row sharding of one layer over G GPUs, with no exchange.

Y = X . W^T splits by output rows: GPU r packs rows row0 .. row0 + rows - 1
of W (whole 128-row groups, so that every shard but the last is made of full
groups of the packed layout), keeps all of X, and writes columns
row0 .. row0 + rows - 1 of Y. The shards' columns are disjoint and together
cover Y; nothing is summed across GPUs. A caller that needs the whole Y on
every GPU gathers the column blocks itself.
"""

from __future__ import annotations

GROUP_ROWS = 128


def row_shards(n: int, world: int, align: int = GROUP_ROWS) -> list[tuple[int, int]]:
    """(row0, rows) of each of `world` shards of n output rows: whole groups
    of `align` rows dealt as evenly as they go (the first n_groups % world
    shards one group more), the last group cut at n. A shard may be empty
    when there are fewer groups than shards."""
    if n < 0 or world < 1 or align < 1:
        raise ValueError("n >= 0, world >= 1 and align >= 1")
    groups = -(-n // align)
    per, extra = divmod(groups, world)
    out, g0 = [], 0
    for r in range(world):
        g = per + (1 if r < extra else 0)
        row0 = min(n, g0 * align)
        out.append((row0, min(n, (g0 + g) * align) - row0))
        g0 += g
    return out


def matmul_row_shard(q4lib, W_shard, X, Y, m: int, k: int, n_total: int, row0: int, rows: int, stream=None):
    """Columns row0 .. row0 + rows - 1 of Y[m x n_total] (row-major, fp32)
    from this shard's packed weights (rows x k, packed by q4_0_pack) and all
    of X[m x k]: the batched-slot call with the identity slot map and Y's
    full row stride, so the shard writes its columns in place."""
    import torch
    if rows == 0 or m == 0:
        return
    slots = torch.arange(m, dtype=torch.int32, device=X.device)
    ws_bytes = q4lib.q4_0_matmul_workspace_size(m, k, rows)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=X.device)
    Ys = Y.view(-1)[row0:]
    q4lib.q4_0_matmul_batched_slots_ws(W_shard, X, k, slots, m, Ys, n_total, k, rows, ws, ws_bytes, stream)
