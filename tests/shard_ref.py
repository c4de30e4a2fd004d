"""Plain numpy statement of the sharded lookup's partition, for the tests: rank r of `world` owns rows
[r * part, (r + 1) * part) with part = ceil(rows / world) (engram-first/lookup page,
`ParallelEngramEmbedding`); an index outside [0, rows) is owned by no rank (bucket `world`). The pack
is a stable sort of the indices by owner; the unpack puts rows back at their positions."""
import numpy as np


def part_of(rows: int, world: int) -> int:
    return max(1, -(-int(rows) // int(world)))


def pack_ref(idx, rows: int, world: int):
    idx = np.asarray(idx, dtype=np.int64).reshape(-1)
    part = part_of(rows, world)
    owned = (idx >= 0) & (idx < rows)
    bucket = np.where(owned, np.where(owned, idx, 0) // part, world)
    order = np.argsort(bucket, kind="stable")
    counts = np.bincount(bucket, minlength=world + 1).astype(np.int64)
    local = np.where(bucket < world, idx - bucket * part, idx)[order]
    return counts, local.astype(np.int64), order.astype(np.int64)


def unpack_ref(rows_back, positions, m: int, n: int, D: int):
    out = np.zeros((n, D), dtype=np.uint16)
    out[np.asarray(positions)[:m]] = np.asarray(rows_back).reshape(m, D)
    return out
