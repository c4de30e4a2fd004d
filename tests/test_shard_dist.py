"""The row-sharded lookup's exchange protocol (sharded_lookup) over real torch.distributed ranks on
the CPU (gloo, world size 2 and 3): each rank holds its shard of the table (rows [r * part,
(r + 1) * part), part = ceil(rows / world)) and looks up its own indices, out-of-range ones included;
every rank's result must equal the world-size-1 oracle lookup on the whole table bit for bit. The
device steps (pack, shard lookup, unpack) run as their plain references here (the numpy partition,
the C oracle); tests/test_gpu_shard.py checks the library's kernels against the same references."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _table(rows, D, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30  # no NaN codes
    scales = rng.uniform(0.01, 1.0, size=(rows, 1)).astype(np.float32)
    return codes, scales


def _rank(rank, world, port, rows, D, same_tokens, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import gram_hash_embedding_gb300 as geng
    import oracle
    from tests import shard_ref as R

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        codes, scales = _table(rows, D, 7)
        part = geng.shard_part(rows, world)
        assert part == R.part_of(rows, world)
        lo, hi = min(rank * part, rows), min((rank + 1) * part, rows)
        W_shard, S_shard = codes[lo:hi], scales[lo:hi]
        rng = np.random.default_rng(100 + (0 if same_tokens else rank))
        idx = rng.integers(-3, rows + 3, size=(5, 37)).astype(np.int64)
        idx[0, :4] = [0, rows - 1, -1, rows]  # the table's edges and just past them

        def pack(i, rows_, world_):
            c, l, p = R.pack_ref(i.numpy(), rows_, world_)
            return torch.from_numpy(c), torch.from_numpy(l), torch.from_numpy(p)

        def lookup(r, W, S):
            bits = oracle.engram_lookup(r.numpy(), W, S, W.shape[0], D, D)
            return torch.from_numpy(bits.view(np.int16))

        def unpack(back, positions, m, D_):
            return torch.from_numpy(R.unpack_ref(back.numpy().view(np.uint16), positions.numpy(), m,
                                                 positions.numel(), D_).view(np.int16))

        got = geng.sharded_lookup(torch.from_numpy(idx), W_shard, S_shard, rows, D, world,
                                  geng.dist_exchange(), ops=(pack, lookup, unpack))
        exp = oracle.engram_lookup(idx, codes, scales, rows, D, D)
        q.put((rank, bool(np.array_equal(got.numpy().view(np.uint16), exp)), got.shape == exp.shape))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,rows,same_tokens", [(2, 1003, False), (2, 1003, True), (3, 10, False),
                                                    (3, 2, False)])
def test_sharded_lookup_equals_the_whole_table(world, rows, same_tokens):
    """rows=2 over 3 ranks leaves the last rank an empty shard; same_tokens is the pages' own case
    (every rank looks up the same indices, as tensor parallelism does)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, rows, 32, same_tokens, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert all(ok and shape for _, ok, shape in res), res


@pytest.mark.parametrize("rows,world", [(1003, 2), (10, 3), (2, 3), (1, 8), (768022850, 8), (5, 1)])
def test_partition_covers_every_row_once(rows, world):
    import gram_hash_embedding_gb300 as geng
    from tests import shard_ref as R

    part = geng.shard_part(rows, world)
    sizes = [max(0, min(rows, (r + 1) * part) - min(rows, r * part)) for r in range(world)]
    assert sum(sizes) == rows and all(s <= part for s in sizes)
    probe = np.array([0, rows - 1, rows, -1, rows // 2], dtype=np.int64)
    c, l, p = R.pack_ref(probe, rows, world)
    assert c[world] == 2 and c.sum() == probe.size
    owned = p[:probe.size - 2]
    assert np.all((l[:probe.size - 2] >= 0) & (l[:probe.size - 2] < part))
    assert set(owned.tolist()) == {0, 1, 4}
