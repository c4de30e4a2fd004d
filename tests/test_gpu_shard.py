"""The sharded lookup's device steps (GPU only): engram_shard_pack and engram_shard_unpack against the
plain numpy partition (tests/shard_ref.py), bit for bit; and the whole protocol (sharded_lookup) with
W ranks emulated in one process, one Python thread per rank on the same GPU, the all-to-all done as
device copies between the threads: every rank's rows equal the oracle's lookup on the whole table."""
import threading

import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
import synth
from tests import gpu_helpers as H
from tests import shard_ref as R

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


@pytest.mark.parametrize("n,rows,world", [(1, 10, 2), (4095, 1000, 3), (4096, 1000, 8), (4097, 7, 64),
                                          (3 * 4096 + 5, 123457, 5), (1_572_864, 384_006_168, 8), (5000, 3, 1)])
def test_pack_matches_the_stable_partition(n, rows, world):
    rng = np.random.default_rng(n + world)
    idx = rng.integers(-rows // 10 - 2, rows + rows // 10 + 2, size=n).astype(np.int64)
    counts, local, pos = geng.engram_shard_pack(torch.from_numpy(idx).cuda(), rows, world)
    ec, el, ep = R.pack_ref(idx, rows, world)
    assert np.array_equal(counts.cpu().numpy(), ec)
    assert np.array_equal(local.cpu().numpy(), el)
    assert np.array_equal(pos.cpu().numpy(), ep)


@pytest.mark.parametrize("n,D,frac", [(1, 16, 1.0), (777, 128, 0.9), (10_000, 256, 0.5), (300, 64, 0.0)])
def test_unpack_scatters_and_zeroes(n, D, frac):
    rng = np.random.default_rng(n + D)
    positions = rng.permutation(n).astype(np.int64)
    m = int(n * frac)
    rows = rng.integers(0, 1 << 16, size=(m, D), dtype=np.uint16)
    out = torch.full((n, D), 1.0, dtype=torch.bfloat16, device="cuda")  # stale contents are overwritten
    r = torch.from_numpy(rows.view(np.int16)).cuda().view(torch.bfloat16)
    geng.engram_shard_unpack(r, torch.from_numpy(positions).cuda(), m, D, out=out)
    H.assert_bits_equal(H.bf16_bits(out), R.unpack_ref(rows, positions, m, n, D), "unpack")


class _ThreadExchange:
    """all-to-all between W threads of one process: each rank leaves its tensor and split sizes, and
    after a barrier takes its slice from every rank's tensor (device copies, rank 0's first)."""

    def __init__(self, world):
        self.world = world
        self.barrier = threading.Barrier(world)
        self.slots = [None] * world

    def for_rank(self, r):
        def exchange(t, send, recv):
            self.slots[r] = (t, [int(c) for c in send])
            self.barrier.wait()
            parts = []
            for s in range(self.world):
                ts, ss = self.slots[s]
                off = sum(ss[:r])
                parts.append(ts[off:off + ss[r]])
            out = torch.cat(parts)
            assert out.shape[0] == sum(int(c) for c in recv)
            torch.cuda.synchronize()
            self.barrier.wait()  # every rank has copied before the slots are reused
            return out

        return exchange


@pytest.mark.parametrize("world", [2, 4, 8])
def test_sharded_lookup_emulated_ranks(world):
    """The prefill layout's layer-0 table (about 24M rows x 128, fp32 scales) split over `world`
    emulated ranks; each rank hashes its own rows of the batch (the hash is replicated) and looks its
    (token, column) pairs up through the exchange. Plus a few out-of-range indices per rank."""
    wl = synth.make_workload(1)
    lay = wl.layout
    Ws, Ss = H.device_tables(wl)
    rows = lay.rows[0]
    part = geng.shard_part(rows, world)
    B, L = 4, 512
    st = H.make_state(wl, B, L)
    ids = H.to_dev(wl.ids[:B, :L].copy())
    hashes = st.hash(ids, 0)
    idx_all = hashes[:, :, 0, :].contiguous()  # [B, L, C] row ids of layer 0
    per_rank = [idx_all[r % B].reshape(-1).clone() for r in range(world)]
    for r in range(world):
        per_rank[r][:3] = torch.tensor([-1, rows, rows + 5], device="cuda")
    shards = [(Ws[0][min(r * part, rows):min((r + 1) * part, rows)], Ss[0][min(r * part, rows):min((r + 1) * part, rows)])
              for r in range(world)]
    ex = _ThreadExchange(world)
    results, errors = [None] * world, []

    def run(r):
        try:
            torch.cuda.set_device(0)
            results[r] = geng.sharded_lookup(per_rank[r], shards[r][0], shards[r][1], rows, lay.block, world,
                                             ex.for_rank(r))
        except Exception as e:  # pragma: no cover - reported below
            errors.append((r, repr(e)))
            ex.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(300)
    assert not errors, errors
    torch.cuda.synchronize()
    for r in range(world):
        idx = per_rank[r].cpu().numpy()
        exp = H.oracle_lookup_rows(wl, 0, idx)
        H.assert_bits_equal(H.bf16_bits(results[r]), exp, f"sharded lookup, rank {r} of {world}")
        whole = geng.engram_lookup(per_rank[r], Ws[0], Ss[0], lay.block)
        assert torch.equal(whole.view(torch.int16), results[r].view(torch.int16))
