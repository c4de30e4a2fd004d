"""The cache-row map (call row b uses cache row cache_rows[b]) vs the oracle given the same map:
sequences that change call rows and call order between calls, dense and packed, hash-only and
fused; rows mapped outside the cache; the identity map (GPU only)."""
import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    H.build_all()
    wl = synth.make_workload(0, full64=True)
    Ws, Ss = H.device_tables(wl)
    yield wl, Ws, Ss
    del Ws, Ss
    torch.cuda.empty_cache()


def _i32(a):
    return H.to_dev(np.asarray(a, dtype=np.int32))


def test_sequences_move_between_call_rows(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    n_seq, total, n_slots = 4, 400, 6
    rng = np.random.default_rng(71)
    ids = rng.integers(0, lay.raw_vocab, size=(n_seq, total))
    mask = rng.random((n_seq, total)) > 0.1
    slot = [5, 0, 3, 2]  # sequence s lives in cache row slot[s]
    st, orc = H.make_state(wl, n_slots, 512), H.make_oracle(wl, n_slots, 512)
    pos = [0] * n_seq
    plan = [([0, 1, 2, 3], 37), ([3, 1], 16), ([2], 64), ([1, 3, 0, 2], 17), ([0, 2], 5), ([3, 2, 1, 0], 1)]
    for k, (order, Lc) in enumerate(plan):
        cid = np.stack([ids[s, pos[s]:pos[s] + Lc] for s in order])
        cm = np.stack([mask[s, pos[s]:pos[s] + Lc] for s in order])
        sp = np.array([pos[s] for s in order], dtype=np.int32)
        rows = np.array([slot[s] for s in order], dtype=np.int32)
        exp_h, fl = orc.hash(cid, sp.astype(np.int64), cm, cache_rows=rows)
        assert fl == 0
        hashes = torch.full((len(order), Lc, 1, 6), -9, dtype=torch.int64, device="cuda")
        if k % 2 == 0:  # fused
            outs = st.hash_lookup(H.to_dev(cid), Ws, Ss, start_pos=_i32(sp), mask=H.to_dev(cm), hashes=hashes,
                                  cache_rows=_i32(rows))
            H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), f"rows {k}")
        else:           # hash only
            st.hash(H.to_dev(cid), _i32(sp), H.to_dev(cm), hashes=hashes, cache_rows=_i32(rows))
        H.assert_bits_equal(hashes.cpu().numpy(), exp_h, f"hashes of call {k}")
        for s in order:
            pos[s] += Lc
    # packed, sequences of different lengths (one empty) in another order
    order, lens = [2, 0, 3, 1], [9, 0, 30, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pid = np.concatenate([ids[s, pos[s]:pos[s] + n] for s, n in zip(order, lens)])
    pm = np.concatenate([mask[s, pos[s]:pos[s] + n] for s, n in zip(order, lens)])
    sp = np.array([pos[s] for s in order], dtype=np.int32)
    rows = np.array([slot[s] for s in order], dtype=np.int32)
    exp_h, fl = orc.hash_varlen(pid, cu, sp, pm, cache_rows=rows)
    assert fl == 0
    hashes = torch.full((pid.size, 1, 6), -9, dtype=torch.int64, device="cuda")
    outs = st.hash_lookup_varlen(H.to_dev(pid), H.to_dev(cu), _i32(sp), Ws, Ss, mask=H.to_dev(pm), hashes=hashes,
                                 max_len=max(lens), cache_rows=_i32(rows))
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "packed hashes")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, 0, :]), "packed rows")
    h2 = st.hash_varlen(H.to_dev(pid[:0]), H.to_dev(np.zeros(5, np.int32)), _i32(sp), max_len=1,
                        cache_rows=_i32(rows))  # empty pack: a no-op
    assert h2.numel() == 0
    assert st.status() == 0


def test_rows_mapped_outside_the_cache(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(72)
    ids = rng.integers(0, lay.raw_vocab, size=(3, 50))
    st, orc = H.make_state(wl, 4, 128), H.make_oracle(wl, 4, 128)
    st.hash(H.to_dev(ids[:, :20]), 0)
    orc.hash(ids[:, :20], 0)
    rows = np.array([4, 1, -1], dtype=np.int32)  # 4 == max_batch: outside, as is -1
    sp = np.full(3, 20, np.int32)
    hashes = torch.full((3, 30, 1, 6), -9, dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(ids[:, 20:]), Ws, Ss, start_pos=_i32(sp), hashes=hashes, cache_rows=_i32(rows))
    exp_h, fl = orc.hash(ids[:, 20:], sp.astype(np.int64), cache_rows=rows)
    assert fl == geng.STATUS_BAD_ROW and st.status() == geng.STATUS_BAD_ROW
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "hashes with bad rows")
    assert (exp_h[[0, 2]] == -1).all()
    assert not outs[0][[0, 2]].view(torch.int16).any()  # +0 rows
    H.assert_bits_equal(H.bf16_bits(outs[0][1]), H.oracle_lookup_rows(wl, 0, exp_h[1, :, 0, :]), "good row")
    # the skipped rows wrote nothing: continuing cache row 0 (never mapped) still sees its own history
    h = st.hash(H.to_dev(ids[:1, 20:30]), 20)
    e, _ = orc.hash(ids[:1, 20:30], 20)
    H.assert_bits_equal(h.cpu().numpy(), e, "cache row 0 after the skipped rows")


def test_identity_map_and_row_groups_equal_one_call(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(73)
    B, L = 5, 96
    ids = H.to_dev(rng.integers(0, lay.raw_vocab, size=(B, L)))
    mask = H.to_dev(rng.random((B, L)) > 0.1)
    sp = _i32([0, 7, 30, 3, 12])
    one = H.make_state(wl, B, 256)
    h1 = torch.empty((B, L, 1, 6), dtype=torch.int64, device="cuda")
    o1 = one.hash_lookup(ids, Ws, Ss, start_pos=sp, mask=mask, hashes=h1)
    ident = H.make_state(wl, B, 256)
    hi = torch.empty_like(h1)
    ident.hash_lookup(ids, Ws, Ss, start_pos=sp, mask=mask, hashes=hi, cache_rows=_i32(np.arange(B)))
    assert torch.equal(h1, hi)
    # groups of rows, each call mapped onto its rows' own cache rows, writing into row slices
    grouped = H.make_state(wl, B, 256)
    h2 = torch.full_like(h1, -7)
    o2 = [torch.full_like(o, 3.0) for o in o1]
    for b0, b1 in ((0, 2), (2, 3), (3, 5)):
        grouped.hash_lookup(ids[b0:b1], Ws, Ss, start_pos=sp[b0:b1], mask=mask[b0:b1],
                            out=[o[b0:b1] for o in o2], hashes=h2[b0:b1], cache_rows=_i32(np.arange(b0, b1)))
    assert torch.equal(h1, h2)
    assert torch.equal(o1[0].view(torch.int16), o2[0].view(torch.int16))
    # and the three caches agree: a continuation of every row hashes alike
    nxt, sp2 = ids[:, :8].contiguous(), sp + L
    a, b, c = one.hash(nxt, sp2), ident.hash(nxt, sp2), grouped.hash(nxt, sp2)
    assert torch.equal(a, b) and torch.equal(a, c)
    assert one.status() == 0 and ident.status() == 0 and grouped.status() == 0


def test_prepared_call_with_a_map(tiny):
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(74)
    B, L = 3, 33
    ids = H.to_dev(rng.integers(0, lay.raw_vocab, size=(B, L)))
    sp = _i32([0, 0, 0])
    rows = _i32([2, 0, 1])
    st, orc = H.make_state(wl, 3, 128), H.make_oracle(wl, 3, 128)
    out = [torch.empty((B, L, 6, lay.head_dim), dtype=torch.bfloat16, device="cuda")]
    hashes = torch.empty((B, L, 1, 6), dtype=torch.int64, device="cuda")
    call = st.prepare_hash_lookup(ids, sp, Ws, Ss, out, hashes=hashes, cache_rows=rows)
    call()
    exp_h, _ = orc.hash(ids.cpu().numpy(), 0, cache_rows=[2, 0, 1])
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "prepared with map")
    # next chunk after a refill in place: rows keep their cache rows
    ids.copy_(H.to_dev(rng.integers(0, lay.raw_vocab, size=(B, L))))
    sp.fill_(L)
    call()
    exp_h, _ = orc.hash(ids.cpu().numpy(), L, cache_rows=[2, 0, 1])
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "prepared with map, second chunk")
    H.assert_bits_equal(H.bf16_bits(out[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), "prepared rows")


def test_a_reused_row_needs_no_reset(tiny):
    """Continuous batching reuses a finished sequence's cache row for a new sequence starting at
    position 0: the new sequence reads only positions it writes itself, so its hash ids equal those
    of the same sequence on a fresh state, while another sequence decodes in the next row."""
    wl, Ws, Ss = tiny
    lay = wl.layout
    rng = np.random.default_rng(73)
    old = rng.integers(0, lay.raw_vocab, size=(1, 300))
    other = rng.integers(0, lay.raw_vocab, size=(1, 301))
    new = rng.integers(0, lay.raw_vocab, size=40)
    st = H.make_state(wl, 2, 512)
    for c0 in range(0, 300, 100):  # the finished sequence: three chunks in row 0
        st.hash(H.to_dev(old[:, c0:c0 + 100]), _i32([c0]), cache_rows=_i32([0]))
    st.hash(H.to_dev(other[:, :300]), _i32([0]), cache_rows=_i32([1]))
    # one packed call: the new sequence (40 tokens at position 0 of row 0), the other decoding at 300
    pid = np.concatenate([new, other[0, 300:301]])
    cu, sp, rows = _i32([0, 40, 41]), _i32([0, 300]), _i32([0, 1])
    h = st.hash_varlen(H.to_dev(pid), cu, sp, max_len=40, cache_rows=rows)
    fresh = H.make_state(wl, 1, 512)
    h_new = fresh.hash(H.to_dev(new.reshape(1, -1)), 0)
    assert torch.equal(h[:40].cpu(), h_new.reshape(40, 1, 6).cpu())
    orc = H.make_oracle(wl, 2, 512)
    orc.hash(other[:, :300], 0, cache_rows=np.array([1]))
    exp_h, fl = orc.hash(other[:, 300:301], np.array([300]), cache_rows=np.array([1]))
    assert fl == 0
    H.assert_bits_equal(h[40:].cpu().numpy().reshape(exp_h.shape), exp_h, "decoding sequence")
    assert st.status() == 0
