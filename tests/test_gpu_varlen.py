"""Packed variable-length sequences (continuous batching) vs the oracle (GPU only)."""
import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


def _pack(full_ids, full_mask, lens, starts):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = np.concatenate([full_ids[b, starts[b]:starts[b] + lens[b]] for b in range(len(lens))]).astype(np.int64)
    mask = np.concatenate([full_mask[b, starts[b]:starts[b] + lens[b]] for b in range(len(lens))])
    return cu, ids, mask


@pytest.mark.parametrize("lens", [[1] * 8, [5, 0, 17, 1, 40, 3, 16, 33], [0, 0, 0, 7], [100, 1, 1, 1, 64, 65, 15, 2]])
def test_packed_matches_oracle(lens):
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    B = len(lens)
    rng = np.random.default_rng(sum(lens) + B)
    total = 256
    full_ids = rng.integers(0, lay.raw_vocab, size=(B, total))
    full_mask = rng.random((B, total)) > 0.1
    starts = rng.integers(0, 40, size=B).astype(np.int32)
    st, orc = H.make_state(wl, B, 512), H.make_oracle(wl, B, 512)
    Ws, Ss = H.device_tables(wl)
    # history: every row prefilled up to its start with the dense call
    pre = int(starts.max())
    if pre > 0:
        st.hash(H.to_dev(full_ids[:, :pre]), 0, H.to_dev(full_mask[:, :pre]))
        orc.hash(full_ids[:, :pre], 0, full_mask[:, :pre])
    cu, ids, mask = _pack(full_ids, full_mask, lens, starts)
    T = ids.size
    hashes = torch.full((T, 1, 6), -9, dtype=torch.int64, device="cuda")
    outs = st.hash_lookup_varlen(H.to_dev(ids), H.to_dev(cu), H.to_dev(starts), Ws, Ss, mask=H.to_dev(mask),
                                 hashes=hashes, max_len=max(lens))
    exp_h, fl = orc.hash_varlen(ids, cu, starts, mask)
    assert fl == 0 and st.status() == 0
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "packed hashes")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, 0, :]), "packed rows")
    # the hash-only packed call, after a second state replays the same history
    st2 = H.make_state(wl, B, 512)
    if pre > 0:
        st2.hash(H.to_dev(full_ids[:, :pre]), 0, H.to_dev(full_mask[:, :pre]))
    h2 = st2.hash_varlen(H.to_dev(ids), H.to_dev(cu), H.to_dev(starts), mask=H.to_dev(mask))  # max_len derived
    H.assert_bits_equal(h2.cpu().numpy(), exp_h, "packed hash-only")


def test_packed_equals_dense_for_equal_lengths():
    wl = synth.make_workload(0)
    B, L = 4, 48
    rng = np.random.default_rng(3)
    ids = rng.integers(0, wl.layout.raw_vocab, size=(B, L)).astype(np.int64)
    starts = np.array([0, 2, 5, 1], dtype=np.int32)
    a, b = H.make_state(wl, B, 128), H.make_state(wl, B, 128)
    Ws, Ss = H.device_tables(wl)
    hd = torch.empty((B, L, 1, 6), dtype=torch.int64, device="cuda")
    od = a.hash_lookup(H.to_dev(ids), Ws, Ss, start_pos=H.to_dev(starts), hashes=hd)
    cu = (np.arange(B + 1) * L).astype(np.int32)
    hp = torch.empty((B * L, 1, 6), dtype=torch.int64, device="cuda")
    op = b.hash_lookup_varlen(H.to_dev(ids.reshape(-1)), H.to_dev(cu), H.to_dev(starts), Ws, Ss, hashes=hp, max_len=L)
    assert torch.equal(hd.view(-1), hp.view(-1))
    assert torch.equal(od[0].view(torch.int16).reshape(-1), op[0].view(torch.int16).reshape(-1))


def test_inconsistent_extent_is_skipped_and_flagged():
    wl = synth.make_workload(0)
    st = H.make_state(wl, 3, 64)
    Ws, Ss = H.device_tables(wl)
    ids = torch.arange(10, dtype=torch.int64, device="cuda")
    cu = torch.tensor([0, 4, 4, 12], dtype=torch.int32, device="cuda")  # sequence 2 runs past T = 10
    starts = torch.zeros(3, dtype=torch.int32, device="cuda")
    hashes = torch.full((10, 1, 6), -9, dtype=torch.int64, device="cuda")
    st.hash_lookup_varlen(ids, cu, starts, Ws, Ss, hashes=hashes, max_len=8)
    assert st.status() == geng.STATUS_BAD_LENGTH
    h = hashes.cpu().numpy()
    assert (h[:4] >= 0).all() and (h[4:] == -9).all()  # sequence 0 done, empty sequence 1, sequence 2 skipped
    # longer than max_len: skipped too
    cu = torch.tensor([0, 2, 4, 10], dtype=torch.int32, device="cuda")
    hashes.fill_(-9)
    st.hash_lookup_varlen(ids, cu, starts, Ws, Ss, hashes=hashes, max_len=4)
    assert st.status() == geng.STATUS_BAD_LENGTH
    assert (hashes.cpu().numpy()[4:] == -9).all()
    with pytest.raises(geng.EngramError) as e:
        st.hash_lookup_varlen(ids, cu, starts, Ws, Ss, max_len=65)  # max_len > max_seq_len
    assert e.value.code == geng.ERR_RANGE


def test_prepared_call_matches_the_plain_call():
    wl = synth.make_workload(0, full64=True)
    B, L = 3, 20
    rng = np.random.default_rng(11)
    ids = torch.from_numpy(rng.integers(0, wl.layout.raw_vocab, size=(B, L)).astype(np.int64)).cuda()
    start = torch.tensor([0, 3, 7], dtype=torch.int32, device="cuda")
    a, b = H.make_state(wl, B, 128), H.make_state(wl, B, 128)
    Ws, Ss = H.device_tables(wl)
    out_a = [torch.empty((B, L, 6, 32), dtype=torch.bfloat16, device="cuda")]
    out_b = [torch.empty((B, L, 6, 32), dtype=torch.bfloat16, device="cuda")]
    ha = torch.empty((B, L, 1, 6), dtype=torch.int64, device="cuda")
    hb = torch.empty_like(ha)
    call = b.prepare_hash_lookup(ids, start, Ws, Ss, out_b, hashes=hb)
    for step in range(3):  # refill the same buffers in place, as a serving loop would
        ids.copy_(torch.from_numpy(rng.integers(0, wl.layout.raw_vocab, size=(B, L)).astype(np.int64)))
        start += L
        a.hash_lookup(ids, Ws, Ss, start_pos=start, out=out_a, hashes=ha)
        call()
        torch.cuda.synchronize()
        assert (ha >= 0).all() and a.status() == 0 and b.status() == 0
        assert torch.equal(ha, hb) and torch.equal(out_a[0].view(torch.int16), out_b[0].view(torch.int16))


def test_many_short_sequences_after_unused_tokens():
    """700 packed sequences, more than a CTA has threads, so the search that maps a CTA to its sequence
    and tile takes two rounds in both kernels; most are 0-2 tokens long, their cache rows permuted, and
    the packed tokens start after 3 unused ones and end 2 before T. Every sequence's hash ids and rows
    equal the oracle's; the unused tokens' outputs are not written."""
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    B, lead, trail = 700, 3, 2
    rng = np.random.default_rng(700)
    lens = rng.choice([0, 1, 1, 1, 2, 5, 9, 33], size=B)
    starts = rng.integers(0, 60, size=B).astype(np.int32)
    rows_map = rng.permutation(B).astype(np.int32)
    cu = (lead + np.concatenate([[0], np.cumsum(lens)])).astype(np.int32)
    T = int(cu[-1]) + trail
    ids = rng.integers(0, lay.raw_vocab, size=T)
    mask = rng.random(T) > 0.1
    hist = rng.integers(0, lay.raw_vocab, size=(B, 60))
    states = []
    for _ in range(2):  # one for the fused call, one for the hash-only call, with the same history
        st = H.make_state(wl, B, 128)
        st.hash(H.to_dev(hist), 0)
        states.append(st)
    orc = H.make_oracle(wl, B, 128)
    orc.hash(hist, 0)
    Ws, Ss = H.device_tables(wl)
    d_ids, d_cu, d_st, d_mask, d_map = (H.to_dev(x) for x in (ids, cu, starts, mask, rows_map))
    hashes = torch.full((T, 1, 6), -9, dtype=torch.int64, device="cuda")
    out = [torch.full((T, 6, lay.head_dim), -7.0, dtype=torch.bfloat16, device="cuda")]
    states[0].hash_lookup_varlen(d_ids, d_cu, d_st, Ws, Ss, mask=d_mask, out=out, hashes=hashes, max_len=33,
                                 cache_rows=d_map)
    h2 = torch.full((T, 1, 6), -9, dtype=torch.int64, device="cuda")
    states[1].hash_varlen(d_ids, d_cu, d_st, mask=d_mask, hashes=h2, max_len=33, cache_rows=d_map)
    exp_h, fl = orc.hash_varlen(ids, cu, starts, mask, cache_rows=rows_map)
    assert fl == 0 and states[0].status() == 0 and states[1].status() == 0
    seq = slice(lead, T - trail)
    H.assert_bits_equal(hashes.cpu().numpy()[seq], exp_h[seq], "packed hashes")
    H.assert_bits_equal(h2.cpu().numpy()[seq], exp_h[seq], "packed hash-only")
    H.assert_bits_equal(H.bf16_bits(out[0])[seq], H.oracle_lookup_rows(wl, 0, exp_h[seq, 0, :]), "packed rows")
    for h in (hashes, h2):
        assert (h[:lead] == -9).all() and (h[T - trail:] == -9).all()
    unused = torch.cat([out[0][:lead], out[0][T - trail:]])
    assert (unused == -7.0).all()


def test_decreasing_extents_are_flagged():
    """Where cu_seqlens decreases, the sequence at the decrease is flagged; which other sequences run
    is unspecified, but the kernels read cu_seqlens only at indices 0..B (the search picks indices,
    never follows values) and both packed kernels return normally."""
    wl = synth.make_workload(0)
    Ws, Ss = H.device_tables(wl)
    ids = torch.arange(10, dtype=torch.int64, device="cuda")
    starts = torch.zeros(3, dtype=torch.int32, device="cuda")
    for cu_list in ([0, 8, 3, 10], [5, 2, 9, 10]):
        st = H.make_state(wl, 3, 64)
        cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
        hashes = torch.full((10, 1, 6), -9, dtype=torch.int64, device="cuda")
        st.hash_lookup_varlen(ids, cu, starts, Ws, Ss, hashes=hashes, max_len=10)
        st.hash_varlen(ids, cu, starts, hashes=hashes, max_len=10)
        torch.cuda.synchronize()
        assert st.status() & geng.STATUS_BAD_LENGTH


@pytest.mark.parametrize("seed", range(6))
def test_random_packed_batches_of_many_sequences(seed):
    """90 to 1,200 packed sequences of 0 to 64 tokens (one or two search rounds in the fused kernel's
    256-thread CTAs, two in the hash-only kernel's 96-thread CTAs), unused tokens around them, cache
    rows permuted: hash ids and rows equal the oracle's."""
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    rng = np.random.default_rng(9000 + seed)
    B = int(rng.integers(90, 1200))
    lens = rng.choice([0, 1, 1, 2, 3, 7, 16, 31, 64], size=B)
    starts = rng.integers(0, 40, size=B).astype(np.int32)
    rows_map = rng.permutation(B).astype(np.int32)
    cu = (int(rng.integers(0, 5)) + np.concatenate([[0], np.cumsum(lens)])).astype(np.int32)
    T = int(cu[-1]) + int(rng.integers(0, 5))
    ids = rng.integers(0, lay.raw_vocab, size=T)
    mask = rng.random(T) > 0.1
    hist = rng.integers(0, lay.raw_vocab, size=(B, 40))
    st, st2, orc = H.make_state(wl, B, 128), H.make_state(wl, B, 128), H.make_oracle(wl, B, 128)
    st.hash(H.to_dev(hist), 0)
    st2.hash(H.to_dev(hist), 0)
    orc.hash(hist, 0)
    Ws, Ss = H.device_tables(wl)
    d_ids, d_cu, d_st, d_mask, d_map = (H.to_dev(x) for x in (ids, cu, starts, mask, rows_map))
    hashes = torch.full((T, 1, 6), -9, dtype=torch.int64, device="cuda")
    outs = st.hash_lookup_varlen(d_ids, d_cu, d_st, Ws, Ss, mask=d_mask, hashes=hashes, max_len=64, cache_rows=d_map)
    h2 = st2.hash_varlen(d_ids, d_cu, d_st, mask=d_mask, max_len=64, cache_rows=d_map)
    exp_h, fl = orc.hash_varlen(ids, cu, starts, mask, cache_rows=rows_map)
    assert fl == 0 and st.status() == 0 and st2.status() == 0
    seq = slice(int(cu[0]), int(cu[-1]))
    H.assert_bits_equal(hashes.cpu().numpy()[seq], exp_h[seq], "packed hashes")
    H.assert_bits_equal(h2.cpu().numpy()[seq], exp_h[seq], "packed hash-only")
    H.assert_bits_equal(H.bf16_bits(outs[0])[seq], H.oracle_lookup_rows(wl, 0, exp_h[seq, 0, :]), "packed rows")
