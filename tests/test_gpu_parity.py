"""CUDA path vs the CPU oracle, bit for bit, through the C ABI (GPU only).

Hash ids are integers: bit-exact. Looked-up rows are one fp32 round-to-nearest
multiply then round-to-nearest-even to bf16 on both sides: bit-exact (0 ulp).
The seeded tables never hold the NaN codes, so no NaN payload is compared;
the all-codes test compares NaN positions only.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


# ----------------------------------------------------------------------------- lookup alone
@pytest.mark.parametrize("D,block", [(16, 16), (32, 32), (64, 16), (128, 128), (128, 32), (256, 128), (512, 256)])
@pytest.mark.parametrize("n_idx", [1, 7, 1000, 4099])
def test_lookup_all_codes(D, block, n_idx):
    rng = np.random.default_rng(D * 7 + n_idx)
    nsc = D // block
    rows = max(256 // D, 1) + 61
    W = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
    W.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)  # every code, NaN codes included
    S = rng.uniform(0.01, 1.0, size=(rows, nsc)).astype(np.float32)
    S[0, 0], S[1, -1], S[2, 0], S[3, 0] = 1e-40, 3.0e38, 2.0 ** -130, -0.75
    idx = rng.integers(-3, rows + 3, size=n_idx).astype(np.int64)
    idx[: min(n_idx, 4)] = np.arange(min(n_idx, 4))
    if n_idx > 10:
        idx[-1], idx[-2] = -(2 ** 62), 2 ** 62
    exp = oracle.engram_lookup(idx, W, S, rows, D, block)
    out = geng.engram_lookup(H.to_dev(idx), H.to_dev(W), H.to_dev(S), block)
    torch.cuda.synchronize()
    got = H.bf16_bits(out)
    nan_e = ((exp & 0x7F80) == 0x7F80) & ((exp & 0x7F) != 0)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_e, nan_g)
    H.assert_bits_equal(np.where(nan_e, 0, got), np.where(nan_e, 0, exp), f"lookup D={D} block={block}")


def test_lookup_empty_and_errors():
    W = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    S = torch.ones((4, 1), dtype=torch.float32, device="cuda")
    idx = torch.zeros((0,), dtype=torch.int64, device="cuda")
    out = geng.engram_lookup(idx, W, S, 128)
    assert out.shape == (0, 128)
    with pytest.raises(geng.EngramError) as e:
        geng.engram_lookup(torch.zeros(3, dtype=torch.int64, device="cuda"), W[:, :48].contiguous(), S, 48)
    assert e.value.code == geng.ERR_UNSUPPORTED
    # misaligned output pointer
    big = torch.empty((3 * 128 + 8,), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(geng.EngramError) as e:
        geng.engram_lookup(torch.zeros(3, dtype=torch.int64, device="cuda"), W, S, 128, out=big[1:1 + 3 * 128].view(3, 128))
    assert e.value.code == geng.ERR_INVALID


# ----------------------------------------------------------------------------- tiny configuration
@pytest.mark.parametrize("full64", [False, True])
def test_tiny_hash_and_lookup(full64):
    wl = synth.make_workload(0, full64=full64)
    st, orc = H.make_state(wl), H.make_oracle(wl)
    Ws, Ss = H.device_tables(wl)
    ids = H.to_dev(wl.ids)
    hashes = torch.empty((1, 64, 1, 6), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(ids, Ws, Ss, start_pos=0, hashes=hashes)
    exp_h, _ = orc.hash(wl.ids, 0)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "tiny hashes")
    exp_rows = H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :])
    H.assert_bits_equal(H.bf16_bits(outs[0]), exp_rows, "tiny rows")
    # hash-only entry point, fresh cache
    st.reset()
    h2 = st.hash(ids, 0)
    H.assert_bits_equal(h2.cpu().numpy(), exp_h, "tiny hash-only")
    # the full tiny table on the host: oracle on the real table, not a compact one
    Wh = Ws[0].cpu().numpy()
    Sh = Ss[0].cpu().numpy()
    H.assert_bits_equal(oracle.engram_lookup(exp_h[:, :, 0, :], Wh, Sh, Wh.shape[0], 32, 32), exp_rows, "compact table")
    assert st.status() == 0


def test_device_fill_matches_host_generator():
    wl = synth.make_workload(0)
    Ws, Ss = H.device_tables(wl)
    rows = wl.layout.rows[0]
    H.assert_bits_equal(Ws[0].cpu().numpy(), synth.table_rows(wl.table_seed, 0, np.arange(rows), 32), "fp8 fill")
    H.assert_bits_equal(Ss[0].cpu().numpy().view(np.uint32),
                        synth.table_scales(wl.table_seed, 0, np.arange(rows), 1).view(np.uint32), "scale fill")


# ----------------------------------------------------------------------------- ragged tiles, chunks, starts
@pytest.mark.parametrize("L", [1, 2, 3, 15, 16, 17, 63, 64, 65, 1000])
def test_ragged_lengths_and_row_starts(L):
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    B, T = 3, 1200
    ids = synth.uniform_int(L, synth.TAG_IDS, B * T, 0, lay.raw_vocab).reshape(B, T)
    mask = synth.uniform_int(L + 1, synth.TAG_IDS, B * T, 0, 6).reshape(B, T) > 0
    st, orc = H.make_state(wl, B, 4096), H.make_oracle(wl, B, 4096)
    Ws, Ss = H.device_tables(wl)
    starts = np.array([0, 5, 2], dtype=np.int32)
    # history first (prefill each row up to its start), then an L-token call at per-row starts
    pre = ids[:, :8]
    st.hash(H.to_dev(pre), 0, H.to_dev(mask[:, :8]))
    orc.hash(pre, 0, mask[:, :8])
    chunk = np.stack([ids[b, starts[b]:starts[b] + L] for b in range(B)])
    cmask = np.stack([mask[b, starts[b]:starts[b] + L] for b in range(B)])
    hashes = torch.empty((B, L, 1, 6), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(chunk), Ws, Ss, start_pos=H.to_dev(starts), mask=H.to_dev(cmask), hashes=hashes)
    exp_h, _ = orc.hash(chunk, starts.astype(np.int64), cmask)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, f"hashes L={L}")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), f"rows L={L}")


def test_bad_start_and_bad_ids_are_flagged_not_faulted():
    wl = synth.make_workload(0)
    st, orc = H.make_state(wl, 2, 64), H.make_oracle(wl, 2, 64)
    Ws, Ss = H.device_tables(wl)
    ids = np.array([[1, 2, 3, 4], [5, -7, 999, 1000]], dtype=np.int64)
    starts = np.array([62, 0], dtype=np.int32)  # row 0: 62 + 4 > 64
    hashes = torch.empty((2, 4, 1, 6), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(ids), Ws, Ss, start_pos=H.to_dev(starts), hashes=hashes)
    flags = st.status()
    assert flags == geng.STATUS_BAD_START | geng.STATUS_BAD_ID
    exp_h, eflags = orc.hash(ids, starts.astype(np.int64))
    assert eflags == flags
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "flagged hashes")
    assert (exp_h[0] == -1).all()
    assert (H.bf16_bits(outs[0])[0] == 0).all()
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), "flagged rows")
    assert st.status() == 0  # cleared


def test_argument_errors():
    wl = synth.make_workload(0)
    st = H.make_state(wl, 2, 64)
    ids = torch.zeros((3, 4), dtype=torch.int64, device="cuda")
    with pytest.raises(geng.EngramError) as e:
        st.hash(ids, 0)  # B > max_batch
    assert e.value.code == geng.ERR_RANGE
    with pytest.raises(geng.EngramError) as e:
        st.hash(torch.zeros((1, 65), dtype=torch.int64, device="cuda"), 0)  # L > max_seq_len
    assert e.value.code == geng.ERR_RANGE
    # empty calls are no-ops
    assert st.hash(torch.zeros((0, 4), dtype=torch.int64, device="cuda"), 0).shape == (0, 4, 1, 6)
    assert st.hash(torch.zeros((2, 0), dtype=torch.int64, device="cuda"), 0).shape == (2, 0, 1, 6)
    with pytest.raises(geng.EngramError) as e:
        geng.engram_state_create(n_layers=1, max_ngram=4, n_heads=2, head_dim=32, block=32, max_batch=1,
                                 max_seq_len=8, token_map=[0, 1], multipliers=[1, 1, 1, 1], primes=[0] * 6,
                                 offsets=[0] * 6)
    assert e.value.code == geng.ERR_INVALID  # prime 0


# ----------------------------------------------------------------------------- prefill configuration
@pytest.fixture(scope="module")
def prefill_tables():
    wl = synth.make_workload(1)
    Ws, Ss = H.device_tables(wl)
    yield wl, Ws, Ss
    del Ws, Ss
    torch.cuda.empty_cache()


@pytest.mark.parametrize("full64", [False, True])
def test_prefill_with_image_spans(prefill_tables, full64):
    wl1, Ws, Ss = prefill_tables
    wl = synth.make_workload(1, full64=full64) if full64 else wl1
    st, orc = H.make_state(wl), H.make_oracle(wl)
    hashes = torch.empty((wl.B, wl.L, 2, 24), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, mask=H.to_dev(wl.mask), hashes=hashes)
    exp_h, fl = orc.hash(wl.ids, 0, wl.mask)
    assert fl == 0 and st.status() == 0
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "prefill hashes")
    for l in range(2):
        H.assert_bits_equal(H.bf16_bits(outs[l]), H.oracle_lookup_rows(wl1, l, exp_h[:, :, l, :]), f"prefill rows l{l}")


def test_decode_per_row_start(prefill_tables):
    _, Ws, Ss = prefill_tables
    wl = synth.make_workload(2)
    st, orc = H.make_state(wl), H.make_oracle(wl)
    # prefill every row with 8192 Zipf tokens, then one decode step at each row's own start
    h_pre = st.hash(H.to_dev(wl.prefill_ids), 0)
    e_pre, _ = orc.hash(wl.prefill_ids, 0)
    H.assert_bits_equal(h_pre.cpu().numpy(), e_pre, "decode prefill hashes")
    hashes = torch.empty((wl.B, 1, 2, 24), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=H.to_dev(wl.start_pos), hashes=hashes)
    exp_h, _ = orc.hash(wl.ids, wl.start_pos.astype(np.int64))
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "decode hashes")
    for l in range(2):
        H.assert_bits_equal(H.bf16_bits(outs[l]), H.oracle_lookup_rows(wl, l, exp_h[:, :, l, :]), f"decode rows l{l}")
    # a decode step equals the same row prefilled in one shot through its new token
    b = int(np.argmax(wl.start_pos))
    s = int(wl.start_pos[b])
    one = H.make_state(wl, 1, wl.max_seq_len)
    seq = np.concatenate([wl.prefill_ids[b, :s], wl.ids[b]])[None]
    h_one = one.hash(H.to_dev(seq), 0)
    assert (h_one[0, -1] == hashes[b, 0]).all()


# ----------------------------------------------------------------------------- both fused paths
def _custom_layout(seed, n_layers, max_ngram, n_heads, D, block, primes=None, vocab=300, cvocab=50):
    if primes is None:
        primes = synth.distinct_primes_in(seed, 997, 2003, (n_layers, max_ngram - 1, n_heads))
    primes = np.asarray(primes, dtype=np.int64).reshape(n_layers, max_ngram - 1, n_heads)
    return synth.Layout(n_layers, max_ngram, n_heads, D, block, vocab, cvocab,
                        synth.uniform_int(seed, synth.TAG_TOKEN_MAP, vocab, 0, cvocab),
                        synth.multipliers(seed, n_layers, max_ngram, full64=True), primes,
                        synth.column_offsets(primes))


def _run_fused_vs_oracle(lay, B, L, rows_override=None, seed=0, with_mask=True):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, lay.raw_vocab, size=(B, L)).astype(np.int64)
    mask = (rng.random((B, L)) > 0.1) if with_mask else None
    st = geng.EngramHash(n_layers=lay.n_layers, max_ngram=lay.max_ngram, n_heads=lay.n_heads, head_dim=lay.head_dim,
                         block=lay.block, max_batch=B, max_seq_len=L, token_map=lay.token_map,
                         multipliers=lay.multipliers, primes=lay.primes, offsets=lay.offsets)
    orc = oracle.OracleState.from_layout(lay, B, L)
    Wh, Sh, Wd, Sd = [], [], [], []
    for l in range(lay.n_layers):
        rows = lay.rows[l] if rows_override is None else rows_override[l]
        W = rng.integers(0, 256, size=(rows, lay.head_dim), dtype=np.uint8)
        W[W == 0x7F] = 0x7E
        W[W == 0xFF] = 0xFE
        S = rng.uniform(0.01, 2.0, size=(rows, lay.head_dim // lay.block)).astype(np.float32)
        Wh.append(W); Sh.append(S); Wd.append(H.to_dev(W)); Sd.append(H.to_dev(S))
    hashes = torch.empty((B, L, lay.n_layers, lay.n_cols), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(ids), Wd, Sd, start_pos=0, mask=None if mask is None else H.to_dev(mask),
                          hashes=hashes)
    exp_h, _ = orc.hash(ids, 0, mask)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "fused hashes")
    for l in range(lay.n_layers):
        exp = oracle.engram_lookup(exp_h[:, :, l, :], Wh[l], Sh[l], Wh[l].shape[0], lay.head_dim, lay.block)
        H.assert_bits_equal(H.bf16_bits(outs[l]), exp, f"fused rows layer {l}")
    assert st.status() == 0


@pytest.mark.parametrize("D,block", [(16, 16), (32, 32), (64, 16), (128, 128), (128, 64), (128, 32), (256, 128),
                                     (512, 128), (512, 64), (128, 8), (256, 16)])
@pytest.mark.parametrize("L", [1, 33, 100])
def test_fused_paths_all_shapes(D, block, L):
    """Every head_dim / block pair the library accepts: a row with one scale block (block == D) takes
    the kernel instantiation that loads one scale per lane; rows with 2 to 64 scale blocks take the one
    that loads the scale of each 8-code half of the lane's 16 codes. Tokens per row 1, 33 and 100 give one
    partial tile, several tiles with a ragged tail, and many tiles."""
    lay = _custom_layout(D + block, 2, 4, 3, D, block)
    _run_fused_vs_oracle(lay, 3, L, seed=D * 1000 + block + L)


@pytest.mark.parametrize("D,block", [(128, 128), (256, 128), (64, 16), (512, 64)])
def test_fused_small_tables_edge_rows(D, block):
    """Bucket ranges of 5 and 7 rows: every row is hit, including the table's last rows and their
    last scales (a read one past them would leave the arrays); passing tables with fewer rows than
    the hash range makes the top hash ids out of range (+0 rows), down to a one-row table."""
    lay = _custom_layout(3, 1, 2, 2, D, block, primes=[[[5, 7]]])
    assert lay.rows == [12]
    _run_fused_vs_oracle(lay, 2, 200, seed=D)
    _run_fused_vs_oracle(lay, 2, 200, rows_override=[9], seed=D + 1)
    _run_fused_vs_oracle(lay, 2, 200, rows_override=[1], seed=D + 2, with_mask=False)


def test_fused_call_replays_from_a_cuda_graph():
    """The fused call allocates nothing and never synchronises, so it can be captured once and
    replayed; the replay recomputes the same cache writes, hash ids and rows."""
    wl = synth.make_workload(0, full64=True)
    st, orc = H.make_state(wl), H.make_oracle(wl)
    Ws, Ss = H.device_tables(wl)
    ids = H.to_dev(wl.ids)
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    hashes = torch.full((1, 64, 1, 6), -7, dtype=torch.int64, device="cuda")
    outs = [torch.zeros((1, 64, 6, 32), dtype=torch.bfloat16, device="cuda")]
    st.hash_lookup(ids, Ws, Ss, start_pos=start, out=outs, hashes=hashes)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.hash_lookup(ids, Ws, Ss, start_pos=start, out=outs, hashes=hashes)
    hashes.fill_(-7)
    outs[0].zero_()
    st.reset()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    exp_h, _ = orc.hash(wl.ids, 0)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "graph hashes")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), "graph rows")


def test_layout_at_the_library_limits():
    """8 layers, n-gram size 8, 9 heads: 504 hash columns per token (limit 512). At 1,216 tiles the
    fused kernel keeps 8-token tiles, and its shared memory (column constants 16 KB, rolling values
    3.5 KB, row ids 31.5 KB) exceeds 48 KB and is requested explicitly; the hash-only kernel stays
    below it."""
    n_layers, max_ngram, n_heads = 8, 8, 9
    primes = synth.distinct_primes_in(77, 2, 4000, (n_layers, max_ngram - 1, n_heads))
    lay = synth.Layout(n_layers, max_ngram, n_heads, 32, 32, 500, 90, synth.uniform_int(77, synth.TAG_TOKEN_MAP, 500, 0, 90),
                       synth.multipliers(77, n_layers, max_ngram, full64=True), primes, synth.column_offsets(primes))
    assert n_layers * lay.n_cols == 504
    rng = np.random.default_rng(77)
    B, L = 2, 608 * 8
    ids = rng.integers(0, 500, size=(B, L)).astype(np.int64)
    mask = rng.random((B, L)) > 0.1
    st = geng.EngramHash(n_layers=n_layers, max_ngram=max_ngram, n_heads=n_heads, head_dim=32, block=32,
                         max_batch=B, max_seq_len=L, token_map=lay.token_map, multipliers=lay.multipliers,
                         primes=lay.primes, offsets=lay.offsets)
    orc = oracle.OracleState.from_layout(lay, B, L)
    Wh = [rng.integers(0, 0x7E, size=(r, 32), dtype=np.uint8) for r in lay.rows]
    Sh = [rng.uniform(0.1, 1.0, size=(r, 1)).astype(np.float32) for r in lay.rows]
    hashes = torch.empty((B, L, n_layers, lay.n_cols), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(ids), [H.to_dev(w) for w in Wh], [H.to_dev(x) for x in Sh], start_pos=0,
                          mask=H.to_dev(mask), hashes=hashes)
    exp_h, _ = orc.hash(ids, 0, mask)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "limit-layout hashes")
    for l in range(n_layers):
        exp = oracle.engram_lookup(exp_h[:, :, l, :], Wh[l], Sh[l], lay.rows[l], 32, 32)
        H.assert_bits_equal(H.bf16_bits(outs[l]), exp, f"limit-layout rows layer {l}")
    st.reset()
    H.assert_bits_equal(st.hash(H.to_dev(ids), 0, H.to_dev(mask)).cpu().numpy(), exp_h, "limit-layout hash-only")
    with pytest.raises(geng.EngramError) as e:  # one more head: 8 x 7 x 10 = 560 columns
        geng.engram_state_create(n_layers=8, max_ngram=8, n_heads=10, head_dim=32, block=32, max_batch=1,
                                 max_seq_len=8, token_map=[0], multipliers=[1] * 64, primes=[3] * 560,
                                 offsets=[0] * 560)
    assert e.value.code == geng.ERR_UNSUPPORTED


def test_hash_moduli_at_the_extremes():
    """The floored mod on the GPU (multiply-high by floor((2^64-1)/P), one correction, 2^64 mod P
    for negative running values) against the oracle's plain int64 `%` for moduli 1, 2, 3, near
    2^31, near 2^62 (the limit) and offsets near the int64 limit, with full 64-bit multipliers so the
    running values cover both signs."""
    moduli = np.array([[[1, 2, 3], [2 ** 31 - 1, 2 ** 31 + 11, 2 ** 40 + 15]],
                       [[2 ** 62 - 1, 2 ** 62 - 57, 2 ** 61 + 1], [97, 2 ** 62 - 3, 5]]], dtype=np.int64)
    offsets = np.zeros((2, 6), dtype=np.int64)
    offsets[0, 1] = 2 ** 63 - 2          # + (P-1) = 1 -> fits exactly
    offsets[1, 0] = -(2 ** 62)
    offsets[1, 5] = 12345
    lay = synth.Layout(2, 3, 3, 16, 16, 256, 200, synth.uniform_int(9, synth.TAG_TOKEN_MAP, 256, 0, 200),
                       synth.multipliers(9, 2, 3, full64=True), moduli, offsets)
    rng = np.random.default_rng(9)
    B, L = 4, 300
    ids = rng.integers(0, 256, size=(B, L)).astype(np.int64)
    st = geng.EngramHash(n_layers=2, max_ngram=3, n_heads=3, head_dim=16, block=16, max_batch=B, max_seq_len=L,
                         token_map=lay.token_map, multipliers=lay.multipliers, primes=lay.primes, offsets=offsets)
    orc = oracle.OracleState.from_layout(lay, B, L)
    got = st.hash(H.to_dev(ids), 0).cpu().numpy()
    exp, _ = orc.hash(ids, 0)
    H.assert_bits_equal(got, exp, "extreme moduli")
    assert (got[:, :, 0, 0] == 0).all()  # modulus 1
    assert len(np.unique(got[:, :, 1, 1])) > 100  # a modulus near 2^62 spreads the ids
    with pytest.raises(geng.EngramError) as e:  # offset + P - 1 past int64
        bad = offsets.copy()
        bad[0, 1] = 2 ** 63 - 1
        geng.engram_state_create(n_layers=2, max_ngram=3, n_heads=3, head_dim=16, block=16, max_batch=1,
                                 max_seq_len=8, token_map=lay.token_map, multipliers=lay.multipliers,
                                 primes=lay.primes, offsets=bad)
    assert e.value.code == geng.ERR_INVALID


def test_batch_at_the_grid_limit():
    """max_batch 65,535 (the largest the library takes; one grid row per sequence, CUDA's
    gridDim.y limit): a dense call over every row, some rows starting exactly at max_seq_len - L,
    some with every token masked, and a packed call over all 65,535 sequences, against the oracle."""
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    B, L, max_seq = 65535, 3, 8
    rng = np.random.default_rng(65535)
    ids = rng.integers(0, lay.raw_vocab, size=(B, L))
    start = rng.integers(0, max_seq - L + 1, size=B).astype(np.int32)
    start[::7] = max_seq - L                       # the last position that fits
    mask = rng.random((B, L)) > 0.1
    mask[::11] = False                             # whole rows masked
    Ws, Ss = H.device_tables(wl)
    st, orc = H.make_state(wl, B, max_seq), H.make_oracle(wl, B, max_seq)
    hashes = torch.empty((B, L, 1, lay.n_cols), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(ids), Ws, Ss, start_pos=H.to_dev(start), mask=H.to_dev(mask), hashes=hashes)
    exp_h, fl = orc.hash(ids, start.astype(np.int64), mask)
    assert fl == 0 and st.status() == 0
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "hashes at B=65535")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), "rows at B=65535")
    # packed: every sequence one token long, at the next position
    cu = np.arange(B + 1, dtype=np.int32)
    ids2 = rng.integers(0, lay.raw_vocab, size=B)
    st2 = start + L
    st2[st2 >= max_seq] = max_seq - 1
    exp2, _ = orc.hash_varlen(ids2, cu, st2, None)
    got2 = st.hash_varlen(H.to_dev(ids2), H.to_dev(cu), H.to_dev(st2), max_len=1)
    H.assert_bits_equal(got2.cpu().numpy(), exp2, "packed hashes at B=65535")
    with pytest.raises(geng.EngramError) as e:
        geng.engram_state_create(n_layers=1, max_ngram=4, n_heads=2, head_dim=32, block=32, max_batch=65536,
                                 max_seq_len=8, token_map=lay.token_map, multipliers=lay.multipliers,
                                 primes=lay.primes, offsets=lay.offsets)
    assert e.value.code == geng.ERR_UNSUPPORTED


def test_binding_refuses_wrong_sizes():
    """One table per engram layer and buffers of the call's sizes, or a ValueError before anything
    is launched (the C calls take raw pointers)."""
    base = synth.make_workload(0, full64=True)
    lay = dataclasses.replace(base.layout, n_layers=2, multipliers=np.concatenate([base.layout.multipliers] * 2),
                              primes=np.concatenate([base.layout.primes] * 2),
                              offsets=np.concatenate([base.layout.offsets] * 2))
    wl = dataclasses.replace(base, layout=lay)
    Ws, Ss = H.device_tables(wl)
    st = H.make_state(wl, 2, 64)
    ids = H.to_dev(np.zeros((2, 8), dtype=np.int64))
    C, D = lay.n_cols, lay.head_dim
    with pytest.raises(ValueError, match="one entry per engram layer"):
        st.hash_lookup(ids, Ws[:1], Ss[:1])
    with pytest.raises(ValueError, match="out"):
        st.hash_lookup(ids, Ws, Ss, out=[torch.empty((2, 8, C, D), dtype=torch.bfloat16, device="cuda"),
                                         torch.empty((2, 7, C, D), dtype=torch.bfloat16, device="cuda")])
    with pytest.raises(ValueError, match="hashes"):
        st.hash_lookup(ids, Ws, Ss, hashes=torch.empty((2, 8, 1, C), dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError, match="mask"):
        st.hash(ids, 0, mask=torch.ones((2, 7), dtype=torch.bool, device="cuda"))
    with pytest.raises(ValueError, match="S\\[1\\]"):
        st.hash_lookup(ids, Ws, [Ss[0], Ss[1][:-1]])
    out = [torch.empty((2, 8, C, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(ValueError, match="start_pos"):
        st.prepare_hash_lookup(ids, torch.zeros(3, dtype=torch.int32, device="cuda"), Ws, Ss, out)
    torch.cuda.synchronize()
    assert st.status() == 0


def test_outputs_only_16_byte_aligned():
    """A lane writes its 32 bytes of a row with one 256-bit store when the output is 32-byte aligned,
    else with two 16-byte stores: outputs that start 16 bytes into their buffer get the same bits,
    from the fused call and from the lookup."""
    wl = synth.make_workload(0)
    lay = wl.layout
    Ws, Ss = H.device_tables(wl)
    ids = H.to_dev(np.random.default_rng(5).integers(0, lay.raw_vocab, size=(1, 64)))
    st, st2 = H.make_state(wl, 1, 64), H.make_state(wl, 1, 64)
    hashes = torch.empty((1, 64, 1, 6), dtype=torch.int64, device="cuda")
    ref = st.hash_lookup(ids, Ws, Ss, hashes=hashes)
    buf = torch.full((ref[0].numel() + 8,), -3.0, dtype=torch.bfloat16, device="cuda")
    out = [buf[8:].view(ref[0].shape)]
    assert out[0].data_ptr() % 32 == 16
    st2.hash_lookup(ids, Ws, Ss, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out[0].view(torch.int16), ref[0].view(torch.int16))
    assert (buf[:8] == -3.0).all()
    idx = hashes[..., 0, :].reshape(-1).contiguous()
    r1 = st.lookup(idx, Ws[0], Ss[0])
    buf2 = torch.empty((r1.numel() + 8,), dtype=torch.bfloat16, device="cuda")
    o2 = buf2[8:].view(r1.shape)
    st.lookup(idx, Ws[0], Ss[0], out=o2)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), r1.view(torch.int16))
