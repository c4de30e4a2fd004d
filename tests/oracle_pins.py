"""Pins for the CPU oracle: each function checks the oracle (given as a bound
library, so planted-mistake builds can be checked too) against something other
than itself, and raises AssertionError on the first mismatch.

What pins what:
  - floored mod            <- Python's floored ``%`` on big integers
  - fp8 E4M3 decode        <- hand values of the E4M3 definition + torch's float8_e4m3fn cast
  - bf16 rounding          <- torch's float32 -> bfloat16 conversion (RNE)
  - lookup                 <- the same library calls the engram-first/lookup page makes
                              (F.embedding, .float(), block multiply, .to(bfloat16), masked_fill),
                              run on torch CPU, with fp32, bf16, UE8M0 and E4M3 scale tensors,
                              plus hand values of each scale format
  - n-gram hash            <- big-integer brute force from explicit n-gram tuples (tests/brute.py),
                              closed forms for one-hot multipliers, and invariants
                              (bucket range, chunked == one-shot, locality, masked == all-pad)
  - cache-row map          <- the same brute force on sequences that change call rows between calls
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from tests import brute

# ----------------------------------------------------------------------------- scalars


def pin_floor_mod(L=None):
    rng = np.random.default_rng(7)
    xs = [0, 1, -1, 2 ** 63 - 1, -(2 ** 63), 123456789, -123456789, -7]
    xs += [int(v) for v in rng.integers(-(2 ** 63), 2 ** 63 - 1, size=400, dtype=np.int64)]
    ps = [1, 2, 3, 5, 997, 2003, 1_000_003, 16_000_057, 2 ** 31 - 1]
    for x in xs:
        for p in ps:
            got = oracle.floor_mod(x, p, L)
            assert got == x % p, (x, p, got, x % p)


def pin_fp8_decode(L=None):
    import torch

    # hand values from the E4M3 definition (bias 7, 3 mantissa bits, exponent 0 subnormal)
    hand = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9,
            0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0xB8: -1.0, 0x30: 0.5, 0x77: 240.0}
    for code, val in hand.items():
        assert oracle.fp8_e4m3_to_f32(code, L) == val, (hex(code), val)
    assert np.signbit(oracle.fp8_e4m3_to_f32(0x80, L)) and oracle.fp8_e4m3_to_f32(0x80, L) == 0.0
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for code in range(256):
        got = np.float32(oracle.fp8_e4m3_to_f32(code, L))
        if np.isnan(ref[code]):
            assert np.isnan(got), hex(code)
        else:
            assert got.view(np.uint32) == ref[code].view(np.uint32), (hex(code), got, ref[code])


def _bf16_torch(x: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_bf16(L=None):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x3F808000, 0x3F818000, 0x3F808001, 0x3F80FFFF, 0x7F7FFFFF,
                        0x7F7F8000, 0x7F7F7FFF, 0x7F800000, 0xFF800000, 0x00000001, 0x00008000, 0x00018000,
                        0x0000FFFF, 0x807F8000, 0x007FFFFF], dtype=np.uint32)
    bits = np.concatenate([special, bits])
    x = bits.view(np.float32)
    ref = _bf16_torch(x)
    for xi, r in zip(x, ref):
        got = oracle.bf16_rne(float(xi), L)
        if np.isnan(xi):
            assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0
        else:
            assert got == r, (hex(np.float32(xi).view(np.uint32)), hex(got), hex(r))


# ----------------------------------------------------------------------------- lookup


def torch_lookup(idx: np.ndarray, W: np.ndarray, S: np.ndarray, D: int, block: int,
                 scale_dtype: int = oracle.SCALE_F32) -> np.ndarray:
    """The engram-first/lookup page's `ParallelEngramEmbedding.forward` at world size 1,
    executed with the same torch library calls on the CPU, with the scale tensor stored as
    `scale_dtype` (float32 values, or the bits of bf16 / UE8M0 / E4M3). Returns bf16 bits."""
    import torch
    import torch.nn.functional as F

    rows = W.shape[0]
    indices = torch.from_numpy(idx.astype(np.int64))
    weight = torch.from_numpy(W.copy()).view(torch.float8_e4m3fn)
    as_dtype = {oracle.SCALE_F32: torch.float32, oracle.SCALE_BF16: torch.bfloat16,
                oracle.SCALE_E8M0: torch.float8_e8m0fnu, oracle.SCALE_E4M3: torch.float8_e4m3fn}[scale_dtype]
    scale = torch.from_numpy(S.copy()).view(as_dtype)
    mask = (indices < 0) | (indices >= rows)
    local = indices.masked_fill(mask, 0)
    values = F.embedding(local, weight)
    scales = F.embedding(local, scale)
    values = values.float().unflatten(-1, (-1, block)) * scales.float().unsqueeze(-1)
    values = values.flatten(-2).to(torch.bfloat16)
    values = values.masked_fill(mask.unsqueeze(-1), 0)
    return values.view(torch.int16).numpy().view(np.uint16)


def _cmp_bf16(got: np.ndarray, ref: np.ndarray):
    g, r = got.reshape(-1), ref.reshape(-1)
    nan_g = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
    nan_r = ((r & 0x7F80) == 0x7F80) & ((r & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_r), "NaN positions differ"
    ok = nan_g | (g == r)
    if not ok.all():
        i = int(np.argmin(ok))
        raise AssertionError(f"bf16 mismatch at {i}: {hex(g[i])} vs {hex(r[i])} ({int((~ok).sum())} total)")


def pin_lookup_vs_torch(L=None):
    rng = np.random.default_rng(3)
    for D, block in ((32, 32), (128, 128), (256, 128), (64, 16)):
        nsc = D // block
        rows = 256 // D * 8 + 40
        W = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
        W[: 256 // D].reshape(-1)[:] = np.arange(256, dtype=np.uint8)  # every code, NaNs included
        S = rng.uniform(0.01, 1.0, size=(rows, nsc)).astype(np.float32)
        S[0, 0] = 1e-40          # subnormal scale
        S[1 % rows, -1] = 3.0e38  # overflow to inf for big codes
        S[2 % rows, 0] = 2.0 ** -130
        S[3 % rows, 0] = -0.75    # negative scale
        idx = np.concatenate([np.arange(rows), rng.integers(-5, rows + 5, size=300), [-1, rows, -(2 ** 62), 2 ** 62]])
        got = oracle.engram_lookup(idx, W, S, rows, D, block, L)
        ref = torch_lookup(idx, W, S, D, block)
        _cmp_bf16(got, ref)
    # hand check: code 0x38 (1.0) times 0.5 is 0.5 = bf16 0x3F00; 0x7E (448) times 1.0 = 0x43E0
    W = np.array([[0x38] * 16, [0x7E] * 16], dtype=np.uint8)
    S = np.array([[0.5], [1.0]], dtype=np.float32)
    out = oracle.engram_lookup(np.array([0, 1, 2]), W, S, 2, 16, 16, L)
    assert (out[0] == 0x3F00).all() and (out[1] == 0x43E0).all() and (out[2] == 0).all()


def pin_scale_dtypes(L=None):
    """The other scale storage types widen exactly to fp32 (`.float()`) before the one fp32
    multiply: every bf16 pattern class, all 256 UE8M0 and E4M3 codes, against the same torch
    library calls, plus hand values of each format's definition."""
    rng = np.random.default_rng(8)
    # every UE8M0 exponent; every E4M3 scale code; bf16: normal, subnormal, zero, inf, NaN patterns
    e8 = np.arange(256, dtype=np.uint8)
    bf = np.concatenate([rng.integers(0, 1 << 16, size=250), [0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80,
                                                              0x7FC0, 0x3F80]]).astype(np.uint16)
    for dtype, codes in ((oracle.SCALE_E8M0, e8), (oracle.SCALE_E4M3, e8), (oracle.SCALE_BF16, bf)):
        for D, block in ((32, 32), (64, 16)):
            nsc = D // block
            rows = -(-codes.size // nsc)
            S = np.resize(codes, rows * nsc).reshape(rows, nsc)
            W = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
            W[0, :16] = [0x00, 0x80, 0x01, 0x81, 0x08, 0x38, 0x7E, 0xFE, 0x7F, 0xFF, 0x30, 0x40, 0x77, 0x06, 0x3F, 0x47]
            idx = np.concatenate([np.arange(rows), rng.integers(-3, rows + 3, size=100)])
            got = oracle.engram_lookup(idx, W, S, rows, D, block, L, scale_dtype=dtype)
            _cmp_bf16(got, torch_lookup(idx, W, S, D, block, dtype))
    # hand values: UE8M0 127 is 1, 0 is 2^-127 (an fp32 subnormal), 130 is 8, 255 is NaN;
    # bf16 0x3FC0 is 1.5; E4M3 scale 0x40 is 2
    assert oracle.e8m0_to_f32(127, L) == 1.0 and oracle.e8m0_to_f32(130, L) == 8.0
    assert oracle.e8m0_to_f32(0, L) == 2.0 ** -127 and np.isnan(oracle.e8m0_to_f32(255, L))
    assert oracle.bf16_to_f32(0x3FC0, L) == 1.5 and oracle.bf16_to_f32(0x8000, L) == 0.0
    W = np.array([[0x38] * 16], dtype=np.uint8)  # 1.0
    for dtype, sc, want in ((oracle.SCALE_E8M0, [[126]], 0x3F00), (oracle.SCALE_BF16, [[0x3FC0]], 0x3FC0),
                            (oracle.SCALE_E4M3, [[0x40]], 0x4000)):
        out = oracle.engram_lookup(np.array([0]), W, np.array(sc), 1, 16, 16, L, scale_dtype=dtype)
        assert (out == want).all(), (dtype, hex(int(out[0, 0])))


# ----------------------------------------------------------------------------- hash


def _history_rows(seqs_ids, seqs_mask, lay):
    """Compressed history per row from the raw sequences (brute-force side)."""
    hist = []
    for ids, msk in zip(seqs_ids, seqs_mask):
        hist.append({q: brute.compress(int(ids[q]), bool(msk[q]), lay.token_map, lay.dead) for q in range(len(ids))})
    return hist


def _tiny_layouts():
    lays = []
    for full64 in (False, True):
        lays.append(synth.make_layout("tiny", 99 + full64, full64=full64))
    # a wider tiny layout: 2 layers, N=5, 3 heads, full 64-bit multipliers
    primes = synth.distinct_primes_in(5, 997, 2003, (2, 4, 3))
    lay = synth.Layout(2, 5, 3, 32, 32, 300, 50, synth.uniform_int(5, synth.TAG_TOKEN_MAP, 300, 0, 50),
                       synth.multipliers(5, 2, 5, full64=True), primes, synth.column_offsets(primes))
    lays.append(lay)
    return lays


def pin_brute_force(L=None):
    for li, lay in enumerate(_tiny_layouts()):
        B, total = 3, 48
        ids = synth.uniform_int(17 + li, synth.TAG_IDS, B * total, -2, lay.raw_vocab + 2).reshape(B, total)
        ids[:, ::11] = 0  # some repeats
        ids[0, 5], ids[1, 7], ids[2, 9] = -1, lay.raw_vocab, -2  # invalid ids: treated as masked, flagged
        mask = synth.uniform_int(18 + li, synth.TAG_IDS, B * total, 0, 5).reshape(B, total) > 0
        hist = _history_rows(ids, mask, lay)
        # one-shot
        st = oracle.OracleState.from_layout(lay, B, 64, L)
        got, flags = st.hash(ids, 0, mask)
        assert flags & oracle.FLAG_BAD_ID  # the ids include -2, -1, vocab, vocab+1
        for b in range(B):
            for t in range(total):
                exp = brute.hashes_at(hist[b], t, lay)
                assert got[b, t].tolist() == exp, (li, b, t, got[b, t].tolist(), exp)
        # chunked with per-row start positions: rows advance by different chunk sizes
        st.reset()
        pos = [0] * B
        sizes = [5, 1, 7, 13, 2, 20]
        for L_c in sizes:
            sp = np.array(pos, dtype=np.int64)
            chunk_ids = np.stack([ids[b, pos[b]:pos[b] + L_c] for b in range(B)])
            chunk_mask = np.stack([mask[b, pos[b]:pos[b] + L_c] for b in range(B)])
            got, _ = st.hash(chunk_ids, sp, chunk_mask)
            for b in range(B):
                for t in range(L_c):
                    exp = brute.hashes_at(hist[b], pos[b] + t, lay)
                    assert got[b, t].tolist() == exp, ("chunked", li, b, pos[b] + t)
            pos = [p + L_c for p in pos]
        # rows at different start positions in one call (decode-like)
        st.reset()
        st.hash(ids[:, :40], 0, mask[:, :40])
        sp = np.array([3, 17, 40], dtype=np.int64)
        one = np.stack([ids[b, sp[b]:sp[b] + 1] for b in range(B)])
        onem = np.stack([mask[b, sp[b]:sp[b] + 1] for b in range(B)])
        got, _ = st.hash(one, sp, onem)
        for b in range(B):
            h = {q: v for q, v in hist[b].items() if q <= sp[b]}
            assert got[b, 0].tolist() == brute.hashes_at(h, int(sp[b]), lay), ("decode", li, b)


def pin_closed_forms(L=None):
    """One-hot multipliers turn the hash into a plain function of one lookback slot.

    N=2, one head, prime P above the compressed vocab, offset O:
      M = [1, 0]  ->  hash[t] = O + (c_t, or pad if c_t is DEAD)
      M = [0, 1]  ->  hash[t] = O + (c_{t-1}, or pad if t == 0 or c_t or c_{t-1} is DEAD)
    and with N=3, M = [0, 0, 1], column 1 (trigram) gives c_{t-2} under the same blocking."""
    rng = np.random.default_rng(5)
    V, CV, P, O, pad, dead = 40, 30, 1009, 77, 2, -1
    tmap = rng.integers(0, CV, size=V)
    T = 200
    ids = rng.integers(0, V, size=(1, T))
    keep = rng.random((1, T)) > 0.2
    c = np.where(keep[0], tmap[ids[0]], dead)
    for mult, shift in (([1, 0], 0), ([0, 1], 1)):
        st = oracle.OracleState(1, 2, 1, tmap, np.array([mult]), np.array([[[P]]]), np.array([[O]]), dead, pad, 1, T, L)
        got, _ = st.hash(ids, 0, keep)
        for t in range(T):
            blocked = any(t - s < 0 or c[t - s] == dead for s in range(shift + 1))
            exp = O + (pad if blocked else int(c[t - shift]))
            assert got[0, t, 0, 0] == exp, (mult, t, got[0, t, 0, 0], exp)
    # N=3 (columns: bigram h0, trigram h0): M=[0,0,1] -> bigram column hashes 0 -> O0, trigram -> c_{t-2}
    primes = np.array([[[1013], [1019]]])
    offs = np.array([[5, 5 + 1013]])
    st = oracle.OracleState(1, 3, 1, tmap, np.array([[0, 0, 1]]), primes, offs, dead, pad, 1, T, L)
    got, _ = st.hash(ids, 0, keep)
    for t in range(T):
        assert got[0, t, 0, 0] == 5
        blocked = any(t - s < 0 or c[t - s] == dead for s in range(3))
        assert got[0, t, 0, 1] == 5 + 1013 + (pad if blocked else int(c[t - 2])), t
    # a negative multiplier: rolling value is negative, the floored mod lands in [0, P)
    st = oracle.OracleState(1, 2, 1, tmap, np.array([[-3, 0]]), np.array([[[P]]]), np.array([[0]]), dead, pad, 1, T, L)
    got, _ = st.hash(ids, 0, None)
    for t in range(T):
        assert got[0, t, 0, 0] == (-3 * int(tmap[ids[0, t]])) % P


def pin_invariants(L=None):
    lay = synth.make_layout("tiny", 31, full64=True)
    B, T = 2, 256
    ids = synth.zipf_ids(31, B * T, vocab=lay.raw_vocab, s=1.3).reshape(B, T)  # repeats n-grams
    mask = np.stack([synth.image_span_mask(31, T, 0.15, lo=8, hi=24, stream=b) for b in range(B)])
    st = oracle.OracleState.from_layout(lay, B, T, L)
    one, _ = st.hash(ids, 0, mask)
    c0 = lay.token_map[ids[:, 0]]
    P = lay.primes.reshape(lay.n_layers, -1)
    O = lay.offsets
    # range: every hash is inside its column's bucket range
    assert ((one >= O[None, None]) & (one < (O + P)[None, None])).all()
    # masked positions hash like the all-pad n-gram
    pad_hash = np.array(brute.hashes_at({}, 10, lay))  # empty history = every slot blocked
    assert (one[~mask] == pad_hash[None]).all()
    # position 0: every n-gram is (c_0, pad, pad, ...), so it depends on c_0 alone
    for b in range(B):
        if mask[b, 0]:
            assert one[b, 0].tolist() == brute.hashes_at({0: int(c0[b])}, 0, lay)
    # locality: equal (n-1)-token lookbacks give equal hashes for n-gram size n
    H = lay.n_heads
    c = np.where(mask, lay.token_map[np.clip(ids, 0, lay.raw_vocab - 1)], lay.dead)
    seen = {}
    hits = 0
    for b in range(B):
        for t in range(lay.max_ngram - 1, T):
            window = tuple(c[b, t - lay.max_ngram + 1:t + 1])
            if lay.dead in window:
                continue
            key = window
            if key in seen:
                hits += 1
                assert (one[b, t] == one[seen[key]]).all()
            else:
                seen[key] = (b, t)
    assert hits > 0, "Zipf input should repeat a 4-gram"
    # chunked prefill == one-shot
    st.reset()
    parts = []
    for s0, s1 in ((0, 1), (1, 3), (3, 100), (100, 101), (101, 256)):
        h, _ = st.hash(ids[:, s0:s1], s0, mask[:, s0:s1])
        parts.append(h)
    assert np.array_equal(np.concatenate(parts, axis=1), one)
    # a row that does not fit the cache is rejected: hash -1, no cache write, flagged
    snap = st.cache.copy()
    h, fl = st.hash(ids[:, :10], np.array([T - 5, 0]), mask[:, :10])
    assert fl & oracle.FLAG_BAD_START and (h[0] == -1).all() and (h[1] >= 0).all()
    assert np.array_equal(st.cache[0], snap[0])


def pin_varlen(L=None):
    """Packed ragged sequences (lengths 0, 1, 5, 17, 40 at different starts) against the brute
    force, and equal-length packs against the dense call."""
    lay = synth.make_layout("tiny", 41, full64=True)
    lens = [5, 0, 17, 1, 40]
    starts = [0, 3, 6, 9, 2]
    B = len(lens)
    rng = np.random.default_rng(41)
    total = 60
    full_ids = rng.integers(0, lay.raw_vocab, size=(B, total))
    full_mask = rng.random((B, total)) > 0.15
    hist = _history_rows(full_ids, full_mask, lay)
    st = oracle.OracleState.from_layout(lay, B, 64, L)
    # history before each start, written with the dense call
    st.hash(full_ids[:, :max(starts)], 0, full_mask[:, :max(starts)])
    cu = np.concatenate([[0], np.cumsum(lens)])
    ids = np.concatenate([full_ids[b, starts[b]:starts[b] + lens[b]] for b in range(B)])
    mask = np.concatenate([full_mask[b, starts[b]:starts[b] + lens[b]] for b in range(B)])
    got, _ = st.hash_varlen(ids, cu, starts, mask)
    for b in range(B):
        h = {q: v for q, v in hist[b].items() if q < starts[b] + lens[b]}
        for t in range(lens[b]):
            assert got[cu[b] + t].tolist() == brute.hashes_at(h, starts[b] + t, lay), ("varlen", b, t)
    # equal lengths: the packed call equals the dense call
    d1 = oracle.OracleState.from_layout(lay, 3, 64, L)
    d2 = oracle.OracleState.from_layout(lay, 3, 64, L)
    dense, _ = d1.hash(full_ids[:3, :20], [0, 4, 7], full_mask[:3, :20])
    packed, _ = d2.hash_varlen(full_ids[:3, :20].reshape(-1), [0, 20, 40, 60], [0, 4, 7],
                               full_mask[:3, :20].reshape(-1))
    assert np.array_equal(dense.reshape(60, lay.n_layers, -1), packed)
    assert np.array_equal(d1.cache, d2.cache)


def pin_cache_rows(L=None):
    """A cache-row map (call row b uses cache row cache_rows[b]) only renames rows: sequences that
    change call rows and call order between calls, each kept in its own cache row, hash like the
    brute force on their own history; dense and packed calls alike."""
    lay = _tiny_layouts()[2]
    n_seq, total = 3, 60
    rng = np.random.default_rng(61)
    ids = rng.integers(0, lay.raw_vocab, size=(n_seq, total))
    mask = rng.random((n_seq, total)) > 0.15
    hist = _history_rows(ids, mask, lay)
    slot = [4, 0, 2]  # sequence s lives in cache row slot[s] of a 5-row cache
    st = oracle.OracleState.from_layout(lay, 5, 64, L)
    pos = [0] * n_seq

    def check(got_rows, order, lens):
        for i, s in enumerate(order):
            h = {q: v for q, v in hist[s].items() if q < pos[s] + lens[i]}
            for t in range(lens[i]):
                assert got_rows[i][t].tolist() == brute.hashes_at(h, pos[s] + t, lay), ("cache_rows", order, s, t)

    for order, Lc in (([0, 1, 2], 7), ([2, 0], 5), ([1], 12), ([1, 2, 0], 3)):
        cid = np.stack([ids[s, pos[s]:pos[s] + Lc] for s in order])
        cm = np.stack([mask[s, pos[s]:pos[s] + Lc] for s in order])
        got, fl = st.hash(cid, [pos[s] for s in order], cm, cache_rows=[slot[s] for s in order])
        assert fl == 0
        check(got, order, [Lc] * len(order))
        for s in order:
            pos[s] += Lc
    # packed: sequences of different lengths (one empty), in yet another order
    order, lens = [2, 1, 0], [4, 0, 6]
    cu = np.concatenate([[0], np.cumsum(lens)])
    pid = np.concatenate([ids[s, pos[s]:pos[s] + n] for s, n in zip(order, lens)])
    pm = np.concatenate([mask[s, pos[s]:pos[s] + n] for s, n in zip(order, lens)])
    got, fl = st.hash_varlen(pid, cu, [pos[s] for s in order], pm, cache_rows=[slot[s] for s in order])
    assert fl == 0
    check([got[cu[i]:cu[i + 1]] for i in range(len(order))], order, lens)
    for s, n in zip(order, lens):
        pos[s] += n
    assert (st.cache[[1, 3]] == lay.dead).all()  # rows no sequence maps to are never written
    # a row mapped outside the cache: hash -1, flagged, no write; the other row is unaffected
    snap = st.cache.copy()
    got, fl = st.hash(np.stack([ids[1, pos[1]:pos[1] + 4], ids[0, pos[0]:pos[0] + 4]]), [pos[1], pos[0]],
                      np.stack([mask[1, pos[1]:pos[1] + 4], mask[0, pos[0]:pos[0] + 4]]), cache_rows=[5, slot[0]])
    assert fl == oracle.FLAG_BAD_ROW and (got[0] == -1).all()
    check(got[1:], [0], [4])
    keep = [r for r in range(5) if r != slot[0]]
    assert np.array_equal(st.cache[keep], snap[keep])
    _, fl = st.hash(ids[:1, :2], [0], None, cache_rows=[-1])
    assert fl == oracle.FLAG_BAD_ROW
    # the identity map is the call without a map
    a = oracle.OracleState.from_layout(lay, 3, 64, L)
    b = oracle.OracleState.from_layout(lay, 3, 64, L)
    ha, _ = a.hash(ids[:, :20], [0, 3, 9], mask[:, :20])
    hb, _ = b.hash(ids[:, :20], [0, 3, 9], mask[:, :20], cache_rows=[0, 1, 2])
    assert np.array_equal(ha, hb) and np.array_equal(a.cache, b.cache)


# ----------------------------------------------------------------------------- Engram gate


def _bf16(x):
    import torch

    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_bf16_from_f64():
    # exact ties and near-ties that a float32 intermediate would round twice
    one = 1.0
    cases = {one + 2 ** -8: 0x3F80, one + 2 ** -8 + 2 ** -40: 0x3F81, one + 3 * 2 ** -8: 0x3F82,
             -(one + 2 ** -8 + 2 ** -40): 0xBF81, 2.0 ** -133: 0x0001, 2.0 ** -134: 0x0000, 0.0: 0x0000}
    for v, bits in cases.items():
        got = int(oracle.f64_to_bf16_bits(np.array([v]))[0])
        assert got == bits, (v, hex(got), hex(bits))


def pin_linear():
    rng = np.random.default_rng(1)
    emb = _bf16(rng.standard_normal((5, 12)))
    # one-hot weight rows pick single input columns: exact
    w = np.zeros((4, 12), dtype=np.float32)
    w[[0, 1, 2, 3], [0, 5, 11, 7]] = 1.0
    kv = oracle.engram_linear(emb, _bf16(w))
    assert np.array_equal(kv, emb[:, [0, 5, 11, 7]])
    # small integers: every product and sum is exact in float32 and bf16
    a = _bf16(rng.integers(-4, 5, size=(3, 6)))
    b = _bf16(rng.integers(-4, 5, size=(2, 6)))
    exp = oracle.bf16_bits_to_f64(a) @ oracle.bf16_bits_to_f64(b).T
    assert np.array_equal(oracle.bf16_bits_to_f64(oracle.engram_linear(a, b)), exp)


def pin_gate(gate=None):
    import torch

    gate = gate or oracle.engram_gate
    rng = np.random.default_rng(2)
    T, hc, dim = 6, 4, 64
    x = _bf16(rng.standard_normal((T, hc, dim)))
    ones = _bf16(np.ones((hc, dim)))
    h = oracle.bf16_bits_to_f64(x)
    # closed form: key = c*h, unit weights -> dot = sign(c) * sqrt(dim) -> gate = sigmoid(sign(c) * dim^(1/4))
    for c in (2.0, -0.5):
        kv = np.concatenate([c * h, rng.standard_normal((T, 1, dim))], axis=1)
        kvb = _bf16(kv.reshape(T, -1))
        out = gate(x, kvb, ones, ones)
        value = oracle.bf16_bits_to_f64(kvb).reshape(T, hc + 1, dim)[:, hc, :]
        g = 1.0 / (1.0 + np.exp(-np.sign(c) * dim ** 0.25))
        assert np.allclose(out, h + g * value[:, None, :], rtol=1e-12, atol=1e-12)
    # a closed gate passes the residual through unchanged
    kvb = _bf16(rng.standard_normal((T, (hc + 1) * dim)))
    mask = np.array([True, False, True, False, False, True])
    out = gate(x, kvb, ones, ones, mask)
    assert np.array_equal(out[~mask], h[~mask])
    # a key orthogonal to h: dot is +0, clamped to 1e-6 -> gate = sigmoid(+1e-3)
    h2 = np.zeros((1, 1, dim))
    h2[0, 0, 0] = 1.0
    k2 = np.zeros((1, 2, dim))
    k2[0, 0, 1] = 1.0
    out = gate(_bf16(h2), _bf16(k2.reshape(1, -1)), _bf16(np.ones((1, dim))), _bf16(np.ones((1, dim))))
    assert out[0, 0, 0] == 1.0  # value row is zero; only the residual remains
    # the page's own code, run in float32 on torch CPU, agrees to float32 accuracy
    qw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
    kw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
    mask = rng.random(T) > 0.3
    ref = gate(x, kvb, qw, kw, mask)
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    tkv = torch.from_numpy(kvb.view(np.int16)).view(torch.bfloat16)
    key, value = tkv.split([hc * dim, dim], dim=-1)
    key = key.float().unflatten(-1, (hc, dim))
    weight = torch.from_numpy(qw.view(np.int16)).view(torch.bfloat16).float() * \
        torch.from_numpy(kw.view(np.int16)).view(torch.bfloat16).float()
    hh = tx.float()
    rstd = torch.rsqrt(hh.square().mean(-1) + 1e-20) * torch.rsqrt(key.square().mean(-1) + 1e-20)
    dot = (hh * weight * key).sum(-1) * rstd * dim ** -0.5
    gate = torch.sigmoid(torch.copysign(dot.abs().clamp_min(1e-6).sqrt(), dot))
    gate = gate.masked_fill(~torch.from_numpy(mask).unsqueeze(-1), 0)
    t32 = (hh + gate.unsqueeze(-1) * value.float().unsqueeze(-2)).numpy().astype(np.float64)
    assert np.allclose(t32, ref, rtol=1e-5, atol=1e-5)


ALL_PINS = [pin_floor_mod, pin_fp8_decode, pin_bf16, pin_lookup_vs_torch, pin_brute_force, pin_closed_forms,
            pin_invariants, pin_varlen, pin_cache_rows, pin_scale_dtypes]
