"""Randomised parity sweep (GPU only): each case draws its own layout (layers, n-gram size, heads,
head_dim / block, scale storage type, 31- or 64-bit multipliers), tables with every fp8 code, batch
shape, per-row start positions, mask, cache-row permutation and dense or packed calls, and checks the
hash ids and bf16 rows of two consecutive chunks (so the second reads the first's cache) against the
oracle given the same inputs."""
import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

D_BLOCKS = [(16, 16), (16, 8), (32, 32), (32, 8), (64, 64), (64, 16), (128, 128), (128, 32), (256, 128), (512, 256)]
STORE = {geng.SCALE_F32: np.float32, geng.SCALE_BF16: np.uint16, geng.SCALE_E8M0: np.uint8, geng.SCALE_E4M3: np.uint8}


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    while True:
        NL, N, Hh = int(rng.integers(1, 9)), int(rng.integers(2, 9)), int(rng.integers(1, 10))
        if NL * (N - 1) * Hh <= 512:
            break
    D, block = D_BLOCKS[int(rng.integers(len(D_BLOCKS)))]
    sdt = int(rng.integers(4))
    if sdt == geng.SCALE_E8M0 and H.SCALE_TORCH_DTYPE[sdt] is None:
        sdt = geng.SCALE_BF16
    V, CV = int(rng.integers(20, 3000)), int(rng.integers(5, 2000))
    pool = np.array([q for q in range(2, 400) if synth._is_prime(q)], dtype=np.int64)
    primes = rng.choice(pool, size=(NL, N - 1, Hh))  # small tables; repeats allowed
    lay = synth.Layout(NL, N, Hh, D, block, V, CV, rng.integers(0, CV, size=V),
                       synth.multipliers(seed + 7, NL, N, full64=bool(seed % 2)), primes, synth.column_offsets(primes),
                       scale_dtype=sdt)
    return rng, lay


def _tables(rng, lay):
    Ws, Ss = [], []
    for rows in lay.rows:
        W = rng.integers(0, 256, size=(rows, lay.head_dim), dtype=np.uint8)
        if lay.scale_dtype == geng.SCALE_F32:
            S = rng.normal(0, 1, size=(rows, lay.n_scales)).astype(np.float32)
        elif lay.scale_dtype == geng.SCALE_BF16:
            S = rng.integers(0, 1 << 16, size=(rows, lay.n_scales)).astype(np.uint16)
        else:
            S = rng.integers(0, 256, size=(rows, lay.n_scales)).astype(np.uint8)
        Ws.append(W)
        Ss.append(S)
    return Ws, Ss


def _rows_equal(got, exp, what):
    nan_e = ((exp & 0x7F80) == 0x7F80) & ((exp & 0x7F) != 0)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_e, nan_g), what
    H.assert_bits_equal(np.where(nan_e, 0, got), np.where(nan_e, 0, exp), what)


@pytest.mark.parametrize("seed", range(200))
def test_random_case(seed):
    rng, lay = _random_case(seed)
    Ws, Ss = _tables(rng, lay)
    tdt = H.SCALE_TORCH_DTYPE[lay.scale_dtype]
    Wd = [H.to_dev(w) for w in Ws]
    Sd = [H.to_dev(x).view(tdt) for x in Ss]
    B = int(rng.integers(1, 7))
    max_batch = B + int(rng.integers(0, 3))
    L1, L2 = int(rng.integers(1, 80)), int(rng.integers(1, 40))
    max_seq = 200
    packed = bool(rng.integers(2))
    st = geng.EngramHash(n_layers=lay.n_layers, max_ngram=lay.max_ngram, n_heads=lay.n_heads, head_dim=lay.head_dim,
                         block=lay.block, max_batch=max_batch, max_seq_len=max_seq, token_map=lay.token_map,
                         multipliers=lay.multipliers, primes=lay.primes, offsets=lay.offsets, dead=lay.dead,
                         pad_id=lay.pad_id, scale_dtype=lay.scale_dtype)
    orc = oracle.OracleState.from_layout(lay, max_batch, max_seq)
    rows_map = rng.permutation(max_batch)[:B].astype(np.int32) if rng.integers(2) else None
    start = rng.integers(0, 60, size=B).astype(np.int32)
    C, NL = lay.n_cols, lay.n_layers
    for chunk, Lc in enumerate((L1, L2)):
        if packed:  # ragged lengths up to Lc, one may be empty
            lens = rng.integers(0, Lc + 1, size=B)
        else:
            lens = np.full(B, Lc)
        ids_rows = [rng.integers(-1, lay.raw_vocab + 1, size=int(n)) for n in lens]  # a few invalid ids
        mask_rows = [rng.random(int(n)) > 0.15 for n in lens]
        cr = None if rows_map is None else H.to_dev(rows_map)
        if packed:
            cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            ids = np.concatenate(ids_rows).astype(np.int64)
            mask = np.concatenate(mask_rows)
            T = ids.size
            exp_h, fl = orc.hash_varlen(ids, cu, start.astype(np.int64), mask, cache_rows=rows_map)
            if T == 0:
                continue
            hashes = torch.full((T, NL, C), -9, dtype=torch.int64, device="cuda")
            outs = st.hash_lookup_varlen(H.to_dev(ids), H.to_dev(cu), H.to_dev(start), Wd, Sd, mask=H.to_dev(mask),
                                         hashes=hashes, max_len=int(lens.max()), cache_rows=cr)
            exp_hv = exp_h
        else:
            ids = np.stack(ids_rows).astype(np.int64)
            mask = np.stack(mask_rows)
            exp_h, fl = orc.hash(ids, start.astype(np.int64), mask, cache_rows=rows_map)
            hashes = torch.full((B, Lc, NL, C), -9, dtype=torch.int64, device="cuda")
            outs = st.hash_lookup(H.to_dev(ids), Wd, Sd, start_pos=H.to_dev(start), mask=H.to_dev(mask),
                                  hashes=hashes, cache_rows=cr)
            exp_hv = exp_h
        what = f"seed {seed} chunk {chunk} (layers {NL}, N {lay.max_ngram}, heads {lay.n_heads}, D {lay.head_dim}/" \
               f"{lay.block}, scale type {lay.scale_dtype}, B {B}, packed {packed}, map {rows_map is not None})"
        H.assert_bits_equal(hashes.cpu().numpy(), exp_hv, "hashes " + what)
        for l in range(NL):
            exp_rows = oracle.engram_lookup(exp_hv[..., l, :], Ws[l], Ss[l], lay.rows[l], lay.head_dim, lay.block,
                                            scale_dtype=lay.scale_dtype)
            _rows_equal(H.bf16_bits(outs[l]), exp_rows, f"rows layer {l} " + what)
        assert st.status() == fl, what  # bad ids flagged alike
        start = start + lens.astype(np.int32)
