"""Full-scale tables (384,006,168 and 384,016,682 rows x 128 fp8, ~98 GB on the device):
the launch configuration the benchmark times, checked against the oracle on every hash id and every
output row of both layers (3,145,728 rows: the oracle regenerates the ~3.1M distinct table rows the
launch touches on the host); the long chunked prefill on every hash id and sampled rows (its chunked
output equals its one-shot output bit for bit); the Engram block's layers with the lookup inside the
projection, bit for bit against the two-step path and on sampled tokens against the oracle chain
(GPU only)."""
import numpy as np
import pytest
import torch

import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full_tables():
    H.build_all()
    wl = synth.make_workload(3)
    assert wl.layout.rows == [384_006_168, 384_016_682]
    Ws, Ss = H.device_tables(wl)
    yield Ws, Ss
    del Ws, Ss
    torch.cuda.empty_cache()


def _sample_positions(rng, B, L, n_layers, C, n):
    b = rng.integers(0, B, n)
    t = rng.integers(0, L, n)
    # tile edges and sequence ends
    edge_t = np.array([0, 1, 3, 4, 7, 8, 9, 15, 16, 17, L - 1])
    b = np.concatenate([b, np.repeat(np.arange(B), len(edge_t))])
    t = np.concatenate([t, np.tile(edge_t, B)])
    l = rng.integers(0, n_layers, b.size)
    c = rng.integers(0, C, b.size)
    return b, t, l, c


def _check_sampled_rows(wl, outs, exp_h, rng, n=20000, tag=""):
    B, L = exp_h.shape[:2]
    b, t, l, c = _sample_positions(rng, B, L, 2, 24, n)
    for layer in range(2):
        sel = l == layer
        bi, ti, ci = (torch.from_numpy(x[sel]).cuda() for x in (b, t, c))
        got = H.bf16_bits(outs[layer][bi, ti, ci])
        exp = H.oracle_lookup_rows(wl, layer, exp_h[b[sel], t[sel], layer, c[sel]])
        H.assert_bits_equal(got, exp, f"{tag} sampled rows layer {layer}")


def test_full_scale_hash_lookup(full_tables):
    Ws, Ss = full_tables
    wl = synth.make_workload(3)
    st, orc = H.make_state(wl), H.make_oracle(wl)
    hashes = torch.empty((wl.B, wl.L, 2, 24), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, hashes=hashes)
    exp_h, _ = orc.hash(wl.ids, 0)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "full-scale hashes")
    P = wl.layout.primes.reshape(2, -1)
    O = wl.layout.offsets
    assert ((exp_h >= O) & (exp_h < O + P)).all()
    # every output row of both layers: [8, 8192, 24, 128] bf16 per layer
    for layer in range(2):
        got = H.bf16_bits(outs[layer])
        exp = H.oracle_lookup_rows(wl, layer, exp_h[:, :, layer, :])
        H.assert_bits_equal(got, exp, f"full-scale rows layer {layer}")
        del got, exp
    assert st.status() == 0


def test_long_chunked_equals_one_shot(full_tables):
    Ws, Ss = full_tables
    wl = synth.make_workload(4)
    total = wl.ids.shape[1]
    Lc = wl.L
    chunked, one = H.make_state(wl), H.make_state(wl)
    ids, mask = H.to_dev(wl.ids), H.to_dev(wl.mask)
    h_chunks, outs_chunks = [], []
    for k in range(wl.chunks):
        hk = torch.empty((1, Lc, 2, 24), dtype=torch.int64, device="cuda")
        o = chunked.hash_lookup(ids[:, k * Lc:(k + 1) * Lc].contiguous(), Ws, Ss, start_pos=k * Lc,
                                mask=mask[:, k * Lc:(k + 1) * Lc].contiguous(), hashes=hk)
        h_chunks.append(hk)
        outs_chunks.append(o)
    h_one = torch.empty((1, total, 2, 24), dtype=torch.int64, device="cuda")
    outs_one = one.hash_lookup(ids, Ws, Ss, start_pos=0, mask=mask, hashes=h_one)
    h_cat = torch.cat(h_chunks, dim=1)
    assert torch.equal(h_cat, h_one), "chunked prefill differs from one-shot hashing"
    for layer in range(2):
        cat = torch.cat([o[layer] for o in outs_chunks], dim=1)
        assert torch.equal(cat.view(torch.int16), outs_one[layer].view(torch.int16))
    orc = H.make_oracle(wl)
    exp_h, _ = orc.hash(wl.ids, 0, wl.mask)
    H.assert_bits_equal(h_one.cpu().numpy(), exp_h, "long one-shot hashes")
    _check_sampled_rows(wl, outs_one, exp_h, np.random.default_rng(4), tag="long")
    # repeated n-grams (Zipf ids) repeat their hash ids
    assert np.unique(exp_h[0, :, 0, -1]).size < total


def test_full_scale_lookup_inside_projection(full_tables):
    """The Engram block's layers at full scale, as `bench.py --block --proj lookahead` runs them:
    65,536 tokens, the full-scale tables, the released width (wkv 25,600 x 3,072; 4 residual copies of
    dim 5,120). The lookup inside the projection, on each layer's slice of the hash output, equals the
    fused hash + lookup followed by the projection bit for bit on every output (keys and value, and
    the gated residual copies); sampled tokens of the gated result against the float64 oracle chain
    (oracle lookup, exact projection, gate) within the gate tests' bound 2^-7 (|out| + |value|)."""
    import gram_hash_embedding_gb300 as geng
    import oracle

    Ws, Ss = full_tables
    wl = synth.make_workload(3)
    lay = wl.layout
    T, C, D = wl.B * wl.L, lay.n_cols, lay.head_dim
    K, hc, dim = C * D, 4, 5120
    st = H.make_state(wl)
    hashes = torch.empty((wl.B, wl.L, 2, C), dtype=torch.int64, device="cuda")
    rows = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, hashes=hashes)
    h = hashes.view(T, 2, C)
    g = torch.Generator(device="cpu").manual_seed(11)
    rng = np.random.default_rng(11)
    sel = np.unique(np.concatenate([np.arange(8), np.arange(T - 8, T), rng.choice(T, 48, replace=False)]))
    x = torch.randn((T, hc, dim), generator=g).to(torch.bfloat16).cuda()
    mask = torch.from_numpy(rng.random(T) > 0.1).cuda()
    for layer in range(2):
        wkv = (torch.randn(((hc + 1) * dim, K), generator=g) * K ** -0.5).to(torch.bfloat16).cuda()
        qw = (torch.rand((hc, dim), generator=g) + 0.5).to(torch.bfloat16).cuda()
        kw = (torch.rand((hc, dim), generator=g) + 0.5).to(torch.bfloat16).cuda()
        emb = rows[layer].view(T, K)
        kv = geng.engram_lookup_project(h[:, layer, :], Ws[layer], Ss[layer], wkv, lay.block)
        assert torch.equal(kv.view(torch.int16), geng.engram_project(emb, wkv).view(torch.int16)), layer
        del kv
        got = geng.engram_lookup_project_gate(x, h[:, layer, :], Ws[layer], Ss[layer], wkv, qw, kw, lay.block, mask)
        two = geng.engram_project_gate(x, emb, wkv, qw, kw, mask)
        assert torch.equal(got.view(torch.int16), two.view(torch.int16)), layer
        del two
        # the oracle chain on the sampled tokens
        emb64 = H.oracle_lookup_rows(wl, layer, hashes.view(T, 2, C)[sel, layer, :].cpu().numpy()).reshape(sel.size, K)
        wk = H.bf16_bits(wkv)
        kv64 = oracle.engram_linear(emb64, wk)
        xs = H.bf16_bits(x[torch.from_numpy(sel).cuda()])
        exp = oracle.engram_gate(xs, kv64, H.bf16_bits(qw), H.bf16_bits(kw), mask.cpu().numpy()[sel])
        value = oracle.bf16_bits_to_f64(kv64).reshape(sel.size, hc + 1, dim)[:, hc:hc + 1, :].repeat(hc, 1)
        g64 = oracle.bf16_bits_to_f64(H.bf16_bits(got[torch.from_numpy(sel).cuda()]))
        bad = np.abs(g64 - exp) > 2.0 ** -7 * (np.abs(exp) + np.abs(value)) + 2.0 ** -130
        assert not bad.any(), f"layer {layer}: {int(bad.sum())} of {bad.size} outside tolerance"
        del got, wkv
    assert geng.engram_device_status() == 0
    assert st.status() == 0
