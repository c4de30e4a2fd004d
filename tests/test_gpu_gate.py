"""The Engram gate kernel and the whole Engram block (lookup -> wkv projection -> gate) vs the
float64 oracle (GPU only).

Tolerance, from the arithmetic: the kernel forms h + gate*value in fp32 and rounds once to bf16
(at most half a bf16 ulp, 2^-9 relative, plus two fp32 roundings), so |out - out64| <= 2^-8 |out64|
covers the rounding. The gate itself comes from fp32 sums over dim terms (relative error ~ dim *
2^-24 on each sum); through sigmoid(signed sqrt) that moves the gate by at most ~1e-3 in the worst
case (|dot| at the 1e-6 clamp, where d gate / d dot peaks at ~125), hence + 1e-3 |value|. Masked
tokens must come out bit-exact (h + 0 * value = h). For the whole block the projection is a
cuBLAS bf16 GEMM (fp32 accumulation, bf16 output) against an exact float64 sum rounded once: one
bf16 ulp (2^-8 relative) on a key or the value, so the bound widens to 2^-7 (|out64| + |value|); the
same holds for the library's tensor-core projection, alone or with the gate fused into it.
"""
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


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _check(out_bits, exp64, value64, rel, vabs, what):
    got = oracle.bf16_bits_to_f64(out_bits)
    tol = rel * np.abs(exp64) + vabs * np.abs(value64) + 2.0 ** -130
    bad = np.abs(got - exp64) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {np.argwhere(bad)[0]}"
    exact = (out_bits == oracle.f64_to_bf16_bits(exp64)).mean()
    assert exact > 0.98, f"{what}: only {exact:.3f} of the values round to the oracle's bf16"


@pytest.mark.parametrize("hc,dim,T", [(4, 1024, 37), (4, 5120, 16), (1, 64, 5), (2, 8, 3), (8, 256, 9)])
def test_gate_vs_oracle(hc, dim, T):
    rng = np.random.default_rng(hc * 1000 + dim + T)
    x = _bf16(rng.standard_normal((T, hc, dim)))
    kv = _bf16(rng.standard_normal((T, (hc + 1) * dim)) * 0.5)
    qw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
    kw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
    mask = rng.random(T) > 0.25
    mask[0] = True
    # one token's keys proportional to its residual copies: dot near +-sqrt(dim), gate saturated
    kvr = oracle.bf16_bits_to_f64(kv).reshape(T, hc + 1, dim)
    kvr[0, :hc] = oracle.bf16_bits_to_f64(x)[0] * np.array([2.0, -0.5, 1.0, -1.0][:hc] + [1.0] * max(0, hc - 4))[:, None]
    kv = oracle.f64_to_bf16_bits(kvr.reshape(T, -1))
    out = geng.engram_gate(_dev_bf16(x), _dev_bf16(kv), _dev_bf16(qw), _dev_bf16(kw), torch.from_numpy(mask).cuda())
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    exp = oracle.engram_gate(x, kv, qw, kw, mask)
    value = oracle.bf16_bits_to_f64(kv).reshape(T, hc + 1, dim)[:, hc:hc + 1, :].repeat(hc, 1)
    _check(got, exp, value, 2.0 ** -8, 1e-3, f"gate hc={hc} dim={dim}")
    assert np.array_equal(got[~mask], x[~mask])  # closed gates: bit-exact pass-through


def test_gate_in_place_and_errors():
    rng = np.random.default_rng(9)
    T, hc, dim = 7, 4, 128
    x = _bf16(rng.standard_normal((T, hc, dim)))
    kv = _bf16(rng.standard_normal((T, (hc + 1) * dim)))
    w = _bf16(np.ones((hc, dim)))
    xd = _dev_bf16(x)
    ref = geng.engram_gate(xd.clone(), _dev_bf16(kv), _dev_bf16(w), _dev_bf16(w))
    geng.engram_gate(xd, _dev_bf16(kv), _dev_bf16(w), _dev_bf16(w), out=xd)
    assert torch.equal(xd.view(torch.int16), ref.view(torch.int16))
    with pytest.raises(geng.EngramError) as e:
        geng.engram_gate(_dev_bf16(_bf16(np.zeros((2, 3, 16)))), _dev_bf16(_bf16(np.zeros((2, 64)))),
                         _dev_bf16(_bf16(np.zeros((3, 16)))), _dev_bf16(_bf16(np.zeros((3, 16)))))
    assert e.value.code == geng.ERR_UNSUPPORTED  # hc = 3
    empty = torch.empty((0, 4, 16), dtype=torch.bfloat16, device="cuda")
    assert geng.engram_gate(empty, torch.empty((0, 80), dtype=torch.bfloat16, device="cuda"),
                            _dev_bf16(_bf16(np.ones((4, 16)))), _dev_bf16(_bf16(np.ones((4, 16))))).shape == (0, 4, 16)


@pytest.mark.parametrize("proj", ["fused", "tcgen05", "cublas"])
def test_engram_block_end_to_end(proj):
    """ids -> fused hash + lookup (this library) -> wkv projection -> gate, for both engram layers of
    the prefill layout, against the oracle chain. The projection and gate run as one fused call
    (engram_project_gate: the tensor-core projection with the gate's sums in its epilogue), as the
    library's projection followed by its gate, or as a cuBLAS GEMM followed by the gate."""
    wl = synth.make_workload(1)
    lay = wl.layout
    B, L = 2, 64
    hc, dim = 4, 256
    ids = wl.ids[:B, :L].copy()
    mask = wl.mask[:B, :L].copy()
    st, orc = H.make_state(wl, B, L), H.make_oracle(wl, B, L)
    Ws, Ss = [], []
    rows_needed = []
    exp_h, _ = orc.hash(ids, 0, mask)
    # only the rows this test touches are materialised (compact tables, indices remapped)
    rng = np.random.default_rng(5)
    for l in range(2):
        flat = exp_h[:, :, l, :].reshape(-1)
        uniq, inv = np.unique(flat, return_inverse=True)
        Wc = synth.table_rows(wl.table_seed, l, uniq, lay.head_dim)
        Sc = synth.table_scales(wl.table_seed, l, uniq, lay.n_scales)
        Ws.append(H.to_dev(Wc))
        Ss.append(H.to_dev(Sc))
        rows_needed.append(inv.reshape(B, L, lay.n_cols))
    emb = []
    for l in range(2):
        idx = torch.from_numpy(rows_needed[l]).cuda()
        emb.append(geng.engram_lookup(idx.reshape(-1), Ws[l], Ss[l], lay.block).view(B * L, lay.n_cols * lay.head_dim))
    K = lay.n_cols * lay.head_dim
    x = _bf16(rng.standard_normal((B * L, hc, dim)))
    md = torch.from_numpy(mask.reshape(-1)).cuda()
    for l in range(2):
        wkv = _bf16(rng.standard_normal((dim * (hc + 1), K)) * K ** -0.5)
        qw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
        kw = _bf16(rng.uniform(0.5, 1.5, (hc, dim)))
        if proj == "fused":
            out = geng.engram_project_gate(_dev_bf16(x), emb[l], _dev_bf16(wkv), _dev_bf16(qw), _dev_bf16(kw), md)
        else:
            kv = geng.engram_project(emb[l], _dev_bf16(wkv)) if proj == "tcgen05" else emb[l] @ _dev_bf16(wkv).t()
            out = geng.engram_gate(_dev_bf16(x), kv.contiguous(), _dev_bf16(qw), _dev_bf16(kw), md)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        # oracle chain: lookup rows (bit-exact against the kernel), exact projection, float64 gate
        rows = oracle.engram_lookup(rows_needed[l].reshape(-1), synth.table_rows(wl.table_seed, l, np.unique(exp_h[:, :, l, :]), lay.head_dim),
                                    synth.table_scales(wl.table_seed, l, np.unique(exp_h[:, :, l, :]), lay.n_scales),
                                    np.unique(exp_h[:, :, l, :]).size, lay.head_dim, lay.block).reshape(B * L, K)
        H.assert_bits_equal(emb[l].view(torch.int16).cpu().numpy().view(np.uint16), rows, "block lookup")
        kv64 = oracle.engram_linear(rows, wkv)
        exp = oracle.engram_gate(x, kv64, qw, kw, mask.reshape(-1))
        value = oracle.bf16_bits_to_f64(kv64).reshape(B * L, hc + 1, dim)[:, hc:hc + 1, :].repeat(hc, 1)
        _check(got, exp, value, 2.0 ** -7, 2.0 ** -7, f"engram block layer {l} ({proj})")
