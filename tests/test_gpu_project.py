"""The tensor-core `wkv` projection (engram_project) and the projection with the gate fused into its
epilogue (engram_project_gate) against the float64 oracle (GPU only).

Tolerance of the projection, from the arithmetic: each product of two bf16 values is exact in fp32;
the kernel adds the K products in fp32 (tensor-core accumulation; even with truncating adds each of
the K-1 additions errs by at most 2^-23 of the running sum's magnitude, bounded by sum|a*b|), then
rounds once to bf16 (8 significant bits: at most 2^-8 relative). The oracle rounds the exact sum to
bf16 once, so two roundings separate the results where the sum lies near a rounding boundary:
|got - oracle| <= 2^-7 (1 + 2^-7) |oracle| + 2 (K-1) 2^-23 sum_k |a_k b_k|. In practice all but a
few outputs round to the oracle's bf16 (the fp32 error is ~2^-24 sqrt(K) sum|ab|, far below half a
bf16 ulp).

The fused path runs the same accumulators, so its keys equal engram_project's bf16 keys bit for bit;
only the order of the fp32 sums of the gate differs from engram_gate's. It is checked against the
oracle chain (oracle.engram_linear, then oracle.engram_gate in float64) with the gate tests'
tolerance for a bf16 projection, 2^-7 (|out| + |value|), and against the unfused library path.
"""
import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield
    assert geng.engram_device_status() == 0


def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(T, K, N, seed):
    rng = np.random.default_rng(seed)
    emb = _bf16_bits(rng.standard_normal((T, K)))
    w = _bf16_bits(rng.standard_normal((N, K)) * K ** -0.5)
    return emb, w


def _check_projection(got, emb, w, what, min_exact=0.97):
    exp = oracle.engram_linear(emb, w)
    e64 = oracle.bf16_bits_to_f64(exp)
    g64 = oracle.bf16_bits_to_f64(got)
    K = emb.shape[1]
    abs_sum = np.abs(oracle.bf16_bits_to_f64(emb)) @ np.abs(oracle.bf16_bits_to_f64(w)).T
    tol = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(e64) + 2.0 * (K - 1) * 2.0 ** -23 * abs_sum + 2.0 ** -133
    bad = np.abs(g64 - e64) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {np.argwhere(bad)[0]}"
    exact = (got == exp).mean()
    assert exact >= min_exact, f"{what}: only {exact:.4f} of the outputs equal the oracle's bf16"


@pytest.mark.parametrize("T,K,N", [
    (1, 64, 256),        # one row, one tile
    (128, 128, 512),     # whole tiles
    (300, 192, 520),     # ragged rows (3 tiles, the last 44 rows) and columns (3 tiles, the last 8 columns)
    (257, 200, 264),     # K not a multiple of 64: the last K block is partly past the matrix (zero-filled)
    (64, 8, 8),          # the smallest K and N
    (1000, 3072, 256),   # the block's K (24 columns x 128) over many K blocks
    (2200, 96, 2056),    # more tiles than SMs: every CTA takes several tiles, both accumulators in turn
])
def test_project_vs_oracle(T, K, N):
    emb, w = _inputs(T, K, N, seed=T * 7 + K * 3 + N)
    got = _host(geng.engram_project(_dev(emb), _dev(w)))
    _check_projection(got, emb, w, f"projection T={T} K={K} N={N}")


def test_project_block_shape_sampled_rows():
    """The released block's shape (65,536 tokens, K = 24 x 128, N = 5 x 5120) and a ragged T: every
    output is checked against cuBLAS within the projection's tolerance (cuBLAS also accumulates in
    fp32: the bound is twice the one above), and 40 sampled rows plus the last rows against the oracle."""
    K, N = 3072, 25600
    for T in (65536, 65536 - 77):
        g = torch.Generator(device="cuda").manual_seed(T)
        emb = torch.randn((T, K), generator=g, device="cuda").to(torch.bfloat16)
        w = (torch.randn((N, K), generator=g, device="cuda") * K ** -0.5).to(torch.bfloat16)
        out = geng.engram_project(emb, w)
        ref = emb @ w.t()
        abs_sum = emb.abs().float() @ w.abs().float().t()
        # whole output vs cuBLAS, in row blocks to bound memory
        for r0 in range(0, T, 8192):
            o = out[r0:r0 + 8192].float()
            r = ref[r0:r0 + 8192].float()
            tol = 2.0 ** -7 * 1.01 * r.abs() + 4.0 * (K - 1) * 2.0 ** -23 * abs_sum[r0:r0 + 8192] * 1.01
            assert bool(((o - r).abs() <= tol).all()), f"block shape T={T}: rows {r0}.. differ from cuBLAS"
            same = (out[r0:r0 + 8192].view(torch.int16) == ref[r0:r0 + 8192].view(torch.int16)).float().mean()
            assert float(same) > 0.97
        rows = np.unique(np.concatenate([np.random.default_rng(T).integers(0, T, 40), np.arange(T - 3, T)]))
        idx = torch.from_numpy(rows).cuda()
        _check_projection(_host(out[idx]), _host(emb[idx]), _host(w), f"block shape T={T} sampled rows")
        del out, ref, abs_sum


def test_project_writes_only_its_output():
    """Rows past T and columns past N are never written: the output is carved out of a larger
    buffer whose guard bands keep their contents."""
    T, K, N = 130, 64, 264
    emb, w = _inputs(T, K, N, seed=5)
    buf = torch.full((T * N + 4096,), 1.5, dtype=torch.bfloat16, device="cuda")
    out = buf[2048:2048 + T * N].view(T, N)
    geng.engram_project(_dev(emb), _dev(w), out=out)
    assert bool((buf[:2048] == 1.5).all()) and bool((buf[2048 + T * N:] == 1.5).all())
    _check_projection(_host(out), emb, w, "projection into a carved buffer")


@pytest.mark.parametrize("T,K,hc,dim", [(200, 3072, 4, 256), (77, 384, 1, 512), (130, 256, 8, 256),
                                        (300, 128, 2, 768), (1, 64, 4, 256)])
def test_project_gate_vs_oracle(T, K, hc, dim):
    rng = np.random.default_rng(T + K + hc + dim)
    emb = _bf16_bits(rng.standard_normal((T, K)))
    wkv = _bf16_bits(rng.standard_normal(((hc + 1) * dim, K)) * K ** -0.5)
    x = _bf16_bits(rng.standard_normal((T, hc, dim)))
    qw = _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim)))
    kw = _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim)))
    mask = rng.random(T) > 0.2
    mask[0] = True
    md = torch.from_numpy(mask).cuda()
    fused = geng.engram_project_gate(_dev(x), _dev(emb), _dev(wkv), _dev(qw), _dev(kw), md)
    got = _host(fused)
    # the oracle chain: exact projection rounded to bf16, then the float64 gate
    kv64 = oracle.engram_linear(emb, wkv)
    exp = oracle.engram_gate(x, kv64, qw, kw, mask)
    value = oracle.bf16_bits_to_f64(kv64).reshape(T, hc + 1, dim)[:, hc:hc + 1, :].repeat(hc, 1)
    g64 = oracle.bf16_bits_to_f64(got)
    tol = 2.0 ** -7 * (np.abs(exp) + np.abs(value)) + 2.0 ** -130
    bad = np.abs(g64 - exp) > tol
    assert not bad.any(), f"fused gate: {int(bad.sum())} of {bad.size} outside tolerance; first {np.argwhere(bad)[0]}"
    assert np.array_equal(got[~mask], x[~mask])  # closed gates pass h through bit for bit
    # against the unfused library path: the same bf16 keys and value, the gate sums in another order
    kv = geng.engram_project(_dev(emb), _dev(wkv))
    unfused = _host(geng.engram_gate(_dev(x), kv, _dev(qw), _dev(kw), md))
    assert (unfused == got).mean() > 0.99


def test_project_gate_in_place_and_workspace_reuse():
    T, K, hc, dim = 150, 256, 4, 256
    rng = np.random.default_rng(3)
    emb = _dev(_bf16_bits(rng.standard_normal((T, K))))
    wkv = _dev(_bf16_bits(rng.standard_normal(((hc + 1) * dim, K)) * K ** -0.5))
    qw = _dev(_bf16_bits(rng.uniform(0.5, 1.5, (hc, dim))))
    kw = _dev(_bf16_bits(rng.uniform(0.5, 1.5, (hc, dim))))
    x = _dev(_bf16_bits(rng.standard_normal((T, hc, dim))))
    ws = torch.empty(geng.engram_project_gate_workspace(T, hc, dim), dtype=torch.uint8, device="cuda")
    ref = geng.engram_project_gate(x.clone(), emb, wkv, qw, kw, workspace=ws)
    y = x.clone()
    geng.engram_project_gate(y, emb, wkv, qw, kw, workspace=ws, out=y)  # in place, same workspace
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    with pytest.raises(ValueError):
        geng.engram_project_gate(x, emb, wkv, qw, kw, workspace=ws[:-1])
    with pytest.raises(geng.EngramError) as e:
        geng.engram_project_gate(x[:, :, :128].contiguous(), emb, wkv[:5 * 128].contiguous(), qw[:, :128].contiguous(),
                                 kw[:, :128].contiguous(), workspace=ws)
    assert e.value.code == geng.ERR_UNSUPPORTED  # dim 128 is not a multiple of 256


def test_project_in_a_cuda_graph():
    """The projection allocates nothing per call and never synchronises: captured once, replayed."""
    T, K, N = 256, 128, 512
    emb, w = _inputs(T, K, N, seed=11)
    e, wd = _dev(emb), _dev(w)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    geng.engram_project(e, wd, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        geng.engram_project(e, wd, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    _check_projection(_host(out), emb, w, "graph replay")
