"""The lookup inside the tensor-core projection (engram_lookup_project, engram_lookup_project_gate)
against the float64 oracle chain and against the library's two-step path (GPU only).

The lookup warps dequantise each row exactly as engram_lookup does and the projection runs the same
tiles, stages and MMAs as engram_project, so the fused result must equal
engram_project(engram_lookup(idx, W, S), wkv) bit for bit (and the gated form engram_project_gate on
those rows): that comparison is exact. Against the oracle (oracle.engram_lookup, then
oracle.engram_linear in float64 and, for the gate, oracle.engram_gate) the projection's tolerance is
the one derived in test_gpu_project.py: two bf16 roundings apart plus the fp32 accumulation bound,
|got - oracle| <= 2^-7 (1 + 2^-7) |oracle| + 2 (K-1) 2^-23 sum_k |a_k b_k|; the gate's is
2^-7 (|out| + |value|) as in test_gpu_gate.py.

Shapes span one chunk of lookup work (8 tokens) up to three tile groups (4,096 tokens each), ragged
rows and columns, head_dim 64 / 128 / 256, scale blocks with one or two scales per 16-code piece,
every scale storage type, ids outside the table (+0 rows) and the strided layer slice of a hash output.
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
    assert geng.engram_device_status() == 0


def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _table(rows, D, block, sdt, layer=0, seed=20261202):
    """A small table of `rows` rows from the seeded generator: host arrays and device tensors."""
    ids = np.arange(rows, dtype=np.int64)
    W = synth.table_rows(seed, layer, ids, D)
    S = synth.table_scales(seed, layer, ids, D // block, sdt)
    return W, S, H.to_dev(W), H.to_dev(S)


def _ids(T, C, rows, stride, seed):
    """Hash ids [T, C] as the first C columns of a [T, stride] buffer; about 1% outside [0, rows)."""
    rng = np.random.default_rng(seed)
    buf = rng.integers(0, rows, size=(T, stride), dtype=np.int64)
    bad = rng.random((T, stride)) < 0.01
    buf[bad] = rng.choice(np.array([-1, rows, rows + 77, 1 << 40, -(1 << 62)], dtype=np.int64), size=int(bad.sum()))
    return buf


def _check_projection(got, emb, w, what):
    exp = oracle.engram_linear(emb, w)
    e64, g64 = oracle.bf16_bits_to_f64(exp), oracle.bf16_bits_to_f64(got)
    K = emb.shape[1]
    abs_sum = np.abs(oracle.bf16_bits_to_f64(emb)) @ np.abs(oracle.bf16_bits_to_f64(w)).T
    tol = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(e64) + 2.0 * (K - 1) * 2.0 ** -23 * abs_sum + 2.0 ** -133
    bad = np.abs(g64 - e64) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {np.argwhere(bad)[0]}"
    assert (got == exp).mean() >= 0.97, f"{what}: too few outputs equal the oracle's bf16"


@pytest.mark.parametrize("T,C,D,block,sdt,N,stride", [
    (1, 2, 64, 64, synth.SCALE_F32, 256, 2),         # one token: one chunk, one tile
    (9, 4, 64, 32, synth.SCALE_BF16, 256, 4),        # two chunks, the second holding one token
    (300, 6, 64, 64, synth.SCALE_F32, 520, 6),       # ragged rows (2 tiles) and columns
    (777, 4, 128, 8, synth.SCALE_E4M3, 264, 4),      # 16 scales per row: two per 16-code piece
    (4096, 24, 128, 128, synth.SCALE_F32, 256, 24),  # exactly one tile group
    (5000, 24, 128, 128, synth.SCALE_F32, 512, 48),  # two groups; one layer's slice of a 2-layer hash output
    (9000, 8, 256, 128, synth.SCALE_E8M0, 256, 8),   # three groups, two scales per row
])
def test_lookup_project_vs_oracle_and_two_step(T, C, D, block, sdt, N, stride):
    rows = 3001
    Wh, Sh, W, S = _table(rows, D, block, sdt)
    buf = _ids(T, C, rows, stride, seed=T + 31 * C + D)
    idx = torch.from_numpy(buf).cuda()[:, :C]
    K = C * D
    rng = np.random.default_rng(T * 3 + N)
    w = _bf16_bits(rng.standard_normal((N, K)) * K ** -0.5)
    wd = _dev_bf16(w)
    got_t = geng.engram_lookup_project(idx, W, S, wd, block, scale_dtype=sdt)
    two_t = geng.engram_project(geng.engram_lookup(idx.contiguous(), W, S, block, scale_dtype=sdt).view(T, K), wd)
    got = H.bf16_bits(got_t)
    H.assert_bits_equal(got, H.bf16_bits(two_t), f"fused vs two-step T={T} C={C} D={D}")
    emb = oracle.engram_lookup(buf[:, :C], Wh, Sh, rows, D, block, scale_dtype=sdt).reshape(T, K)
    _check_projection(got, emb, w, f"lookup projection T={T} C={C} D={D} block={block}")


def test_empty_table_gives_zero_rows():
    """rows == 0: every id is outside the table, so A is all +0 and so is the projection."""
    T, C, D, N = 40, 3, 64, 64
    idx = torch.zeros((T, C), dtype=torch.int64, device="cuda")
    W = torch.empty((0, D), dtype=torch.uint8, device="cuda")
    S = torch.empty((0, 1), dtype=torch.float32, device="cuda")
    w = _dev_bf16(_bf16_bits(np.ones((N, C * D))))
    out = geng.engram_lookup_project(idx, W, S, w, 64)
    assert (H.bf16_bits(out) == 0).all()


def test_workspace_reused_by_calls_in_a_row():
    """Two calls on one workspace, the second with other ids: its counters start again at zero and
    its rows replace the first call's (T = 4,100: two tile groups, a 4-token tail)."""
    T, C, D, block, N = 4100, 8, 128, 128, 256
    rows = 2000
    Wh, Sh, W, S = _table(rows, D, block, synth.SCALE_F32, layer=1)
    rng = np.random.default_rng(9)
    w = _dev_bf16(_bf16_bits(rng.standard_normal((N, C * D)) * (C * D) ** -0.5))
    ws = torch.empty(geng.engram_lookup_project_workspace(T, C, D), dtype=torch.uint8, device="cuda")
    outs, idxs = [], []
    for seed in (1, 2):
        idx = torch.from_numpy(_ids(T, C, rows, C, seed)).cuda()
        idxs.append(idx)
        outs.append(geng.engram_lookup_project(idx, W, S, w, block, workspace=ws))
    for idx, out in zip(idxs, outs):
        two = geng.engram_project(geng.engram_lookup(idx, W, S, block).view(T, C * D), w)
        H.assert_bits_equal(H.bf16_bits(out), H.bf16_bits(two), "calls in a row")


@pytest.mark.parametrize("T,hc,dim,stride", [(300, 4, 256, 24), (5000, 2, 512, 48)])
def test_lookup_project_gate_vs_two_step_and_oracle(T, hc, dim, stride):
    C, D, block, rows = 24, 128, 128, 4001
    Wh, Sh, W, S = _table(rows, D, block, synth.SCALE_F32, layer=1)
    buf = _ids(T, C, rows, stride, seed=T + hc)
    idx = torch.from_numpy(buf).cuda()[:, :C]
    K = C * D
    rng = np.random.default_rng(hc * 100 + dim)
    x = _bf16_bits(rng.standard_normal((T, hc, dim)))
    wkv = _bf16_bits(rng.standard_normal(((hc + 1) * dim, K)) * K ** -0.5)
    qw = _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim)))
    kw = _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim)))
    mask = rng.random(T) > 0.2
    md = torch.from_numpy(mask).cuda()
    args = (_dev_bf16(wkv), _dev_bf16(qw), _dev_bf16(kw))
    got_t = geng.engram_lookup_project_gate(_dev_bf16(x), idx, W, S, args[0], args[1], args[2], block, md)
    emb_t = geng.engram_lookup(idx.contiguous(), W, S, block).view(T, K)
    two_t = geng.engram_project_gate(_dev_bf16(x), emb_t, *args, md)
    got = H.bf16_bits(got_t)
    H.assert_bits_equal(got, H.bf16_bits(two_t), f"gated fused vs two-step T={T}")
    # the oracle chain on a sample of tokens (the float64 projection of all T rows is the slow part)
    sel = np.unique(np.concatenate([np.arange(min(T, 64)), np.arange(max(0, T - 64), T),
                                    rng.choice(T, size=min(T, 256), replace=False)]))
    emb = oracle.engram_lookup(buf[sel, :C], Wh, Sh, rows, D, block).reshape(sel.size, K)
    kv64 = oracle.engram_linear(emb, wkv)
    exp = oracle.engram_gate(x[sel], kv64, qw, kw, mask[sel])
    value = oracle.bf16_bits_to_f64(kv64).reshape(sel.size, hc + 1, dim)[:, hc:hc + 1, :].repeat(hc, 1)
    g64 = oracle.bf16_bits_to_f64(got[sel])
    tol = 2.0 ** -7 * (np.abs(exp) + np.abs(value)) + 2.0 ** -130
    bad = np.abs(g64 - exp) > tol
    assert not bad.any(), f"gated T={T}: {int(bad.sum())} outside tolerance; first {np.argwhere(bad)[0]}"


def test_block_from_hash_output():
    """ids -> engram_hash (both layers, one call) -> per layer engram_lookup_project_gate on that layer's
    strided slice of the hash output, the first launched right after the hash on the same stream (the
    projection reads ids that the previous kernel wrote); equal bit for bit to the fused hash + lookup
    followed by engram_project_gate. Prefill layout: two tables of ~24M rows on the device."""
    wl = synth.make_workload(1)
    lay = wl.layout
    B, L = 2, 700
    hc, dim = 4, 256
    T, C, D = B * L, lay.n_cols, lay.head_dim
    K = C * D
    Ws, Ss = H.device_tables(wl)
    st = H.make_state(wl, B, L)
    ids = torch.from_numpy(wl.ids[:B, :L].copy()).cuda()
    mask = torch.from_numpy(wl.mask[:B, :L].copy()).cuda()
    rng = np.random.default_rng(3)
    x = _dev_bf16(_bf16_bits(rng.standard_normal((T, hc, dim))))
    weights = [tuple(_dev_bf16(a) for a in (_bf16_bits(rng.standard_normal(((hc + 1) * dim, K)) * K ** -0.5),
                                            _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim))),
                                            _bf16_bits(rng.uniform(0.5, 1.5, (hc, dim)))))
               for _ in range(lay.n_layers)]
    md = mask.reshape(-1)
    h = st.hash(ids, 0, mask).view(T, lay.n_layers, C)
    got = [geng.engram_lookup_project_gate(x, h[:, l, :], Ws[l], Ss[l], *weights[l], lay.block, md)
           for l in range(lay.n_layers)]
    st.reset()
    rows = st.hash_lookup(ids, Ws, Ss, 0, mask)
    for l in range(lay.n_layers):
        two = geng.engram_project_gate(x, rows[l].view(T, K), *weights[l], md)
        H.assert_bits_equal(H.bf16_bits(got[l]), H.bf16_bits(two), f"block from hash output, layer {l}")
    del Ws, Ss
    torch.cuda.empty_cache()


def test_argument_errors():
    T, C, D = 16, 2, 64
    W = torch.zeros((10, D), dtype=torch.uint8, device="cuda")
    S = torch.ones((10, 1), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, C), dtype=torch.int64, device="cuda")
    w = torch.zeros((64, C * D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        geng.engram_lookup_project(idx.t(), W, S, w, 64)  # C not unit-stride
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        geng.engram_lookup_project(idx, W, S, w, 64, workspace=small)
    with pytest.raises(geng.EngramError) as e:
        geng.engram_lookup_project(idx, W, S, w, 48)  # block does not divide head_dim
    assert e.value.code == geng.ERR_UNSUPPORTED
    assert geng.engram_lookup_project(idx[:0], W, S, w, 64).shape == (0, 64)
