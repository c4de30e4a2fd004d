"""Scale tensors stored as bf16, UE8M0 or E4M3 (the lookup page leaves `scale_dtype` open and widens
it with `.float()`): the lookup over every scale code, the fused path on small tables, and the
released head_dim with UE8M0 scales on the full-scale tables, all against the oracle (GPU only)."""
import dataclasses

import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
import synth
from tests import gpu_helpers as H
from tests.test_gpu_fullscale import _check_sampled_rows

pytestmark = pytest.mark.gpu

KINDS = [(geng.SCALE_BF16, torch.bfloat16, np.uint16), (geng.SCALE_E8M0, getattr(torch, "float8_e8m0fnu", None), np.uint8),
         (geng.SCALE_E4M3, torch.float8_e4m3fn, np.uint8)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


def _nan_aware_equal(got, exp, what):
    nan_e = ((exp & 0x7F80) == 0x7F80) & ((exp & 0x7F) != 0)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_e, nan_g), what
    H.assert_bits_equal(np.where(nan_e, 0, got), np.where(nan_e, 0, exp), what)


@pytest.mark.parametrize("sdt,tdt,store", KINDS)
@pytest.mark.parametrize("D,block", [(16, 16), (64, 16), (128, 128), (256, 128), (512, 128)])
def test_lookup_every_scale_code(sdt, tdt, store, D, block):
    rng = np.random.default_rng(D + 31 * sdt)
    nsc = D // block
    if store is np.uint8:
        codes = np.arange(256, dtype=np.uint8)  # every UE8M0 exponent / E4M3 code, NaN included
    else:
        codes = np.concatenate([rng.integers(0, 1 << 16, size=500), [0, 0x8000, 1, 0x807F, 0x7F80, 0xFF80, 0x7FC0]])
    rows = -(-codes.size // nsc) + 9
    S = np.resize(codes, rows * nsc).astype(store).reshape(rows, nsc)
    W = rng.integers(0, 256, size=(rows, D), dtype=np.uint8)
    idx = np.concatenate([np.arange(rows), rng.integers(-3, rows + 3, size=700)]).astype(np.int64)
    exp = oracle.engram_lookup(idx, W, S, rows, D, block, scale_dtype=sdt)
    Sd = H.to_dev(S)
    if tdt is not None:  # as the torch scale dtype, and as raw bits with the type given explicitly
        out = geng.engram_lookup(H.to_dev(idx), H.to_dev(W), Sd.view(tdt), block)
        _nan_aware_equal(H.bf16_bits(out), exp, f"lookup scale type {sdt} D={D}")
    out = geng.engram_lookup(H.to_dev(idx), H.to_dev(W), Sd, block, scale_dtype=sdt)
    _nan_aware_equal(H.bf16_bits(out), exp, f"lookup scale type {sdt} D={D} (bits)")


@pytest.mark.parametrize("sdt", [geng.SCALE_BF16, geng.SCALE_E8M0, geng.SCALE_E4M3])
@pytest.mark.parametrize("D,block", [(32, 32), (64, 16), (256, 128)])
def test_fused_small_tables(sdt, D, block):
    base = synth.make_workload(0, full64=True)
    lay = dataclasses.replace(base.layout, head_dim=D, block=block, scale_dtype=sdt)
    wl = dataclasses.replace(base, layout=lay)
    if H.SCALE_TORCH_DTYPE[sdt] is None:
        pytest.skip("this torch has no float8_e8m0fnu")
    Ws, Ss = H.device_tables(wl)
    st, orc = H.make_state(wl), H.make_oracle(wl)
    hashes = torch.empty((1, 64, 1, lay.n_cols), dtype=torch.int64, device="cuda")
    outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, hashes=hashes)
    exp_h, _ = orc.hash(wl.ids, 0)
    H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "hashes")
    H.assert_bits_equal(H.bf16_bits(outs[0]), H.oracle_lookup_rows(wl, 0, exp_h[:, :, 0, :]), f"rows type {sdt}")
    # scales of the wrong storage type are refused before anything runs
    with pytest.raises(TypeError):
        st.hash_lookup(H.to_dev(wl.ids), Ws, [torch.zeros(s.shape, dtype=torch.float32, device="cuda") for s in Ss])


def test_full_scale_head_dim_256_ue8m0_scales():
    torch.cuda.empty_cache()
    wl = synth.make_workload(8)
    lay = wl.layout
    if H.SCALE_TORCH_DTYPE[lay.scale_dtype] is None:
        pytest.skip("this torch has no float8_e8m0fnu")
    assert lay.head_dim == 256 and lay.scale_bytes == 1 and lay.rows == [384_006_168, 384_016_682]
    free, _ = torch.cuda.mem_get_info()
    need = sum(lay.rows) * (lay.head_dim + lay.scale_bytes * lay.n_scales) + 4 * 2 ** 30
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB free on the device, {free / 1e9:.0f} GB available")
    Ws, Ss = H.device_tables(wl)
    try:
        st, orc = H.make_state(wl), H.make_oracle(wl)
        hashes = torch.empty((wl.B, wl.L, 2, 24), dtype=torch.int64, device="cuda")
        outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, hashes=hashes)
        exp_h, _ = orc.hash(wl.ids, 0)
        H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "ue8m0 hashes")
        _check_sampled_rows(wl, outs, exp_h, np.random.default_rng(8), n=8000, tag="ue8m0")
        # the standalone lookup on the same tables agrees with the fused rows
        idx = hashes[0, :64, 1, :].contiguous().view(-1)
        lk = st.lookup(idx, Ws[1], Ss[1])
        assert torch.equal(lk.view(torch.int16), outs[1][0, :64].reshape(-1, 256).view(torch.int16))
        assert st.status() == 0
    finally:
        del Ws, Ss
        torch.cuda.empty_cache()
