"""The released head_dim: full-scale tables of 256 fp8 values per row with two fp32 scales per row
(~203 GB on the device), checked against the oracle on every hash id and on sampled rows (GPU only)."""
import numpy as np
import pytest
import torch

import synth
from tests import gpu_helpers as H
from tests.test_gpu_fullscale import _check_sampled_rows

pytestmark = pytest.mark.gpu


def test_full_scale_head_dim_256():
    H.build_all()
    torch.cuda.empty_cache()
    wl = synth.make_workload(6)
    lay = wl.layout
    assert lay.head_dim == 256 and lay.n_scales == 2 and lay.rows == [384_006_168, 384_016_682]
    free, _ = torch.cuda.mem_get_info()
    need = sum(lay.rows) * (lay.head_dim + 4 * lay.n_scales) + 4 * 2 ** 30
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB free on the device, {free / 1e9:.0f} GB available")
    Ws, Ss = H.device_tables(wl)
    try:
        st, orc = H.make_state(wl), H.make_oracle(wl)
        hashes = torch.empty((wl.B, wl.L, 2, 24), dtype=torch.int64, device="cuda")
        outs = st.hash_lookup(H.to_dev(wl.ids), Ws, Ss, start_pos=0, hashes=hashes)
        exp_h, _ = orc.hash(wl.ids, 0)
        H.assert_bits_equal(hashes.cpu().numpy(), exp_h, "d256 hashes")
        _check_sampled_rows(wl, outs, exp_h, np.random.default_rng(6), n=8000, tag="d256")
        assert st.status() == 0
    finally:
        del Ws, Ss
        torch.cuda.empty_cache()
