"""bench.py's end-to-end leg (GPU only): the pipelined steps, which alternate two sets of buffers and
overlap one step's calls with the previous step's copies, bring back the bf16 rows of one fused call
on the same ids."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from tests import gpu_helpers as H  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    H.build_all()
    yield


def test_pipelined_steps_return_the_rows_of_one_call():
    r = bench.Runner(5, 0, torch.device("cuda", 0))  # B4 x L4096 on ~1 GB of tables
    r.setup_mode("fused")
    r.e2e_buffers()
    assert len(r.e2e_pieces) > 1  # the pipelined leg: one call per group of batch rows
    steps = 5
    for k in range(steps):  # no wait between steps but the last
        r.e2e_step(k, drain=k == steps - 1)
    torch.cuda.synchronize()
    for k in (steps - 2, steps - 1):  # the last step of each buffer set
        j = k % len(r.ids)
        host_rows = r.e2e_sets[k % 2][4]
        ref = [torch.empty_like(o) for o in r.out]
        r.geng.engram_hash_lookup(r.state.handle, r.ids[j], r.starts[j % len(r.starts)], r.W, r.S,
                                  r.masks[j % len(r.masks)], ref)
        torch.cuda.synchronize()
        for got, exp in zip(host_rows, ref):
            assert torch.equal(got.view(torch.int16), exp.cpu().view(torch.int16)), f"step {k}"
    assert r.state.status() == 0
