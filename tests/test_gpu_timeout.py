"""The projection's failure path (GPU only): every mbarrier wait of the tensor-core kernel gives up
after one second, raises ENGRAM_STATUS_TIMEOUT and ends the kernel instead of hanging the GPU. The
test hook engram_project_withhold makes one tile's completion signal never arrive (nothing sends it),
so that tile's epilogue waits run out; the call must finish within seconds with the flag raised, and
the same context must then compute a correct projection."""
import ctypes
import time

import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
import oracle
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    H.build_all()
    L = geng._lib()
    L.engram_project_withhold.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    L.engram_project_withhold.restype = ctypes.c_int
    return L


def _operands(T, K, N, seed):
    rng = np.random.default_rng(seed)
    emb = torch.from_numpy(rng.standard_normal((T, K)).astype(np.float32)).to(torch.bfloat16).cuda()
    w = torch.from_numpy((rng.standard_normal((N, K)) * K ** -0.5).astype(np.float32)).to(torch.bfloat16).cuda()
    return emb, w


@pytest.mark.parametrize("T,K,N,tile", [
    (512, 256, 512, 0),     # 4 tiles: four clusters with one tile each, that tile never signalled
    (4096, 128, 2048, 0),   # clusters with two tiles: the second is signalled, the first never drains
])
def test_withheld_completion_ends_with_timeout_flag(lib, T, K, N, tile):
    assert geng.engram_device_status() == 0  # a clean start (reads and clears)
    emb, w = _operands(T, K, N, T + N)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    rc = lib.engram_project_withhold(emb.data_ptr(), w.data_ptr(), T, K, N, out.data_ptr(), tile,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == geng.OK
    torch.cuda.synchronize()  # returns: the kernel ended on its own
    elapsed = time.time() - t0
    assert elapsed < 30.0, elapsed
    assert geng.engram_device_status() & geng.STATUS_TIMEOUT
    assert geng.engram_device_status() == 0  # the read cleared it

    # the context is still usable: a normal projection right after is correct
    got = geng.engram_project(emb, w).view(torch.int16).cpu().numpy().view(np.uint16)
    e = emb.view(torch.int16).cpu().numpy().view(np.uint16)
    wb = w.view(torch.int16).cpu().numpy().view(np.uint16)
    exp = oracle.engram_linear(e, wb)
    e64, g64 = oracle.bf16_bits_to_f64(exp), oracle.bf16_bits_to_f64(got)
    abs_sum = np.abs(oracle.bf16_bits_to_f64(e)) @ np.abs(oracle.bf16_bits_to_f64(wb)).T
    tol = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(e64) + 2.0 * (K - 1) * 2.0 ** -23 * abs_sum + 2.0 ** -133
    assert not (np.abs(g64 - e64) > tol).any()
    assert geng.engram_device_status() == 0


def test_withhold_argument_checks(lib):
    a = ctypes.c_void_p(4096)  # rejected before a launch: never dereferenced
    assert lib.engram_project_withhold(a, a, 8, 64, 64, a, -1, None) == geng.ERR_INVALID
    assert lib.engram_project_withhold(a, a, 8, 60, 64, a, 0, None) == geng.ERR_UNSUPPORTED
