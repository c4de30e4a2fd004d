"""engram_shard_pack_static, the pack for callers that may not allocate device memory where they pack
(a serving loop whose memory is all handed out by its own pool up front, code running during a CUDA
graph capture, a hot path that must not take an allocation's latency): its scratch is a fixed array
inside the library instead of a caller's workspace. Called through the C ABI, it must give exactly
what engram_shard_pack gives, call after call on the shared array, and refuse sizes beyond the array.

This file is collected last (its name), so a run that stops at the first failure has run every other
test before it; it passes alone in a fresh process as well as after the others (GPU only)."""
import ctypes

import numpy as np
import pytest
import torch

import gram_hash_embedding_gb300 as geng
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int32


@pytest.fixture(scope="module")
def lib():
    H.build_all()
    L = ctypes.CDLL(geng.library_path())
    L.engram_shard_pack_static.argtypes = [P, I64, I64, I32, P, P, P, P]
    L.engram_shard_pack_static.restype = ctypes.c_int
    L.engram_shard_pack.argtypes = [P, I64, I64, I32, P, P, P, P, ctypes.c_uint64, P]
    L.engram_shard_pack.restype = ctypes.c_int
    L.engram_shard_pack_workspace.argtypes = [I64, I32]
    L.engram_shard_pack_workspace.restype = ctypes.c_uint64
    return L


def _pack(L, idx, rows, world, static):
    n = idx.numel()
    counts = torch.full((world + 1,), -7, dtype=torch.int64, device="cuda")
    local = torch.full((n,), -7, dtype=torch.int64, device="cuda")
    pos = torch.full((n,), -7, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if static:
        rc = L.engram_shard_pack_static(idx.data_ptr(), n, rows, world, counts.data_ptr(), local.data_ptr(),
                                        pos.data_ptr(), s)
    else:
        nbytes = int(L.engram_shard_pack_workspace(n, world))
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        rc = L.engram_shard_pack(idx.data_ptr(), n, rows, world, counts.data_ptr(), local.data_ptr(), pos.data_ptr(),
                                 ws.data_ptr(), ws.numel(), s)
    assert rc == geng.OK, geng.engram_strerror(rc)
    torch.cuda.synchronize()
    return counts.cpu(), local.cpu(), pos.cpu()


@pytest.mark.parametrize("n,rows,world", [(1_572_864, 384_006_168, 8), (70_000, 999, 3)])
def test_static_pack_equals_the_workspace_pack_twice(lib, n, rows, world):
    rng = np.random.default_rng(n)
    for call in range(2):  # the second call finds the first call's counts in the shared array
        idx = torch.from_numpy(rng.integers(-5, rows + 5, size=n).astype(np.int64)).cuda()
        got = _pack(lib, idx, rows, world, static=True)
        exp = _pack(lib, idx, rows, world, static=False)
        for g, e, what in zip(got, exp, ("counts", "local rows", "positions")):
            assert torch.equal(g, e), f"call {call}: {what} differ"
        assert int(got[0].sum()) == n


def test_static_pack_refuses_sizes_beyond_its_array(lib):
    world = 8
    limit = (16384 // (world + 1)) * 4096
    # rejected before anything is launched, so the pointers are never dereferenced
    a = P(4096)
    assert lib.engram_shard_pack_static(a, limit + 1, 10, world, a, a, a, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_shard_pack_static(a, 10, 10, 0, a, a, a, None) == geng.ERR_UNSUPPORTED
    idx = torch.zeros(limit, dtype=torch.int64, device="cuda")
    counts, local, pos = _pack(lib, idx, 10, world, static=True)  # exactly at the limit: accepted
    assert int(counts[0]) == limit and torch.equal(pos, torch.arange(limit))
