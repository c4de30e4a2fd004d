"""The C ABI without a GPU: the header compiles as plain C, the library loads and
exports every function the header declares, argument checks that need no device
answer with the documented codes, and the product path fails loudly when the
library is missing."""
import ctypes
import os
import re
import subprocess

import pytest

import gram_hash_embedding_gb300 as geng

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "engram.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(engram_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    geng.build()
    return ctypes.CDLL(geng.library_path())


def test_header_is_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "engram.h"\nint main(void){engram_layout l; (void)l; return 0;}\n')
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER),
                           str(src)])


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"engram_state_create", "engram_state_destroy", "engram_hash", "engram_lookup",
            "engram_hash_lookup", "engram_cache_reset", "engram_state_status", "engram_strerror"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in engram.h but not exported"


def test_host_side_checks_need_no_gpu(lib):
    lib.engram_strerror.restype = ctypes.c_char_p
    assert lib.engram_strerror(0) == b"ok"
    assert b"invalid" in lib.engram_strerror(-1)
    # null out pointer / null layout
    assert lib.engram_state_create(None, None, None, None, None, None, None) == geng.ERR_INVALID
    out = ctypes.c_void_p()
    assert lib.engram_state_create(None, None, None, None, None, None, ctypes.byref(out)) == geng.ERR_INVALID
    lay = geng._Layout(1, 4, 2, 48, 16, 1, 8, 10, -1, 2)  # head_dim 48 unsupported
    tm = (ctypes.c_int64 * 10)()
    arr = (ctypes.c_int64 * 16)()
    assert lib.engram_state_create(ctypes.byref(lay), tm, arr, arr, arr, None, ctypes.byref(out)) == geng.ERR_UNSUPPORTED
    lay = geng._Layout(1, 1, 2, 32, 32, 1, 8, 10, -1, 2)  # max_ngram 1
    assert lib.engram_state_create(ctypes.byref(lay), tm, arr, arr, arr, None, ctypes.byref(out)) == geng.ERR_INVALID
    lay = geng._Layout(9, 4, 2, 32, 32, 1, 8, 10, -1, 2)  # too many layers
    assert lib.engram_state_create(ctypes.byref(lay), tm, arr, arr, arr, None, ctypes.byref(out)) == geng.ERR_UNSUPPORTED
    lay = geng._Layout(1, 4, 2, 32, 32, 1, 8, 10, 1 << 40, 2)  # DEAD beyond int32
    assert lib.engram_state_create(ctypes.byref(lay), tm, arr, arr, arr, None, ctypes.byref(out)) == geng.ERR_INVALID
    lay = geng._Layout(1, 4, 2, 32, 32, 1, 8, 10, -1, 2, 4)  # no scale storage type 4
    assert lib.engram_state_create(ctypes.byref(lay), tm, arr, arr, arr, None, ctypes.byref(out)) == geng.ERR_UNSUPPORTED
    # lookup: unsupported head_dim / block, and an empty call, need no device
    L = lib
    L.engram_lookup.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    assert L.engram_lookup(None, 5, None, None, 4, 48, 16, 0, None, None) == geng.ERR_UNSUPPORTED
    assert L.engram_lookup(None, 5, None, None, 4, 128, 12, 0, None, None) == geng.ERR_UNSUPPORTED
    assert L.engram_lookup(None, 5, None, None, 4, 128, 128, 4, None, None) == geng.ERR_UNSUPPORTED  # scale type
    assert L.engram_lookup(None, 0, None, None, 4, 128, 128, geng.SCALE_E8M0, None, None) == geng.OK
    assert L.engram_lookup(None, -1, None, None, 4, 128, 128, 0, None, None) == geng.ERR_INVALID
    # scale pointers must be aligned to their storage type's width (rejected before any launch:
    # only rejected cases are tried, the addresses are never dereferenced)
    base = 1 << 20
    assert L.engram_lookup(base, 5, base, base + 2, 4, 128, 128, geng.SCALE_F32, base, None) == geng.ERR_INVALID
    assert L.engram_lookup(base, 5, base, base + 1, 4, 128, 128, geng.SCALE_BF16, base, None) == geng.ERR_INVALID
    assert L.engram_lookup(base + 4, 5, base, base, 4, 128, 128, geng.SCALE_E8M0, base, None) == geng.ERR_INVALID
    assert L.engram_lookup(base, 5, base + 8, base, 4, 128, 128, geng.SCALE_E4M3, base, None) == geng.ERR_INVALID
    assert lib.engram_state_destroy(None) == 0
    lib.engram_set_l2_fetch_granularity.argtypes = [ctypes.c_int32, ctypes.c_void_p]
    for bad in (7, -32, 256):  # refused before the CUDA runtime is called
        assert lib.engram_set_l2_fetch_granularity(bad, None) == geng.ERR_INVALID


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(geng, "_LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(geng, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="not built"):
        geng.engram_strerror(0)


def test_oracle_is_not_referenced_by_the_product():
    pkg = os.path.join(ROOT, "gram_hash_embedding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read().lower()
                assert "oracle" not in text, f"{f} mentions the oracle"


def test_binding_checks_sizes_before_any_pointer():
    """Buffers of the wrong size are refused by the binding before it takes a pointer (the C calls
    take raw pointers and cannot tell); CPU tensors reach the size checks first, so no GPU is needed."""
    import torch

    idx = torch.zeros(10, dtype=torch.int64)
    W = torch.zeros((4, 128), dtype=torch.uint8)
    with pytest.raises(ValueError, match="S has"):
        geng.engram_lookup(idx, W, torch.zeros((4, 2), dtype=torch.float32), 128)      # 1 scale per row expected
    with pytest.raises(ValueError, match="out has"):
        geng.engram_lookup(idx, W, torch.zeros((4, 1), dtype=torch.float32), 128,
                           out=torch.empty((9, 128), dtype=torch.bfloat16))
    x = torch.zeros((3, 4, 64), dtype=torch.bfloat16)
    w = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="kv has"):
        geng.engram_gate(x, torch.zeros((3, 4 * 64), dtype=torch.bfloat16), w, w)      # the value row is missing
    with pytest.raises(ValueError, match="mask has"):
        geng.engram_gate(x, torch.zeros((3, 5 * 64), dtype=torch.bfloat16), w, w, mask=torch.ones(4, dtype=torch.bool))


def test_lookup_projection_binding_checks_need_no_gpu():
    """engram_lookup_project(_gate): the hash ids must be an int64 CUDA tensor [T, C] with unit stride
    along C; the binding refuses anything else before taking a pointer."""
    import torch

    W = torch.zeros((4, 128), dtype=torch.uint8)
    S = torch.zeros((4, 1), dtype=torch.float32)
    wkv = torch.zeros((64, 2 * 128), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="int64 CUDA"):
        geng.engram_lookup_project(torch.zeros((8, 2), dtype=torch.int64), W, S, wkv, 128)  # a CPU tensor
    with pytest.raises(TypeError, match="int64 CUDA"):
        geng.engram_lookup_project(torch.zeros((8, 2), dtype=torch.int32), W, S, wkv, 128)
    x = torch.zeros((8, 4, 256), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="int64 CUDA"):
        geng.engram_lookup_project_gate(x, torch.zeros((8, 2), dtype=torch.int64), W, S, wkv, wkv, wkv, 128)


def test_projection_checks_need_no_gpu(lib):
    P = ctypes.c_void_p
    lib.engram_project.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P]
    lib.engram_project_gate_workspace.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    lib.engram_project_gate_workspace.restype = ctypes.c_uint64
    lib.engram_project_gate.argtypes = [P, P, P, P, P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_float, P, ctypes.c_uint64, P, P]
    a = P(4096)  # never dereferenced: every call below is rejected (or is a no-op) before a launch
    assert lib.engram_project(a, a, 0, 64, 64, a, None) == geng.OK  # T == 0: nothing to do
    assert lib.engram_project(a, a, -1, 64, 64, a, None) == geng.ERR_INVALID
    assert lib.engram_project(a, a, 5, 60, 64, a, None) == geng.ERR_UNSUPPORTED  # K not a multiple of 8
    assert lib.engram_project(a, a, 5, 64, 4, a, None) == geng.ERR_UNSUPPORTED   # N below 8
    assert lib.engram_project(a, a, 1 << 31, 64, 64, a, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_project(None, a, 5, 64, 64, a, None) == geng.ERR_INVALID
    assert lib.engram_project(P(4098), a, 5, 64, 64, a, None) == geng.ERR_INVALID  # misaligned
    # workspace: value rows (T x dim bf16) + 3 partial sums per (128-token block, key tile, token)
    # partial sums are kept for whole 256-row tiles (a pair of 128-row blocks); key tiles are 128
    # columns wide for calls of at most 256 tokens, 256 columns wide above
    assert lib.engram_project_gate_workspace(128, 4, 256) == 128 * 256 * 2 + 2 * 8 * 3 * 128 * 4
    assert lib.engram_project_gate_workspace(129, 4, 5120) == (129 * 5120 * 2 + 255) // 256 * 256 + 2 * 160 * 3 * 128 * 4
    assert lib.engram_project_gate_workspace(257, 4, 5120) == \
        (257 * 5120 * 2 + 255) // 256 * 256 + 2 * 2 * 80 * 3 * 128 * 4
    assert lib.engram_project_gate_workspace(0, 4, 256) == 0
    assert lib.engram_project_gate_workspace(8, 3, 256) == 0 and lib.engram_project_gate_workspace(8, 4, 200) == 0
    need = lib.engram_project_gate_workspace(8, 4, 256)
    assert lib.engram_project_gate(a, a, a, a, a, None, 8, 64, 3, 256, 1e-20, a, need, a, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_project_gate(a, a, a, a, a, None, 8, 64, 4, 320, 1e-20, a, need, a, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_project_gate(a, a, a, a, a, None, 8, 64, 4, 256, 1e-20, a, need - 1, a, None) == geng.ERR_INVALID
    assert lib.engram_project_gate(a, a, a, a, a, None, 8, 64, 4, 256, 1e-20, P(4096 + 16), need, a, None) == \
        geng.ERR_INVALID  # workspace must be 256-byte aligned
    assert lib.engram_project_gate(a, a, a, a, a, None, 0, 64, 4, 256, 1e-20, None, 0, a, None) == geng.OK


def test_lookup_projection_checks_need_no_gpu(lib):
    """engram_lookup_project(_gate): shapes, pointers and the workspace are checked before any launch."""
    P = ctypes.c_void_p
    L = geng._lib()  # the binding's argtypes, with the table struct
    a = P(4096)  # never dereferenced
    tb = geng._Table(4096, 4096, 100, 128, 128, geng.SCALE_F32)
    need = L.engram_lookup_project_workspace(300, 24, 128)
    # the looked-up rows (T x n_cols x head_dim bf16), then 1 + ceil(T / 4096) counters, each part 256-byte rounded
    assert need == (300 * 24 * 128 * 2 + 255) // 256 * 256 + 256
    assert L.engram_lookup_project_workspace(4097, 24, 128) == 4097 * 24 * 128 * 2 + 256
    assert L.engram_lookup_project_workspace(0, 24, 128) == 0
    ok = dict(idx=a, stride=24, T=300, C=24, wkv=a, N=256, ws=a, nbytes=need, out=a)

    def call(**kw):
        v = {**ok, **kw}
        return L.engram_lookup_project(v["idx"], v["stride"], v["T"], v["C"], ctypes.byref(kw.get("tb", tb)), v["wkv"],
                                       v["N"], v["ws"], v["nbytes"], v["out"], None)
    assert call(T=0) == geng.OK
    assert call(T=-1) == geng.ERR_INVALID
    assert call(stride=23) == geng.ERR_INVALID          # rows of ids overlap
    assert call(nbytes=need - 1) == geng.ERR_INVALID    # workspace too small
    assert call(ws=P(4096 + 64)) == geng.ERR_INVALID    # workspace not 256-byte aligned
    assert call(idx=P(4100)) == geng.ERR_INVALID        # ids not 8-byte aligned
    assert call(out=None) == geng.ERR_INVALID
    assert call(N=4) == geng.ERR_UNSUPPORTED
    assert call(T=1 << 31) == geng.ERR_UNSUPPORTED
    assert call(tb=geng._Table(4096, 4096, 100, 128, 48, geng.SCALE_F32)) == geng.ERR_UNSUPPORTED  # block
    assert call(tb=geng._Table(4096, 4096, 100, 96, 32, geng.SCALE_F32)) == geng.ERR_UNSUPPORTED   # head_dim
    assert call(tb=geng._Table(4096, 4096, 100, 128, 128, 7)) == geng.ERR_UNSUPPORTED              # scale type
    assert call(tb=geng._Table(4098, 4096, 100, 128, 128, geng.SCALE_F32)) == geng.ERR_INVALID     # W misaligned
    assert call(tb=geng._Table(4096, 4096, -1, 128, 128, geng.SCALE_F32)) == geng.ERR_INVALID
    assert L.engram_lookup_project(a, 24, 8, 24, None, a, 256, a, need, a, None) == geng.ERR_INVALID  # no table
    gneed = L.engram_lookup_project_gate_workspace(300, 24, 128, 4, 256)
    assert gneed == need + L.engram_project_gate_workspace(300, 4, 256)
    assert L.engram_lookup_project_gate_workspace(300, 24, 128, 3, 256) == 0
    g = lambda hc, dim, nbytes, T=300: L.engram_lookup_project_gate(a, a, 24, T, 24, ctypes.byref(tb), a, a, a, None,
                                                                    hc, dim, 1e-20, a, nbytes, a, None)
    assert g(3, 256, gneed) == geng.ERR_UNSUPPORTED
    assert g(4, 200, gneed) == geng.ERR_UNSUPPORTED
    assert g(4, 256, gneed - 1) == geng.ERR_INVALID
    assert g(4, 256, gneed, T=0) == geng.OK


def test_shard_checks_need_no_gpu(lib):
    P = ctypes.c_void_p
    lib.engram_shard_pack_workspace.argtypes = [ctypes.c_int64, ctypes.c_int32]
    lib.engram_shard_pack_workspace.restype = ctypes.c_uint64
    lib.engram_shard_pack.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, P, P, P, P, ctypes.c_uint64, P]
    lib.engram_shard_unpack.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, P, P]
    a = P(4096)  # never dereferenced: every call below is rejected (or is a no-op) before a launch
    # one int32 count per (segment of 4096 indices, bucket), rounded up to 256 bytes
    assert lib.engram_shard_pack_workspace(4096, 8) == 256
    assert lib.engram_shard_pack_workspace(1_572_864, 8) == (384 * 9 * 4 + 255) // 256 * 256
    assert lib.engram_shard_pack_workspace(10, 0) == 0 and lib.engram_shard_pack_workspace(10, 65) == 0
    ws = lib.engram_shard_pack_workspace(100, 4)
    assert lib.engram_shard_pack(a, 0, 10, 4, a, a, a, a, ws, None) == geng.OK
    assert lib.engram_shard_pack(a, 100, 10, 0, a, a, a, a, ws, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_shard_pack(a, 100, 10, 65, a, a, a, a, ws, None) == geng.ERR_UNSUPPORTED
    assert lib.engram_shard_pack(a, 100, -1, 4, a, a, a, a, ws, None) == geng.ERR_INVALID
    assert lib.engram_shard_pack(a, 100, 10, 4, a, a, a, a, ws - 1, None) == geng.ERR_INVALID
    assert lib.engram_shard_pack(None, 100, 10, 4, a, a, a, a, ws, None) == geng.ERR_INVALID
    assert lib.engram_shard_unpack(a, a, 5, 4, 128, a, None) == geng.ERR_INVALID  # m > n
    assert lib.engram_shard_unpack(a, a, 1, 4, 12, a, None) == geng.ERR_UNSUPPORTED  # head_dim not a multiple of 8
    assert lib.engram_shard_unpack(None, a, 0, 0, 128, a, None) == geng.OK
