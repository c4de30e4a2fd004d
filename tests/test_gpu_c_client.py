"""The C ABI from a plain C program (no Python or torch in the loop): tests/c_client/engram_client.c
is compiled with gcc against include/engram.h, libengram.so and the CUDA runtime, run on a tiny
workload, and its hash ids, bf16 rows and the lookup inside the projection are compared with the
oracle (GPU only)."""
import os
import subprocess

import numpy as np
import pytest

import gram_hash_embedding_gb300 as geng
import oracle
import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_plain_c_client(tmp_path):
    geng.build()
    pkg = os.path.dirname(geng.library_path())
    exe = tmp_path / "engram_client"
    subprocess.check_call(["gcc", "-std=c99", "-O1", "-Wall", "-o", str(exe),
                           os.path.join(ROOT, "tests", "c_client", "engram_client.c"),
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                           "-L", pkg, "-lengram", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                           f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"])
    wl = synth.make_workload(0, full64=True)
    lay = wl.layout
    B, L = 2, 40
    ids = synth.uniform_int(5, synth.TAG_IDS, B * L, 0, lay.raw_vocab).reshape(B, L)
    start = np.array([0, 3], dtype=np.int32)
    rows = lay.rows[0]
    W = synth.table_rows(wl.table_seed, 0, np.arange(rows), lay.head_dim)
    S = synth.table_scales(wl.table_seed, 0, np.arange(rows), lay.n_scales)
    d = tmp_path
    np.array([lay.n_layers, lay.max_ngram, lay.n_heads, lay.head_dim, lay.block, B, 64, lay.dead, lay.pad_id, B, L],
             dtype=np.int64).tofile(d / "layout.bin")
    for name, a in (("token_map", lay.token_map), ("multipliers", lay.multipliers), ("primes", lay.primes),
                    ("offsets", lay.offsets), ("ids", ids)):
        np.ascontiguousarray(a, dtype=np.int64).tofile(d / f"{name}.bin")
    start.tofile(d / "start.bin")
    W.tofile(d / "W.bin")
    S.tofile(d / "S.bin")
    K, N = lay.n_cols * lay.head_dim, 64
    rng = np.random.default_rng(6)
    wkv = (rng.standard_normal((N, K)) * K ** -0.5).astype(np.float32)
    wkv_bits = (wkv.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16: any bf16 weights will do
    wkv_bits.tofile(d / "wkv.bin")
    r = subprocess.run([str(exe), str(d)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
    C = lay.n_cols
    hashes = np.fromfile(d / "hashes.out", dtype=np.int64).reshape(B, L, lay.n_layers, C)
    orc = oracle.OracleState.from_layout(lay, B, 64)
    # the client's cache starts DEAD too; its rows sit at per-row starts 0 and 3 of cache rows B-1-b
    exp_h, _ = orc.hash(ids, start.astype(np.int64), cache_rows=np.arange(B)[::-1])
    assert np.array_equal(hashes, exp_h)
    exp_rows = oracle.engram_lookup(exp_h[:, :, 0, :], W, S, rows, lay.head_dim, lay.block)
    assert np.array_equal(np.fromfile(d / "rows0.out", dtype=np.uint16).reshape(exp_rows.shape), exp_rows)
    assert np.array_equal(np.fromfile(d / "lookup0.out", dtype=np.uint16).reshape(exp_rows.shape), exp_rows)
    assert int(np.fromfile(d / "status.out", dtype=np.uint32)[0]) == 0
    # the lookup inside the projection against the oracle chain (tolerance of tests/test_gpu_project.py)
    assert int(np.fromfile(d / "device_status.out", dtype=np.uint32)[0]) == 0
    got = np.fromfile(d / "kv0.out", dtype=np.uint16).reshape(B * L, N)
    emb = exp_rows.reshape(B * L, K)
    exp = oracle.engram_linear(emb, wkv_bits)
    e64, g64 = oracle.bf16_bits_to_f64(exp), oracle.bf16_bits_to_f64(got)
    abs_sum = np.abs(oracle.bf16_bits_to_f64(emb)) @ np.abs(oracle.bf16_bits_to_f64(wkv_bits)).T
    tol = 2.0 ** -7 * (1 + 2.0 ** -7) * np.abs(e64) + 2.0 * (K - 1) * 2.0 ** -23 * abs_sum + 2.0 ** -133
    assert not (np.abs(g64 - e64) > tol).any()
