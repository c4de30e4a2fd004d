"""Shared plumbing of the GPU parity tests: device tables from the seeded generator,
oracle evaluation on the rows a test touches, bit-level comparison."""
from __future__ import annotations

import numpy as np
import torch

import gram_hash_embedding_gb300 as geng
import oracle
import synth


def build_all():
    geng.build()
    synth.build()
    oracle.build()


def make_state(wl: synth.Workload, max_batch=None, max_seq_len=None) -> geng.EngramHash:
    lay = wl.layout
    return geng.EngramHash(n_layers=lay.n_layers, max_ngram=lay.max_ngram, n_heads=lay.n_heads,
                           head_dim=lay.head_dim, block=lay.block, max_batch=max_batch or wl.max_batch,
                           max_seq_len=max_seq_len or wl.max_seq_len, token_map=lay.token_map,
                           multipliers=lay.multipliers, primes=lay.primes, offsets=lay.offsets, dead=lay.dead,
                           pad_id=lay.pad_id, scale_dtype=lay.scale_dtype)


def make_oracle(wl: synth.Workload, max_batch=None, max_seq_len=None) -> oracle.OracleState:
    return oracle.OracleState.from_layout(wl.layout, max_batch or wl.max_batch, max_seq_len or wl.max_seq_len)


SCALE_TORCH_DTYPE = {synth.SCALE_F32: torch.float32, synth.SCALE_BF16: torch.bfloat16,
                     synth.SCALE_E8M0: getattr(torch, "float8_e8m0fnu", None), synth.SCALE_E4M3: torch.float8_e4m3fn}


def device_tables(wl: synth.Workload, device="cuda"):
    """Per-layer fp8 tables and scales (in the layout's scale storage type), filled on the device by
    the counter-based generator."""
    lay = wl.layout
    Ws, Ss = [], []
    for l, rows in enumerate(lay.rows):
        W = torch.empty((rows, lay.head_dim), dtype=torch.uint8, device=device)
        S = torch.empty((rows, lay.n_scales), dtype=SCALE_TORCH_DTYPE[lay.scale_dtype], device=device)
        synth.fill_table_device(W, S, wl.table_seed, l, lay.scale_dtype)
        Ws.append(W)
        Ss.append(S)
    torch.cuda.synchronize()
    return Ws, Ss


def oracle_lookup_rows(wl: synth.Workload, layer: int, idx: np.ndarray) -> np.ndarray:
    """Oracle lookup of the given table indices of one layer. Only the rows touched are
    generated on the host (same generator as the device table), as a compact table;
    indices outside [0, rows) stay out of range there."""
    lay = wl.layout
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    valid = (flat >= 0) & (flat < lay.rows[layer])
    uniq, inv = np.unique(flat[valid], return_inverse=True)
    W = synth.table_rows(wl.table_seed, layer, uniq, lay.head_dim)
    S = synth.table_scales(wl.table_seed, layer, uniq, lay.n_scales, lay.scale_dtype)
    local = np.full(flat.shape, -1, dtype=np.int64)
    local[valid] = inv
    out = oracle.engram_lookup(local, W, S, len(uniq), lay.head_dim, lay.block, scale_dtype=lay.scale_dtype)
    return out.reshape(np.asarray(idx).shape + (lay.head_dim,))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bits_equal(got: np.ndarray, exp: np.ndarray, what: str):
    got = np.asarray(got)
    exp = np.asarray(exp)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    bad = got != exp
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} differ; first at {tuple(i)}: "
                             f"got {got[tuple(i)]!r} expected {exp[tuple(i)]!r}")


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()
