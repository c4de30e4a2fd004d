"""CPU oracle for the Engram n-gram hash and the fp8 row lookup.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The product library never
calls it, and it shares no code with the CUDA path.

``engram_oracle.c`` is a plain restatement of the "DeepSeek V4.1" pages
(blocks/stack-hashes page: the n-gram hash ``forward``; engram-first/lookup
page: ``ParallelEngramEmbedding.forward``). This module compiles it with gcc and
calls it through ctypes. The ``Engram`` gate and its ``wkv`` projection
(blocks/stack-hashes page, ``Engram.forward``) are restated below in numpy,
in float64.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, invariants, library reductions, the released table
sizes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "engram_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FLAG_BAD_START = 1
FLAG_BAD_ID = 2
FLAG_BAD_ROW = 8


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle (portable C, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-o", out + ".tmp",
           src, "-lm"]
    subprocess.check_call(cmd)
    os.replace(out + ".tmp", out)
    return out


_P = ctypes.c_void_p
_I = ctypes.c_int64


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_fp8_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_fp8_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_floor_mod.argtypes = [_I, _I]
    lib.oracle_floor_mod.restype = _I
    lib.oracle_engram_hash.argtypes = [_I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _P,
                                       _P]
    lib.oracle_engram_hash.restype = ctypes.c_int
    lib.oracle_engram_hash_varlen.argtypes = [_I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P,
                                              _I, _P, _P]
    lib.oracle_engram_hash_varlen.restype = ctypes.c_int
    lib.oracle_engram_lookup.argtypes = [_P, _I, _P, _P, _I, _I, _I, _I, _P]
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_e8m0_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_to_f32.restype = ctypes.c_float
    lib.oracle_engram_lookup.restype = ctypes.c_int
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


def load_variant(path: str):
    """Bind another build of the same source (used to check that the pins catch planted mistakes)."""
    return _bind(path)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def fp8_e4m3_to_f32(code: int, L=None) -> float:
    return (L or lib()).oracle_fp8_e4m3_to_f32(code)


def bf16_rne(x: float, L=None) -> int:
    return (L or lib()).oracle_bf16_rne(x)


def floor_mod(x: int, p: int, L=None) -> int:
    return (L or lib()).oracle_floor_mod(x, p)


class OracleState:
    """The hash module's parameters plus its compressed-token cache (int64, starts DEAD)."""

    def __init__(self, n_layers, max_ngram, n_heads, token_map, multipliers, primes, offsets, dead, pad_id,
                 max_batch, max_seq_len, L=None):
        self.lib = L or lib()
        self.n_layers, self.max_ngram, self.n_heads = int(n_layers), int(max_ngram), int(n_heads)
        self.n_cols = (self.max_ngram - 1) * self.n_heads
        self.token_map = np.ascontiguousarray(token_map, dtype=np.int64)
        self.multipliers = np.ascontiguousarray(multipliers, dtype=np.int64).reshape(self.n_layers, self.max_ngram)
        self.primes = np.ascontiguousarray(primes, dtype=np.int64).reshape(self.n_layers, self.max_ngram - 1,
                                                                           self.n_heads)
        self.offsets = np.ascontiguousarray(offsets, dtype=np.int64).reshape(self.n_layers, self.n_cols)
        self.dead, self.pad_id = int(dead), int(pad_id)
        self.max_batch, self.max_seq_len = int(max_batch), int(max_seq_len)
        self.cache = np.full((self.max_batch, self.max_seq_len), self.dead, dtype=np.int64)

    @classmethod
    def from_layout(cls, lay, max_batch, max_seq_len, L=None):
        return cls(lay.n_layers, lay.max_ngram, lay.n_heads, lay.token_map, lay.multipliers, lay.primes, lay.offsets,
                   lay.dead, lay.pad_id, max_batch, max_seq_len, L)

    def reset(self):
        self.cache[:] = self.dead

    def hash(self, ids, start_pos, mask=None, cache_rows=None):
        """ids int64 [B, L]; start_pos int or [B]; mask bool [B, L] or None; cache_rows [B] or None
        (row b uses cache row cache_rows[b], else b). Returns (hashes int64 [B, L, n_layers, C], flags)."""
        ids = np.ascontiguousarray(ids, dtype=np.int64)
        B, L = ids.shape
        sp = np.ascontiguousarray(np.broadcast_to(np.asarray(start_pos, dtype=np.int64), (B,)))
        m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
        cr = None if cache_rows is None else np.ascontiguousarray(cache_rows, dtype=np.int64).reshape(B)
        out = np.empty((B, L, self.n_layers, self.n_cols), dtype=np.int64)
        flags = ctypes.c_uint32(0)
        rc = self.lib.oracle_engram_hash(
            self.n_layers, self.max_ngram, self.n_heads, _ptr(self.token_map), self.token_map.size, self.dead,
            self.pad_id, _ptr(self.multipliers), _ptr(self.primes), _ptr(self.offsets), _ptr(self.cache),
            self.max_batch, self.max_seq_len, _ptr(ids), _ptr(m), _ptr(sp), _ptr(cr), B, L, _ptr(out),
            ctypes.byref(flags))
        if rc != 0:
            raise ValueError(f"oracle_engram_hash rejected its arguments ({rc})")
        return out, flags.value


    def hash_varlen(self, ids, cu_seqlens, start_pos, mask=None, cache_rows=None):
        """Packed sequences: ids int64 [T]; cu_seqlens [B+1]; start_pos [B]; mask bool [T] or None.
        Sequence b uses cache row b (or cache_rows[b]). Returns (hashes int64 [T, n_layers, C], flags)."""
        ids = np.ascontiguousarray(ids, dtype=np.int64).reshape(-1)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64).reshape(-1)
        B = cu.size - 1
        sp = np.ascontiguousarray(np.broadcast_to(np.asarray(start_pos, dtype=np.int64), (B,)))
        m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8).reshape(-1)
        cr = None if cache_rows is None else np.ascontiguousarray(cache_rows, dtype=np.int64).reshape(B)
        out = np.empty((ids.size, self.n_layers, self.n_cols), dtype=np.int64)
        flags = ctypes.c_uint32(0)
        rc = self.lib.oracle_engram_hash_varlen(
            self.n_layers, self.max_ngram, self.n_heads, _ptr(self.token_map), self.token_map.size, self.dead,
            self.pad_id, _ptr(self.multipliers), _ptr(self.primes), _ptr(self.offsets), _ptr(self.cache),
            self.max_batch, self.max_seq_len, _ptr(ids), _ptr(m), _ptr(cu), _ptr(sp), _ptr(cr), B, _ptr(out),
            ctypes.byref(flags))
        if rc != 0:
            raise ValueError(f"oracle_engram_hash_varlen rejected its arguments ({rc})")
        return out, flags.value


SCALE_F32, SCALE_BF16, SCALE_E8M0, SCALE_E4M3 = 0, 1, 2, 3
_SCALE_STORAGE = {SCALE_F32: np.float32, SCALE_BF16: np.uint16, SCALE_E8M0: np.uint8, SCALE_E4M3: np.uint8}


def bf16_to_f32(h: int, L=None) -> float:
    return (L or lib()).oracle_bf16_to_f32(h)


def e8m0_to_f32(e: int, L=None) -> float:
    return (L or lib()).oracle_e8m0_to_f32(e)


def engram_lookup(idx, W, S, rows, D, block, L=None, scale_dtype=SCALE_F32) -> np.ndarray:
    """idx int64 [...]; W uint8 [rows, D]; S [rows, D/block] stored as scale_dtype (float32 values, or
    the uint16 bits of bf16, or the uint8 codes of UE8M0 / E4M3). Returns bf16 bits uint16 [..., D]."""
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=_SCALE_STORAGE[scale_dtype])
    out = np.empty(idx.shape + (D,), dtype=np.uint16)
    rc = (L or lib()).oracle_engram_lookup(_ptr(idx), idx.size, _ptr(W), _ptr(S), int(rows), int(D), int(block),
                                           int(scale_dtype), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_engram_lookup rejected its arguments ({rc})")
    return out


# ----------------------------------------------------------------------------- Engram gate (float64)
def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), straight from float64 (no float32 step).
    Finite inputs only; values beyond the bf16 range become infinities."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    sign = np.signbit(x)
    a = np.abs(x)
    nz = a > 0
    m, e = np.frexp(np.where(nz, a, 1.0))  # a = m * 2^e, m in [0.5, 1)
    # bf16 keeps 8 significant bits; below the normal range (2^-126) the step is fixed at 2^-133
    q = np.where(e - 1 >= -126, np.ldexp(np.rint(np.ldexp(m, 8)), e - 8), np.ldexp(np.rint(np.ldexp(a, 133)), -133))
    q = np.where(nz, q, 0.0)
    f = q.astype(np.float32)  # exact: q has at most 8 significant bits (or overflows to inf)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out[...] = np.where(sign, bits | np.uint16(0x8000), bits)
    return out


def engram_linear(emb_bits, w_bits) -> np.ndarray:
    """The `wkv` projection of the Engram block on bf16 inputs: exact float64 products and sums,
    rounded once to bf16. emb [T, K], w [N, K] (bf16 bits) -> kv bits [T, N]."""
    e = bf16_bits_to_f64(emb_bits)
    w = bf16_bits_to_f64(w_bits)
    return f64_to_bf16_bits(e @ w.T)


def engram_gate(x_bits, kv_bits, qw_bits, kw_bits, mask=None, eps=1e-20, clamp=1e-6) -> np.ndarray:
    """`Engram.forward` after the projection (blocks/stack-hashes page), in float64:
    x [T, hc, dim] (the residual copies), kv [T, (hc+1)*dim] = hc keys then one shared value,
    q_weight / k_weight [hc, dim], mask [T] (False closes the gate). Returns the float64 result
    h + gate * value, [T, hc, dim], before its conversion to x's dtype."""
    h = bf16_bits_to_f64(x_bits)
    T, hc, dim = h.shape
    kv = bf16_bits_to_f64(kv_bits).reshape(T, hc + 1, dim)
    key, value = kv[:, :hc, :], kv[:, hc, :]
    weight = bf16_bits_to_f64(qw_bits) * bf16_bits_to_f64(kw_bits)            # [hc, dim]
    # normalized per (token, hc copy) over dim
    rstd = 1.0 / np.sqrt((h * h).mean(-1) + eps) / np.sqrt((key * key).mean(-1) + eps)
    dot = (h * weight[None] * key).sum(-1) * rstd * dim ** -0.5              # [T, hc]
    signed_sqrt = np.copysign(np.sqrt(np.maximum(np.abs(dot), clamp)), dot)
    gate = 1.0 / (1.0 + np.exp(-signed_sqrt))
    if mask is not None:
        gate = np.where(np.asarray(mask, dtype=bool)[:, None], gate, 0.0)
    return h + gate[..., None] * value[:, None, :]
