"""Seeded synthetic inputs for the Engram n-gram hash + fp8 lookup workloads.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It holds generators only: it computes no hash, no modulo reduction into
buckets, no fp8 decode and no dequantisation. Everything it makes is an *input*
of the method (token ids, masks, start positions, the token map, the hash
multipliers, the bucket primes and their offsets, the fp8 table and its
scales).

Counter-based generator (one definition, used on host and device)
-----------------------------------------------------------------
``mix64`` is the splitmix64 output function (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; constants as in
Vigna's public-domain splitmix64.c)::

    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31

A stream is keyed by ``(seed, tag)``::

    base       = mix64(seed ^ (tag * 0xD1B54A32D192ED03))
    word(ctr)  = mix64(base + (ctr + 1) * 0x9E3779B97F4A7C15)      (all mod 2^64)

The fp8 table of layer ``l`` is the flat byte stream of tag ``TAG_TABLE + l``:
byte ``4*g + j`` of the table is ``lut[(word(g) >> 16*j) & 0xFFFF]``, so row
``r`` of a ``[rows, D]`` table is words ``r*D/4 .. (r+1)*D/4 - 1``. ``lut`` maps
a 16-bit uniform to the E4M3 code of the standard normal quantile
``Phi^-1((u + 0.5) / 65536)`` (rounded by torch's float->float8_e4m3fn cast), so
codes follow N(0,1) and never take the NaN codes 0x7F/0xFF.

The fp32 scale ``f`` (flat index ``r*(D/block) + k``) of layer ``l`` comes from
tag ``TAG_SCALE + l``: ``0.01f + 0.99f * ((word(f) >> 40) * 2^-24)``, each
operation a single fp32 round-to-nearest step, i.e. uniform on [0.01, 1).

The device side of these two fills lives in ``synth/fill.cu`` and is checked
against :func:`table_rows` / :func:`table_scales` bit for bit.
"""
from __future__ import annotations

import ctypes
import math
import os
import statistics
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libengram_synth.so")

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
TAG_MUL = 0xD1B54A32D192ED03

# stream tags
TAG_TOKEN_MAP = 1
TAG_IDS = 2
TAG_MULTIPLIERS = 3
TAG_PRIME_PICK = 4
TAG_SPANS = 5
TAG_START = 6
TAG_SAMPLE = 7
TAG_TABLE = 100
TAG_SCALE = 200

# the pages' vocabulary facts (DeepSeek V4.1 config: vocab_size, image_token_id,
# engram_compressed_vocab_size, engram_pad_id, engram_vocab_size)
RAW_VOCAB = 129280
IMAGE_TOKEN_ID = 129264
COMPRESSED_VOCAB = 99092
PAD_ID = 2
DEAD = -1
FULL_SCALE_PRIME_START = 16_000_000


# ----------------------------------------------------------------------------- generator
def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wraps mod 2^64)."""
    z = np.asarray(z, dtype=np.uint64).copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def _mix64_int(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z


def stream_base(seed: int, tag: int) -> int:
    """Key of the stream ``(seed, tag)`` as a Python int in [0, 2^64)."""
    return _mix64_int((seed & MASK64) ^ ((tag * TAG_MUL) & MASK64))


def words(seed: int, tag: int, counters) -> np.ndarray:
    """``word(ctr)`` of stream ``(seed, tag)`` for every counter (uint64 array)."""
    c = np.asarray(counters, dtype=np.uint64)
    base = np.uint64(stream_base(seed, tag))
    with np.errstate(over="ignore"):
        z = base + (c + np.uint64(1)) * np.uint64(GOLDEN)
    return mix64(z)


def uniform01(seed: int, tag: int, counters) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of each word."""
    w = words(seed, tag, counters)
    return (w >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_int(seed: int, tag: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """n integers in [lo, hi) (modulo of a 64-bit word; bias below 2^-40 here)."""
    w = words(seed, tag, np.arange(offset, offset + n, dtype=np.uint64))
    return (w % np.uint64(hi - lo)).astype(np.int64) + lo


# ----------------------------------------------------------------------------- token-level inputs
def token_map(seed: int, raw_vocab: int = RAW_VOCAB, compressed_vocab: int = COMPRESSED_VOCAB) -> np.ndarray:
    """A seeded stand-in for the tokenizer's compression map: raw id -> [0, compressed_vocab)."""
    return uniform_int(seed, TAG_TOKEN_MAP, raw_vocab, 0, compressed_vocab)


def uniform_ids(seed: int, n: int, vocab: int = RAW_VOCAB, offset: int = 0) -> np.ndarray:
    return uniform_int(seed, TAG_IDS, n, 0, vocab, offset)


_ZIPF_CACHE: dict = {}


def zipf_ids(seed: int, n: int, vocab: int = RAW_VOCAB, s: float = 1.1, offset: int = 0, tag: int = TAG_IDS) -> np.ndarray:
    """Zipf(s) over ``vocab`` ids: rank k (1-based) has weight k^-s and maps to id k-1.

    Sampled by inverse CDF: a host table of cumulative weights (double), searched
    with the 53-bit uniform of each counter."""
    key = (vocab, s)
    if key not in _ZIPF_CACHE:
        w = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
        cdf = np.cumsum(w)
        _ZIPF_CACHE[key] = cdf / cdf[-1]
    cdf = _ZIPF_CACHE[key]
    u = uniform01(seed, tag, np.arange(offset, offset + n, dtype=np.uint64))
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int64)


def image_span_mask(seed: int, length: int, frac: float, lo: int = 64, hi: int = 1024,
                    stream: int = 0) -> np.ndarray:
    """Token mask of one sequence: False inside non-overlapping contiguous "image" spans.

    Span lengths are uniform in [lo, hi] (the last one trimmed) until exactly
    round(frac * length) tokens are covered; the remaining free positions are
    split into seeded gaps before, between and after the spans."""
    mask = np.ones(length, dtype=bool)
    target = min(length, int(round(frac * length)))
    if target <= 0:
        return mask
    ctr = stream * 1_000_003
    spans, covered = [], 0
    while covered < target:
        w = int(words(seed, TAG_SPANS, [ctr])[0])
        ctr += 1
        span = min(lo + w % (hi - lo + 1), target - covered)
        spans.append(span)
        covered += span
    free = length - target
    cuts = np.sort(words(seed, TAG_SPANS, np.arange(ctr, ctr + len(spans), dtype=np.uint64)) % np.uint64(free + 1))
    pos = 0
    for cut, span in zip(cuts.astype(np.int64), spans):
        start = int(cut) + pos
        mask[start:start + span] = False
        pos += span
    return mask


# ----------------------------------------------------------------------------- layout parameters
def multipliers(seed: int, n_layers: int, max_ngram: int, full64: bool = False) -> np.ndarray:
    """Hash multipliers [n_layers, max_ngram]: seeded odd values in [1, 2^31).

    ``full64`` gives full 64-bit odd values instead (stored as int64, so about
    half are negative), which makes the products wrap mod 2^64."""
    n = n_layers * max_ngram
    w = words(seed, TAG_MULTIPLIERS, np.arange(n, dtype=np.uint64))
    if full64:
        m = (w | np.uint64(1)).view(np.int64)
    else:
        m = ((w >> np.uint64(34)) << np.uint64(1)) | np.uint64(1)  # 30 bits, then odd: [1, 2^31)
        m = m.astype(np.int64)
    return m.reshape(n_layers, max_ngram)


def _is_prime(v: int) -> bool:
    """Deterministic Miller-Rabin for v < 3.3e24 (bases: first 12 primes)."""
    if v < 2:
        return False
    small = (2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37)
    for p in small:
        if v % p == 0:
            return v == p
    d, r = v - 1, 0
    while d % 2 == 0:
        d //= 2
        r += 1
    for a in small:
        x = pow(a, d, v)
        if x in (1, v - 1):
            continue
        for _ in range(r - 1):
            x = x * x % v
            if x == v - 1:
                break
        else:
            return False
    return True


def primes_after(start: int, count: int) -> list:
    """The ``count`` consecutive primes greater than ``start``, ascending."""
    out, v = [], start + 1
    while len(out) < count:
        if _is_prime(v):
            out.append(v)
        v += 1
    return out


def layered_primes(start: int, n_layers: int, max_ngram: int, n_heads: int) -> np.ndarray:
    """Bucket primes [n_layers, max_ngram-1, n_heads].

    The n_layers*(max_ngram-1)*n_heads consecutive primes above ``start`` are
    dealt in ascending order to (layer, n-gram size, head), layer slowest. With
    start 16,000,000 and 2 x 3 x 8 this reproduces the released table sizes."""
    n = n_layers * (max_ngram - 1) * n_heads
    return np.array(primes_after(start, n), dtype=np.int64).reshape(n_layers, max_ngram - 1, n_heads)


def distinct_primes_in(seed: int, lo: int, hi: int, shape) -> np.ndarray:
    """Seeded distinct primes from [lo, hi], in the order drawn."""
    pool = [v for v in range(lo, hi + 1) if _is_prime(v)]
    n = int(np.prod(shape))
    keys = words(seed, TAG_PRIME_PICK, np.arange(len(pool), dtype=np.uint64))
    order = np.argsort(keys, kind="stable")
    return np.array([pool[i] for i in order[:n]], dtype=np.int64).reshape(shape)


def column_offsets(primes: np.ndarray) -> np.ndarray:
    """Offsets [n_layers, C]: exclusive prefix sums of each layer's primes in column order,
    column = (n-2)*n_heads + head for n-gram size n, so the columns tile [0, sum)."""
    n_layers = primes.shape[0]
    flat = primes.reshape(n_layers, -1).astype(np.int64)
    return np.concatenate([np.zeros((n_layers, 1), np.int64), np.cumsum(flat, axis=1)[:, :-1]], axis=1)


# ----------------------------------------------------------------------------- fp8 table + scales
_LUT = None


def fp8_normal_lut() -> np.ndarray:
    """uint8[65536]: 16-bit uniform -> E4M3 code of the N(0,1) quantile (clipped to +-448)."""
    global _LUT
    if _LUT is None:
        import torch

        nd = statistics.NormalDist()
        x = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)], dtype=np.float64)
        x = np.clip(x, -448.0, 448.0)
        codes = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        _LUT = codes.copy()
    return _LUT


def table_rows(seed: int, layer: int, rows, D: int) -> np.ndarray:
    """fp8 codes of the given rows of layer ``layer``'s table: uint8 [len(rows), D]."""
    assert D % 4 == 0
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1)
    wpr = D // 4
    ctr = (rows[:, None] * np.uint64(wpr) + np.arange(wpr, dtype=np.uint64)[None, :]).reshape(-1)
    w = words(seed, TAG_TABLE + layer, ctr)
    lut = fp8_normal_lut()
    # piece j of a word is bits [16j, 16j+16): on a little-endian host, uint16 element j of its view
    pieces = w.astype("<u8", copy=False).view("<u2")
    return lut[pieces].reshape(rows.size, D)


# scale storage types (the same numbering as the library's and the oracle's, defined here on its own)
SCALE_F32, SCALE_BF16, SCALE_E8M0, SCALE_E4M3 = 0, 1, 2, 3
SCALE_BYTES = {SCALE_F32: 4, SCALE_BF16: 2, SCALE_E8M0: 1, SCALE_E4M3: 1}


def scale_codes(w: np.ndarray, scale_dtype: int) -> np.ndarray:
    """Scale bit patterns straight from generator words (integer operations only, so host and device
    agree by construction): bf16 with exponent 2^-7..2^0 and 7 random mantissa bits; UE8M0
    exponents 120..127 (2^-7..1); positive normal E4M3 codes with exponent 2^-3..2^0."""
    w = np.asarray(w, dtype=np.uint64)
    if scale_dtype == SCALE_BF16:
        return (((np.uint64(120) + (w & np.uint64(7))) << np.uint64(7)) | ((w >> np.uint64(8)) & np.uint64(0x7F))
                ).astype(np.uint16)
    if scale_dtype == SCALE_E8M0:
        return (np.uint64(120) + (w & np.uint64(7))).astype(np.uint8)
    if scale_dtype == SCALE_E4M3:
        return (((np.uint64(4) + (w & np.uint64(3))) << np.uint64(3)) | ((w >> np.uint64(8)) & np.uint64(7))
                ).astype(np.uint8)
    raise ValueError(scale_dtype)


def table_scales(seed: int, layer: int, rows, n_scales: int, scale_dtype: int = SCALE_F32) -> np.ndarray:
    """Scales of the given rows, [len(rows), n_scales]: fp32 values uniform on [0.01, 1), or the bit
    patterns of the other storage types (`scale_codes`)."""
    rows = np.asarray(rows, dtype=np.uint64).reshape(-1)
    ctr = (rows[:, None] * np.uint64(n_scales) + np.arange(n_scales, dtype=np.uint64)[None, :]).reshape(-1)
    w = words(seed, TAG_SCALE + layer, ctr)
    if scale_dtype != SCALE_F32:
        return scale_codes(w, scale_dtype).reshape(rows.size, n_scales)
    t = (w >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    s = np.float32(0.01) + np.float32(0.99) * t
    return s.astype(np.float32).reshape(rows.size, n_scales)


# ----------------------------------------------------------------------------- device fill (ctypes)
def build(force: bool = False) -> str:
    """Compile ``fill.cu`` into ``libengram_synth.so`` next to it (sm_103a)."""
    src = os.path.join(_HERE, "fill.cu")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-shared",
           "-Xcompiler", "-fPIC", "-o", _LIB_PATH + ".tmp", src]
    subprocess.check_call(cmd)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("synth device library not built: call synth.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_fill_fp8.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_fill_fp8.restype = ctypes.c_int
        lib.synth_fill_scales.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_fill_scales.restype = ctypes.c_int
        lib.synth_fill_scale_codes.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int,
                                               ctypes.c_void_p]
        lib.synth_fill_scale_codes.restype = ctypes.c_int
        _lib = lib
    return _lib


_LUT_DEV: dict = {}


def fill_table_device(W, S, seed: int, layer: int, scale_dtype: int = SCALE_F32) -> None:
    """Fill device tensors W (uint8 [rows, D]) and S ([rows, n_scales]: float32, or any tensor of the
    storage type's width for the other scale types) with layer ``layer``'s table from the
    counter-based generator, on torch's current stream."""
    import torch

    lib = _load()
    dev = W.device
    if dev not in _LUT_DEV:
        _LUT_DEV[dev] = torch.from_numpy(fp8_normal_lut()).to(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    assert W.dtype == torch.uint8 and W.is_contiguous() and W.numel() % 16 == 0
    assert S.element_size() == SCALE_BYTES[scale_dtype] and S.is_contiguous()
    assert scale_dtype != SCALE_F32 or S.dtype == torch.float32
    rc = lib.synth_fill_fp8(W.data_ptr(), W.numel(), stream_base(seed, TAG_TABLE + layer), _LUT_DEV[dev].data_ptr(), stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_fp8 failed: {rc}")
    if scale_dtype == SCALE_F32:
        rc = lib.synth_fill_scales(S.data_ptr(), S.numel(), stream_base(seed, TAG_SCALE + layer), stream)
    else:
        rc = lib.synth_fill_scale_codes(S.data_ptr(), S.numel(), stream_base(seed, TAG_SCALE + layer), scale_dtype,
                                        stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_scales failed: {rc}")


# ----------------------------------------------------------------------------- workloads
@dataclass
class Layout:
    """The hash module's parameters (the pages leave their values open)."""
    n_layers: int
    max_ngram: int
    n_heads: int
    head_dim: int
    block: int
    raw_vocab: int
    compressed_vocab: int
    token_map: np.ndarray
    multipliers: np.ndarray
    primes: np.ndarray
    offsets: np.ndarray
    dead: int = DEAD
    pad_id: int = PAD_ID
    scale_dtype: int = SCALE_F32  # storage type of the scale tensors (SCALE_*)

    @property
    def n_cols(self) -> int:
        return (self.max_ngram - 1) * self.n_heads

    @property
    def rows(self) -> list:
        return [int(self.primes[l].sum()) for l in range(self.n_layers)]

    @property
    def n_scales(self) -> int:
        return self.head_dim // self.block

    @property
    def scale_bytes(self) -> int:
        return SCALE_BYTES[self.scale_dtype]


@dataclass
class Workload:
    """One seeded configuration: layout, token-level inputs and table seed."""
    name: str
    layout: Layout
    B: int
    L: int
    ids: np.ndarray            # int64 [B, L] (or [chunks, B, L] for chunked runs)
    mask: np.ndarray | None    # bool like ids, or None
    start_pos: np.ndarray      # int32 [B] (or [chunks, B])
    table_seed: int
    max_batch: int
    max_seq_len: int
    prefill_ids: np.ndarray | None = None   # decode: int64 [B, P] written first at start 0
    chunks: int = 1
    extra: dict = field(default_factory=dict)


MASTER_SEED = 20261202


def make_layout(kind: str, seed: int, full64: bool = False) -> Layout:
    if kind == "tiny":
        tm = uniform_int(seed, TAG_TOKEN_MAP, 1000, 0, 800)
        primes = distinct_primes_in(seed, 997, 2003, (1, 3, 2))
        return Layout(1, 4, 2, 32, 32, 1000, 800, tm, multipliers(seed, 1, 4, full64), primes,
                      column_offsets(primes))
    if kind == "prefill":   # primes about 1e6: ~24M rows per layer
        primes = layered_primes(1_000_000, 2, 4, 8)
    elif kind == "full":    # the released table sizes
        primes = layered_primes(FULL_SCALE_PRIME_START, 2, 4, 8)
    elif kind == "profile":  # same shapes, ~0.5 GB per layer: small enough for a full ncu capture
        primes = layered_primes(160_000, 2, 4, 8)
    elif kind in ("full256", "full256e8"):  # the released table sizes and head_dim (2 scales per row)
        primes = layered_primes(FULL_SCALE_PRIME_START, 2, 4, 8)
        return Layout(2, 4, 8, 256, 128, RAW_VOCAB, COMPRESSED_VOCAB, token_map(seed), multipliers(seed, 2, 4, full64),
                      primes, column_offsets(primes),
                      scale_dtype=SCALE_E8M0 if kind == "full256e8" else SCALE_F32)
    else:
        raise ValueError(kind)
    return Layout(2, 4, 8, 128, 128, RAW_VOCAB, COMPRESSED_VOCAB, token_map(seed), multipliers(seed, 2, 4, full64),
                  primes, column_offsets(primes))


def make_workload(cfg: int, seed: int = MASTER_SEED, full64: bool = False) -> Workload:
    """The five seeded configurations (tiny, prefill, decode, full-scale, long chunked)."""
    s = seed + cfg
    if cfg == 0:
        lay = make_layout("tiny", s, full64)
        ids = uniform_int(s, TAG_IDS, 64, 0, 1000).reshape(1, 64)
        return Workload("tiny B1xL64", lay, 1, 64, ids, None, np.zeros(1, np.int32), s, 1, 64)
    if cfg == 1:
        lay = make_layout("prefill", s, full64)
        B, L = 4, 4096
        ids = uniform_ids(s, B * L).reshape(B, L)
        mask = np.stack([image_span_mask(s, L, 0.10, stream=b) for b in range(B)])
        ids = np.where(mask, ids, IMAGE_TOKEN_ID)
        return Workload("prefill B4xL4096", lay, B, L, ids, mask, np.zeros(B, np.int32), s, B, L)
    if cfg == 2:
        lay = make_layout("prefill", s, full64)
        B, P = 256, 8192
        pre = zipf_ids(s, B * P).reshape(B, P)
        start = uniform_int(s, TAG_START, B, 1, P + 1).astype(np.int32)
        ids = zipf_ids(s, B, offset=B * P).reshape(B, 1)
        # same tables as the prefill configuration (24M rows per layer)
        return Workload("decode B256xL1", lay, B, 1, ids, None, start, seed + 1, B, P + 1, prefill_ids=pre)
    if cfg == 3:
        lay = make_layout("full", s, full64)
        B, L = 8, 8192
        ids = uniform_ids(s, B * L).reshape(B, L)
        return Workload("full-scale B8xL8192", lay, B, L, ids, None, np.zeros(B, np.int32), s, B, L)
    if cfg == 4:
        lay = make_layout("full", s, full64)
        chunks, Lc = 8, 8192
        total = chunks * Lc
        ids = zipf_ids(s, total)
        mask = np.ones(total, dtype=bool)
        mask[:Lc] = image_span_mask(s, Lc, 0.15)
        ids = np.where(mask, ids, IMAGE_TOKEN_ID)
        # same full-scale tables as configuration 3
        return Workload("long chunked B1x65536 (8x8192)", lay, 1, Lc, ids.reshape(1, total), mask.reshape(1, total),
                        np.zeros(1, np.int32), seed + 3, 1, total, chunks=chunks)
    if cfg == 6:  # released head_dim: full-scale tables of 256 fp8 values per row (~197 GB + 6 GB of scales)
        lay = make_layout("full256", s, full64)
        B, L = 8, 8192
        ids = uniform_ids(s, B * L).reshape(B, L)
        return Workload("full-scale head_dim 256 B8xL8192", lay, B, L, ids, None, np.zeros(B, np.int32), s, B, L)
    if cfg == 8:  # released head_dim with power-of-two (UE8M0) scales: ~197 GB of codes + 1.5 GB of scales
        lay = make_layout("full256e8", s, full64)
        B, L = 8, 8192
        ids = uniform_ids(s, B * L).reshape(B, L)
        return Workload("full-scale head_dim 256 UE8M0 scales B8xL8192", lay, B, L, ids, None, np.zeros(B, np.int32),
                        s, B, L)
    if cfg == 7:  # continuous batching on the full-scale tables: 192 decode steps + 64 prefill chunks
        lay = make_layout("full", s, full64)
        B, P = 256, 8192
        is_prefill = np.zeros(B, dtype=bool)
        is_prefill[np.argsort(words(s, TAG_SAMPLE, np.arange(B, dtype=np.uint64)), kind="stable")[:64]] = True
        lens = np.where(is_prefill, uniform_int(s, TAG_SAMPLE, B, 64, 513, offset=100), 1).astype(np.int64)
        start = np.array([int(uniform_int(s, TAG_START, 1, 1, P - int(n) + 1, offset=b)[0]) for b, n in enumerate(lens)],
                         dtype=np.int32)
        ids = zipf_ids(s, int(lens.sum()), offset=B * P)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        pre = zipf_ids(s, B * P).reshape(B, P)
        return Workload("continuous batching 192 decode + 64 prefill (64-512) on full-scale tables", lay, B,
                        int(lens.max()), ids, None, start, seed + 3, B, P + 512, prefill_ids=pre,
                        extra={"cu_seqlens": cu, "lens": lens})
    if cfg == 5:  # profiling case: prefill shapes on ~1 GB of tables (still far above L2)
        lay = make_layout("profile", s, full64)
        B, L = 4, 4096
        ids = uniform_ids(s, B * L).reshape(B, L)
        return Workload("profile B4xL4096 (1 GB tables)", lay, B, L, ids, None, np.zeros(B, np.int32), s, B, L)
    raise ValueError(cfg)
