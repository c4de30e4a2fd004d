"""Engram n-gram hash + fp8 row lookup on GB300 (sm_103a): thin Python binding.

The work is done by ``libengram.so`` (CUDA kernels behind the C ABI declared in
``include/engram.h``). This module only marshals torch tensors into pointers,
sizes and the current CUDA stream; it has no compute path of its own and no
fallback: if the library is missing, every call raises.

Functions carry the C names: :func:`engram_state_create`,
:func:`engram_state_destroy`, :func:`engram_cache_reset`,
:func:`engram_state_status`, :func:`engram_hash`, :func:`engram_lookup`,
:func:`engram_hash_lookup` (and their packed forms), the Engram block after
the lookup (:func:`engram_project`, :func:`engram_gate`,
:func:`engram_project_gate`, and with the lookup inside the projection
:func:`engram_lookup_project`, :func:`engram_lookup_project_gate`), and the
row-sharded lookup's two ends (:func:`engram_shard_pack`,
:func:`engram_shard_unpack`). :class:`EngramHash` bundles a state with them.

Method: the "DeepSeek V4.1" pages -- blocks/stack-hashes page (the n-gram hash
``forward``, ``Engram.forward``) and engram-first/lookup page
(``ParallelEngramEmbedding.forward``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH
from ._build import build

__all__ = [
    "EngramError", "EngramHash", "build", "engram_state_create", "engram_state_destroy", "engram_cache_reset",
    "engram_state_status", "engram_hash", "engram_lookup", "engram_hash_lookup", "engram_hash_varlen",
    "engram_hash_lookup_varlen", "engram_gate", "PreparedHashLookup", "engram_strerror", "STATUS_BAD_START",
    "STATUS_BAD_ID", "STATUS_BAD_LENGTH", "STATUS_BAD_ROW", "STATUS_CHECK", "SCALE_F32", "SCALE_BF16", "SCALE_E8M0", "SCALE_E4M3",
    "library_path", "set_l2_fetch_granularity", "engram_project", "engram_project_gate",
    "engram_project_gate_workspace", "engram_device_status", "STATUS_TIMEOUT", "engram_shard_pack",
    "engram_shard_unpack", "shard_part", "sharded_lookup", "dist_exchange", "engram_lookup_project",
    "engram_lookup_project_workspace", "engram_lookup_project_gate", "engram_lookup_project_gate_workspace",
]

OK, ERR_INVALID, ERR_RANGE, ERR_CUDA, ERR_NOMEM, ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5
STATUS_BAD_START = 1
STATUS_BAD_ID = 2
STATUS_BAD_LENGTH = 4
STATUS_BAD_ROW = 8
STATUS_CHECK = 16  # checked builds only: a kernel skipped an access outside the call's buffers
STATUS_TIMEOUT = 32  # a tensor-core kernel gave up a wait (engram_device_status)
# storage types of the scale tensors (ENGRAM_SCALE_*)
SCALE_F32, SCALE_BF16, SCALE_E8M0, SCALE_E4M3 = 0, 1, 2, 3
_SCALE_BYTES = {SCALE_F32: 4, SCALE_BF16: 2, SCALE_E8M0: 1, SCALE_E4M3: 1}
_SCALE_OF_DTYPE = {torch.float32: SCALE_F32, torch.bfloat16: SCALE_BF16, torch.float8_e4m3fn: SCALE_E4M3}
if hasattr(torch, "float8_e8m0fnu"):
    _SCALE_OF_DTYPE[torch.float8_e8m0fnu] = SCALE_E8M0
MAX_LAYERS = 8


class EngramError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {engram_strerror(code)} ({code})")


class _Layout(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("max_ngram", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int64), ("raw_vocab", ctypes.c_int64), ("dead", ctypes.c_int64),
                ("pad_id", ctypes.c_int64), ("scale_dtype", ctypes.c_int32)]


class _Table(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("S", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("head_dim", ctypes.c_int32), ("block", ctypes.c_int32), ("scale_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_lib_handle = None


def library_path() -> str:
    return _LIB_PATH


def _lib():
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libengram.so is not built ({_LIB_PATH}); run gram_hash_embedding_gb300.build()")
        L = ctypes.CDLL(_LIB_PATH)
        L.engram_state_create.argtypes = [ctypes.POINTER(_Layout), _P, _P, _P, _P, _P, ctypes.POINTER(_P)]
        L.engram_state_destroy.argtypes = [_P]
        L.engram_cache_reset.argtypes = [_P, _P]
        L.engram_state_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.engram_hash.argtypes = [_P, _P, _P, _P, _P, _I32, _I64, _P, _P]
        L.engram_lookup.argtypes = [_P, _I64, _P, _P, _I64, _I32, _I32, _I32, _P, _P]
        L.engram_hash_lookup.argtypes = [_P, _P, _P, _P, _P, _I32, _I64, _P, _P, _P, _P, _P, _P]
        L.engram_hash_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _P, _P]
        L.engram_hash_lookup_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _P, _P, _P, _P, _P, _P]
        L.engram_state_layout.argtypes = [_P, ctypes.POINTER(_Layout)]
        L.engram_gate.argtypes = [_P, _P, _P, _P, _P, _I64, _I32, _I32, ctypes.c_float, _P, _P]
        L.engram_project.argtypes = [_P, _P, _I64, _I32, _I32, _P, _P]
        L.engram_project_gate_workspace.argtypes = [_I64, _I32, _I32]
        L.engram_project_gate_workspace.restype = ctypes.c_uint64
        L.engram_project_gate.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, ctypes.c_float, _P,
                                          ctypes.c_uint64, _P, _P]
        L.engram_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.engram_lookup_project_workspace.argtypes = [_I64, _I32, _I32]
        L.engram_lookup_project_workspace.restype = ctypes.c_uint64
        L.engram_lookup_project.argtypes = [_P, _I64, _I64, _I32, ctypes.POINTER(_Table), _P, _I32, _P,
                                            ctypes.c_uint64, _P, _P]
        L.engram_lookup_project_gate_workspace.argtypes = [_I64, _I32, _I32, _I32, _I32]
        L.engram_lookup_project_gate_workspace.restype = ctypes.c_uint64
        L.engram_lookup_project_gate.argtypes = [_P, _P, _I64, _I64, _I32, ctypes.POINTER(_Table), _P, _P, _P, _P,
                                                 _I32, _I32, ctypes.c_float, _P, ctypes.c_uint64, _P, _P]
        L.engram_shard_pack_workspace.argtypes = [_I64, _I32]
        L.engram_shard_pack_workspace.restype = ctypes.c_uint64
        L.engram_shard_pack.argtypes = [_P, _I64, _I64, _I32, _P, _P, _P, _P, ctypes.c_uint64, _P]
        L.engram_shard_unpack.argtypes = [_P, _P, _I64, _I64, _I32, _P, _P]
        L.engram_strerror.argtypes = [ctypes.c_int]
        L.engram_set_l2_fetch_granularity.argtypes = [_I32, ctypes.POINTER(_I32)]
        L.engram_strerror.restype = ctypes.c_char_p
        for name in ("engram_state_create", "engram_state_destroy", "engram_cache_reset", "engram_state_status",
                     "engram_hash", "engram_lookup", "engram_hash_lookup", "engram_state_layout",
                     "engram_hash_varlen", "engram_hash_lookup_varlen", "engram_gate", "engram_project",
                     "engram_project_gate", "engram_device_status", "engram_shard_pack", "engram_shard_unpack",
                     "engram_lookup_project", "engram_lookup_project_gate"):
            getattr(L, name).restype = ctypes.c_int
        _lib_handle = L
    return _lib_handle


def engram_strerror(code: int) -> str:
    return _lib().engram_strerror(int(code)).decode()


def _check(rc: int, where: str):
    if rc != OK:
        raise EngramError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _launch_stream(stream, temps=()) -> int:
    """The stream handle a call launches on. The wrapper's own temporaries (a start_pos array built
    from an int, outputs it allocates) are made on the current stream; when the caller names another
    stream, that stream first waits for the current one, and each temporary is marked as in use on it
    so the caching allocator does not hand its memory out again before the library's kernel is done."""
    cur = torch.cuda.current_stream()
    if stream is None:
        return cur.cuda_stream
    if not isinstance(stream, torch.cuda.Stream):
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        if handle == cur.cuda_stream:
            return handle
        stream = torch.cuda.ExternalStream(handle)
    if stream.cuda_stream != cur.cuda_stream:
        stream.wait_stream(cur)
        for t in temps:
            if isinstance(t, torch.Tensor):
                t.record_stream(stream)
    return stream.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host_i64(a, n: int, name: str):
    t = torch.as_tensor(a, dtype=torch.int64).reshape(-1).contiguous()
    if t.numel() != n:
        raise ValueError(f"{name}: expected {n} values, got {t.numel()}")
    return t


# ----------------------------------------------------------------------------- C-named functions
def engram_state_create(*, n_layers, max_ngram, n_heads, head_dim, block, max_batch, max_seq_len, token_map,
                        multipliers, primes, offsets, dead=-1, pad_id=2, stream=None, scale_dtype=SCALE_F32) -> int:
    """Create a state; returns the opaque handle (an int). Host arrays: token_map [raw_vocab],
    multipliers [n_layers, max_ngram], primes [n_layers, max_ngram-1, n_heads], offsets [n_layers, C].
    scale_dtype: storage type of the tables' scales (SCALE_*)."""
    tm = torch.as_tensor(token_map, dtype=torch.int64).reshape(-1).contiguous()
    C = (max_ngram - 1) * n_heads
    mu = _host_i64(multipliers, n_layers * max_ngram, "multipliers")
    pr = _host_i64(primes, n_layers * C, "primes")
    of = _host_i64(offsets, n_layers * C, "offsets")
    lay = _Layout(n_layers, max_ngram, n_heads, head_dim, block, max_batch, max_seq_len, tm.numel(), dead, pad_id,
                  int(scale_dtype))
    h = _P()
    _check(_lib().engram_state_create(ctypes.byref(lay), tm.data_ptr(), mu.data_ptr(), pr.data_ptr(), of.data_ptr(),
                                      _stream(stream), ctypes.byref(h)), "engram_state_create")
    return h.value


def engram_state_destroy(state: int) -> None:
    _check(_lib().engram_state_destroy(state), "engram_state_destroy")


def engram_cache_reset(state: int, stream=None) -> None:
    _check(_lib().engram_cache_reset(state, _stream(stream)), "engram_cache_reset")


def engram_state_status(state: int, clear: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib().engram_state_status(state, _stream(stream), ctypes.byref(v), int(bool(clear))),
           "engram_state_status")
    return v.value


def engram_state_layout(state: int) -> dict:
    lay = _Layout()
    _check(_lib().engram_state_layout(state, ctypes.byref(lay)), "engram_state_layout")
    return {f: getattr(lay, f) for f, _ in _Layout._fields_}


def _scale_dtype_of(S: torch.Tensor, scale_dtype=None) -> int:
    """The storage type of a scale tensor: given explicitly (then S may hold the raw bits in any
    dtype of that width), or read from S's dtype (float32, bfloat16, float8_e8m0fnu, float8_e4m3fn)."""
    if scale_dtype is not None:
        return int(scale_dtype)
    if S.dtype not in _SCALE_OF_DTYPE:
        raise TypeError(f"cannot tell the scale storage type of a {S.dtype} tensor; pass scale_dtype")
    return _SCALE_OF_DTYPE[S.dtype]


def _dev_scales(S: torch.Tensor, scale_dtype: int, name: str = "S") -> int:
    if not isinstance(S, torch.Tensor) or not S.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if scale_dtype not in _SCALE_BYTES or S.element_size() != _SCALE_BYTES[scale_dtype]:
        raise TypeError(f"{name}: {S.dtype} does not hold scales of storage type {scale_dtype}")
    if S.dtype in _SCALE_OF_DTYPE and _SCALE_OF_DTYPE[S.dtype] != scale_dtype:
        raise TypeError(f"{name} is {S.dtype} but the scales are stored as type {scale_dtype}")
    if not S.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return S.data_ptr()


def _start_tensor(start_pos, B: int, device) -> torch.Tensor:
    if isinstance(start_pos, torch.Tensor):
        return start_pos
    return torch.full((B,), int(start_pos), dtype=torch.int32, device=device)


def set_l2_fetch_granularity(nbytes: int) -> int:
    """Set the current device context's L2 fetch granularity limit (0, 32, 64 or 128 bytes; a hint)
    and return the previous value. Process-wide and not stream-ordered: call it at set-up. At 32 a
    random 4-byte scale read costs one 32-byte DRAM sector instead of a 128-byte line."""
    prev = _I32(0)
    _check(_lib().engram_set_l2_fetch_granularity(int(nbytes), ctypes.byref(prev)), "engram_set_l2_fetch_granularity")
    return prev.value


def _size(t, n: int, name: str) -> None:
    """Sizes are checked here, before any pointer reaches the library: the C calls take raw pointers
    and would read or write past a buffer that is too small."""
    if t is not None and isinstance(t, torch.Tensor) and t.numel() != n:
        raise ValueError(f"{name} has {t.numel()} elements, expected {n}")


def _tables(lay: dict, W: list, S: list, out: list | None, n_rows_out: int) -> None:
    """Per-layer tables of a fused call: one W, S (and out) per engram layer of the state, W [rows, D],
    S holding rows * D / block scales, out holding n_rows_out * C rows of D values."""
    n = lay["n_layers"]
    if len(W) != n or len(S) != n or (out is not None and len(out) != n):
        raise ValueError(f"W, S and out need one entry per engram layer ({n})")
    D, C = lay["head_dim"], (lay["max_ngram"] - 1) * lay["n_heads"]
    for l in range(n):
        if W[l].dim() != 2 or W[l].shape[1] != D:
            raise ValueError(f"W[{l}] must be [rows, {D}], got {tuple(W[l].shape)}")
        _size(S[l], W[l].shape[0] * (D // lay["block"]), f"S[{l}]")
        if out is not None:
            _size(out[l], n_rows_out * C * D, f"out[{l}]")


def _rows_ptr(cache_rows):
    return None if cache_rows is None else _dev(cache_rows, torch.int32, "cache_rows")


def engram_hash(state: int, ids: torch.Tensor, start_pos, mask: torch.Tensor | None = None,
                hashes: torch.Tensor | None = None, n_layers: int | None = None, n_cols: int | None = None,
                stream=None, cache_rows: torch.Tensor | None = None) -> torch.Tensor:
    """ids int64 [B, L] (CUDA); start_pos int or int32 [B]; mask bool/uint8 [B, L] or None;
    cache_rows int32 [B] or None (row b uses cache row cache_rows[b], else b).
    Returns (or fills) int64 hash ids [B, L, n_layers, C]."""
    B, L = ids.shape
    lay = engram_state_layout(state)
    NC = lay["n_layers"] * (lay["max_ngram"] - 1) * lay["n_heads"]
    temps = []
    if hashes is None:
        hashes = torch.empty((B, L, lay["n_layers"], (lay["max_ngram"] - 1) * lay["n_heads"]), dtype=torch.int64,
                             device=ids.device)
        temps.append(hashes)
    _size(hashes, B * L * NC, "hashes")
    _size(mask, B * L, "mask")
    _size(cache_rows, B, "cache_rows")
    _size(start_pos, B, "start_pos")
    sp = _start_tensor(start_pos, B, ids.device)
    if sp is not start_pos:
        temps.append(sp)
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    _check(_lib().engram_hash(state, _dev(ids, torch.int64, "ids"), m, _dev(sp, torch.int32, "start_pos"),
                              _rows_ptr(cache_rows), B, L, _dev(hashes, torch.int64, "hashes"),
                              _launch_stream(stream, temps)), "engram_hash")
    return hashes


def _as_u8(mask: torch.Tensor) -> torch.Tensor:
    return mask.view(torch.uint8) if mask.dtype == torch.bool else mask


def engram_lookup(idx: torch.Tensor, W: torch.Tensor, S: torch.Tensor, block: int, out: torch.Tensor | None = None,
                  stream=None, scale_dtype: int | None = None) -> torch.Tensor:
    """idx int64 [...]; W fp8 (float8_e4m3fn or uint8) [rows, D]; S [rows, D/block] scales (float32,
    bfloat16, float8_e8m0fnu or float8_e4m3fn; or raw bits with scale_dtype). Returns (or fills) bf16 [..., D]."""
    sdt = _scale_dtype_of(S, scale_dtype)
    rows, D = W.shape
    temps = []
    if out is None:
        out = torch.empty(tuple(idx.shape) + (D,), dtype=torch.bfloat16, device=idx.device)
        temps.append(out)
    _size(out, idx.numel() * D, "out")
    if int(block) > 0 and D % int(block) == 0:
        _size(S, rows * (D // int(block)), "S")
    Wu = W.view(torch.uint8)
    _check(_lib().engram_lookup(_dev(idx, torch.int64, "idx"), idx.numel(), _dev(Wu, torch.uint8, "W"),
                                _dev_scales(S, sdt), rows, D, int(block), sdt, _dev(out, torch.bfloat16, "out"),
                                _launch_stream(stream, temps)), "engram_lookup")
    return out


def engram_hash_lookup(state: int, ids: torch.Tensor, start_pos, W: list, S: list, mask: torch.Tensor | None = None,
                       out: list | None = None, hashes: torch.Tensor | None = None, stream=None,
                       cache_rows: torch.Tensor | None = None) -> list:
    """Hash + per-layer lookup in one launch. W/S: per-layer tables. Returns (or fills) the
    per-layer bf16 outputs [B, L, C, D]. An int start_pos costs a small fill kernel before the call;
    in a loop of calls pass a device int32 [B] tensor (or use PreparedHashLookup): consecutive calls of
    this library overlap their launches only when no other kernel or copy runs between them."""
    B, L = ids.shape
    lay = engram_state_layout(state)
    n = len(W)
    D, C = lay["head_dim"], (lay["max_ngram"] - 1) * lay["n_heads"]
    temps = []
    if out is None and len(W) == lay["n_layers"]:
        out = [torch.empty((B, L, C, D), dtype=torch.bfloat16, device=ids.device) for _ in range(n)]
        temps.extend(out)
    _tables(lay, W, S, out, B * L)
    _size(hashes, B * L * lay["n_layers"] * C, "hashes")
    _size(mask, B * L, "mask")
    _size(cache_rows, B, "cache_rows")
    _size(start_pos, B, "start_pos")
    sp = _start_tensor(start_pos, B, ids.device)
    if sp is not start_pos:
        temps.append(sp)
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    Wp = (_P * n)(*[_dev(w.view(torch.uint8), torch.uint8, "W") for w in W])
    sdt = lay["scale_dtype"]
    Sp = (_P * n)(*[_dev_scales(s, sdt) for s in S])
    Rp = (_I64 * n)(*[w.shape[0] for w in W])
    Op = (_P * n)(*[_dev(o, torch.bfloat16, "out") for o in out])
    hp = None if hashes is None else _dev(hashes, torch.int64, "hashes")
    _check(_lib().engram_hash_lookup(state, _dev(ids, torch.int64, "ids"), m, _dev(sp, torch.int32, "start_pos"),
                                     _rows_ptr(cache_rows), B, L, Wp, Sp, Rp, Op, hp, _launch_stream(stream, temps)),
           "engram_hash_lookup")
    return out


def _max_len(cu_seqlens: torch.Tensor, max_len) -> int:
    if max_len is not None:
        return int(max_len)
    # convenience only: reads the extents back (a device-to-host copy); pass max_len to avoid it
    return int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if cu_seqlens.numel() > 1 else 0


def engram_hash_varlen(state: int, ids: torch.Tensor, cu_seqlens: torch.Tensor, start_pos: torch.Tensor,
                       mask: torch.Tensor | None = None, hashes: torch.Tensor | None = None, max_len: int | None = None,
                       stream=None, cache_rows: torch.Tensor | None = None) -> torch.Tensor:
    """Packed sequences: ids int64 [T]; cu_seqlens int32 [B+1]; start_pos int32 [B]; mask [T] or None.
    Returns (or fills) int64 hash ids [T, n_layers, C]."""
    T = ids.numel()
    B = cu_seqlens.numel() - 1
    lay = engram_state_layout(state)
    temps = []
    if hashes is None:
        hashes = torch.empty((T, lay["n_layers"], (lay["max_ngram"] - 1) * lay["n_heads"]), dtype=torch.int64,
                             device=ids.device)
        temps.append(hashes)
    _size(hashes, T * lay["n_layers"] * (lay["max_ngram"] - 1) * lay["n_heads"], "hashes")
    _size(mask, T, "mask")
    _size(start_pos, B, "start_pos")
    _size(cache_rows, B, "cache_rows")
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    _check(_lib().engram_hash_varlen(state, _dev(ids, torch.int64, "ids"), m, _dev(cu_seqlens, torch.int32, "cu_seqlens"),
                                     _dev(start_pos, torch.int32, "start_pos"), _rows_ptr(cache_rows), B, T,
                                     _max_len(cu_seqlens, max_len), _dev(hashes, torch.int64, "hashes"),
                                     _launch_stream(stream, temps)), "engram_hash_varlen")
    return hashes


def engram_hash_lookup_varlen(state: int, ids: torch.Tensor, cu_seqlens: torch.Tensor, start_pos: torch.Tensor,
                              W: list, S: list, mask: torch.Tensor | None = None, out: list | None = None,
                              hashes: torch.Tensor | None = None, max_len: int | None = None, stream=None,
                              cache_rows: torch.Tensor | None = None) -> list:
    """Packed sequences, hash + per-layer lookup in one launch. Returns (or fills) per-layer bf16
    outputs [T, C, D]."""
    T = ids.numel()
    B = cu_seqlens.numel() - 1
    lay = engram_state_layout(state)
    n = len(W)
    D, C = lay["head_dim"], (lay["max_ngram"] - 1) * lay["n_heads"]
    temps = []
    if out is None and len(W) == lay["n_layers"]:
        out = [torch.empty((T, C, D), dtype=torch.bfloat16, device=ids.device) for _ in range(n)]
        temps.extend(out)
    _tables(lay, W, S, out, T)
    _size(hashes, T * lay["n_layers"] * C, "hashes")
    _size(mask, T, "mask")
    _size(start_pos, B, "start_pos")
    _size(cache_rows, B, "cache_rows")
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    Wp = (_P * n)(*[_dev(w.view(torch.uint8), torch.uint8, "W") for w in W])
    sdt = lay["scale_dtype"]
    Sp = (_P * n)(*[_dev_scales(x, sdt) for x in S])
    Rp = (_I64 * n)(*[w.shape[0] for w in W])
    Op = (_P * n)(*[_dev(o, torch.bfloat16, "out") for o in out])
    hp = None if hashes is None else _dev(hashes, torch.int64, "hashes")
    _check(_lib().engram_hash_lookup_varlen(state, _dev(ids, torch.int64, "ids"), m,
                                            _dev(cu_seqlens, torch.int32, "cu_seqlens"),
                                            _dev(start_pos, torch.int32, "start_pos"), _rows_ptr(cache_rows), B, T,
                                            _max_len(cu_seqlens, max_len), Wp, Sp, Rp, Op, hp,
                                            _launch_stream(stream, temps)),
           "engram_hash_lookup_varlen")
    return out


def engram_gate(x: torch.Tensor, kv: torch.Tensor, q_weight: torch.Tensor, k_weight: torch.Tensor,
                mask: torch.Tensor | None = None, eps: float = 1e-20, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """The Engram gate on bf16 tensors: x [T, hc, dim] (or [..., hc, dim]), kv [..., (hc+1)*dim],
    q_weight / k_weight [hc, dim], mask [...] bool or None. Returns (or fills; may be x) bf16 [..., hc, dim]."""
    hc, dim = x.shape[-2], x.shape[-1]
    T = x.numel() // (hc * dim)
    temps = []
    if out is None:
        out = torch.empty_like(x)
        temps.append(out)
    _size(kv, T * (hc + 1) * dim, "kv")
    _size(q_weight, hc * dim, "q_weight")
    _size(k_weight, hc * dim, "k_weight")
    _size(mask, T, "mask")
    _size(out, T * hc * dim, "out")
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    _check(_lib().engram_gate(_dev(x, torch.bfloat16, "x"), _dev(kv, torch.bfloat16, "kv"),
                              _dev(q_weight, torch.bfloat16, "q_weight"), _dev(k_weight, torch.bfloat16, "k_weight"),
                              m, T, hc, dim, float(eps), _dev(out, torch.bfloat16, "out"),
                              _launch_stream(stream, temps)), "engram_gate")
    return out


def engram_project(emb: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The `wkv` projection on the tensor cores: emb bf16 [..., K] (T rows), w bf16 [N, K].
    Returns (or fills) bf16 [..., N] = bf16(emb @ w^T), fp32 accumulation."""
    K = emb.shape[-1]
    T = emb.numel() // K if K else 0
    N = w.shape[0]
    if w.dim() != 2 or w.shape[1] != K:
        raise ValueError(f"w must be [N, {K}], got {tuple(w.shape)}")
    temps = []
    if out is None:
        out = torch.empty(tuple(emb.shape[:-1]) + (N,), dtype=torch.bfloat16, device=emb.device)
        temps.append(out)
    _size(out, T * N, "out")
    _check(_lib().engram_project(_dev(emb, torch.bfloat16, "emb"), _dev(w, torch.bfloat16, "w"), T, K, N,
                                 _dev(out, torch.bfloat16, "out"), _launch_stream(stream, temps)), "engram_project")
    return out


def engram_project_gate_workspace(T: int, hc: int, dim: int) -> int:
    """Bytes of workspace engram_project_gate needs (0 for T == 0 or an unsupported hc / dim)."""
    return int(_lib().engram_project_gate_workspace(int(T), int(hc), int(dim)))


def engram_project_gate(x: torch.Tensor, emb: torch.Tensor, wkv: torch.Tensor, q_weight: torch.Tensor,
                        k_weight: torch.Tensor, mask: torch.Tensor | None = None, eps: float = 1e-20,
                        workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """The Engram block after the lookup, fused: the `wkv` projection with the gate's sums in its
    epilogue (keys never written), then the gate. x bf16 [T, hc, dim]; emb bf16 [T, K];
    wkv bf16 [(hc+1)*dim, K]; q_weight / k_weight bf16 [hc, dim]; mask [T] bool or None;
    workspace: a uint8 CUDA tensor of at least engram_project_gate_workspace(T, hc, dim) bytes
    (allocated here when None). Returns (or fills; may be x) bf16 [T, hc, dim]."""
    hc, dim = x.shape[-2], x.shape[-1]
    T = x.numel() // (hc * dim)
    K = emb.shape[-1]
    temps = []
    if out is None:
        out = torch.empty_like(x)
        temps.append(out)
    _size(emb, T * K, "emb")
    _size(wkv, (hc + 1) * dim * K, "wkv")
    _size(q_weight, hc * dim, "q_weight")
    _size(k_weight, hc * dim, "k_weight")
    _size(mask, T, "mask")
    _size(out, T * hc * dim, "out")
    need = engram_project_gate_workspace(T, hc, dim)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
        temps.append(workspace)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, need {need}")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    _check(_lib().engram_project_gate(_dev(x, torch.bfloat16, "x"), _dev(emb, torch.bfloat16, "emb"),
                                      _dev(wkv, torch.bfloat16, "wkv"), _dev(q_weight, torch.bfloat16, "q_weight"),
                                      _dev(k_weight, torch.bfloat16, "k_weight"), m, T, K, hc, dim, float(eps),
                                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      _dev(out, torch.bfloat16, "out"), _launch_stream(stream, temps)),
           "engram_project_gate")
    return out


def _table(W: torch.Tensor, S: torch.Tensor, block: int, scale_dtype=None) -> _Table:
    sdt = _scale_dtype_of(S, scale_dtype)
    rows, D = W.shape
    if int(block) > 0 and D % int(block) == 0:
        _size(S, rows * (D // int(block)), "S")
    return _Table(_dev(W.view(torch.uint8), torch.uint8, "W"), _dev_scales(S, sdt), rows, D, int(block), sdt)


def _hash_ids(idx: torch.Tensor):
    """idx int64 [T, C] with unit stride along C (e.g. one layer of an engram_hash output viewed as
    [T, n_layers, C][:, layer]): returns (pointer, row stride, T, C)."""
    if not isinstance(idx, torch.Tensor) or not idx.is_cuda or idx.dtype != torch.int64:
        raise TypeError("idx must be an int64 CUDA tensor")
    if idx.dim() != 2 or (idx.shape[1] > 1 and idx.stride(1) != 1):
        raise ValueError(f"idx must be [T, C] with unit stride along C, got shape {tuple(idx.shape)} "
                         f"strides {idx.stride()}")
    T, C = idx.shape
    stride = idx.stride(0) if T > 1 else C
    if stride < C:
        raise ValueError("idx rows overlap")
    return idx.data_ptr(), stride, T, C


def _workspace(workspace, need: int, device, temps: list) -> tuple:
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        temps.append(workspace)
    nbytes = workspace.numel() * workspace.element_size()
    if nbytes < need:
        raise ValueError(f"workspace holds {nbytes} bytes, need {need}")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), nbytes


def engram_lookup_project_workspace(T: int, n_cols: int, head_dim: int) -> int:
    """Bytes of workspace engram_lookup_project needs."""
    return int(_lib().engram_lookup_project_workspace(int(T), int(n_cols), int(head_dim)))


def engram_lookup_project(idx: torch.Tensor, W: torch.Tensor, S: torch.Tensor, wkv: torch.Tensor, block: int,
                          out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None,
                          scale_dtype: int | None = None) -> torch.Tensor:
    """The lookup and the `wkv` projection in one kernel: idx int64 [T, C] hash ids of one layer (unit
    stride along C); W, S that layer's table (as engram_lookup); wkv bf16 [N, C * head_dim].
    Returns (or fills) bf16 [T, N], bit-identical to engram_project(engram_lookup(idx, W, S), wkv).
    workspace: uint8 CUDA tensor of engram_lookup_project_workspace(T, C, head_dim) bytes (allocated
    here when None)."""
    ptr, stride, T, C = _hash_ids(idx)
    tb = _table(W, S, block, scale_dtype)
    N = wkv.shape[0]
    _size(wkv, N * C * tb.head_dim, "wkv")
    temps = []
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=idx.device)
        temps.append(out)
    _size(out, T * N, "out")
    ws, nbytes = _workspace(workspace, engram_lookup_project_workspace(T, C, tb.head_dim), idx.device, temps)
    _check(_lib().engram_lookup_project(ptr, stride, T, C, ctypes.byref(tb), _dev(wkv, torch.bfloat16, "wkv"), N,
                                        ws, nbytes, _dev(out, torch.bfloat16, "out"), _launch_stream(stream, temps)),
           "engram_lookup_project")
    return out


def engram_lookup_project_gate_workspace(T: int, n_cols: int, head_dim: int, hc: int, dim: int) -> int:
    """Bytes of workspace engram_lookup_project_gate needs (0 for T == 0 or an unsupported shape)."""
    return int(_lib().engram_lookup_project_gate_workspace(int(T), int(n_cols), int(head_dim), int(hc), int(dim)))


def engram_lookup_project_gate(x: torch.Tensor, idx: torch.Tensor, W: torch.Tensor, S: torch.Tensor,
                               wkv: torch.Tensor, q_weight: torch.Tensor, k_weight: torch.Tensor, block: int,
                               mask: torch.Tensor | None = None, eps: float = 1e-20,
                               workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                               stream=None, scale_dtype: int | None = None) -> torch.Tensor:
    """The whole Engram block of one layer from its hash ids: the lookup inside the `wkv` projection,
    the gate's sums in its epilogue, then the gate. x bf16 [T, hc, dim]; idx int64 [T, C]; W, S the
    layer's table; wkv bf16 [(hc+1)*dim, C * head_dim]; q_weight / k_weight bf16 [hc, dim]; mask [T]
    bool or None. Returns (or fills; may be x) bf16 [T, hc, dim], bit-identical to
    engram_project_gate(x, engram_lookup(idx, W, S).view(T, -1), wkv, ...)."""
    ptr, stride, T, C = _hash_ids(idx)
    tb = _table(W, S, block, scale_dtype)
    hc, dim = x.shape[-2], x.shape[-1]
    if x.numel() != T * hc * dim:
        raise ValueError(f"x holds {x.numel()} values, expected T * hc * dim = {T * hc * dim}")
    temps = []
    if out is None:
        out = torch.empty_like(x)
        temps.append(out)
    _size(wkv, (hc + 1) * dim * C * tb.head_dim, "wkv")
    _size(q_weight, hc * dim, "q_weight")
    _size(k_weight, hc * dim, "k_weight")
    _size(mask, T, "mask")
    _size(out, T * hc * dim, "out")
    need = engram_lookup_project_gate_workspace(T, C, tb.head_dim, hc, dim)
    ws, nbytes = _workspace(workspace, need, x.device, temps)
    m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
    _check(_lib().engram_lookup_project_gate(_dev(x, torch.bfloat16, "x"), ptr, stride, T, C, ctypes.byref(tb),
                                             _dev(wkv, torch.bfloat16, "wkv"),
                                             _dev(q_weight, torch.bfloat16, "q_weight"),
                                             _dev(k_weight, torch.bfloat16, "k_weight"), m, hc, dim, float(eps), ws,
                                             nbytes, _dev(out, torch.bfloat16, "out"), _launch_stream(stream, temps)),
           "engram_lookup_project_gate")
    return out


def engram_device_status(clear: bool = True, stream=None) -> int:
    """Status flags of the kernels that have no state object (STATUS_TIMEOUT) on the current device;
    synchronises the stream."""
    v = ctypes.c_uint32(0)
    _check(_lib().engram_device_status(_stream(stream), ctypes.byref(v), int(bool(clear))), "engram_device_status")
    return v.value


def shard_part(rows: int, world: int) -> int:
    """Rows per rank of a table split over `world` ranks, as `ParallelEngramEmbedding` splits it:
    rank r holds rows [r * part, (r + 1) * part)."""
    return -(-int(rows) // int(world))


def engram_shard_pack(idx: torch.Tensor, rows: int, world: int, stream=None):
    """Group the indices of one lookup by the rank that owns their row. Returns (counts int64
    [world + 1], local_rows int64 [n], positions int64 [n]): bucket r = rank r's rows as rows of its
    shard, then the indices no rank owns; each bucket in index order; positions index into idx."""
    n = idx.numel()
    dev = idx.device
    counts = torch.zeros(world + 1, dtype=torch.int64, device=dev)
    local_rows = torch.empty(n, dtype=torch.int64, device=dev)
    positions = torch.empty(n, dtype=torch.int64, device=dev)
    ws = torch.empty(max(int(_lib().engram_shard_pack_workspace(n, int(world))), 16), dtype=torch.uint8, device=dev)
    _check(_lib().engram_shard_pack(_dev(idx, torch.int64, "idx"), n, int(rows), int(world), counts.data_ptr(),
                                    local_rows.data_ptr(), positions.data_ptr(), ws.data_ptr(), ws.numel(),
                                    _launch_stream(stream, (counts, local_rows, positions, ws))), "engram_shard_pack")
    return counts, local_rows, positions


def engram_shard_unpack(rows: torch.Tensor, positions: torch.Tensor, m: int, head_dim: int,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[positions[i]] = rows[i] for i < m, +0 rows at positions[m:] (the unowned indices).
    rows bf16 [m, head_dim]; returns (or fills) bf16 [n, head_dim]."""
    n = positions.numel()
    temps = []
    if out is None:
        out = torch.empty((n, head_dim), dtype=torch.bfloat16, device=positions.device)
        temps.append(out)
    _size(out, n * head_dim, "out")
    _size(rows, int(m) * head_dim, "rows")
    rp = _dev(rows, torch.bfloat16, "rows") if int(m) > 0 else None
    _check(_lib().engram_shard_unpack(rp, _dev(positions, torch.int64, "positions"), int(m), n, int(head_dim),
                                      _dev(out, torch.bfloat16, "out"), _launch_stream(stream, temps)),
           "engram_shard_unpack")
    return out


def dist_exchange(group=None):
    """The all-to-all of sharded_lookup over a torch.distributed process group (NCCL on GPUs):
    exchange(t, send_splits, recv_splits) sends t's first send_splits[0] rows to rank 0, the next
    send_splits[1] to rank 1, ..., and returns the rows received, rank 0's first."""
    import torch.distributed as dist

    def exchange(t: torch.Tensor, send_splits, recv_splits) -> torch.Tensor:
        # moved as raw bytes (row = dim 0): any element type travels, on every backend
        rest = tuple(t.shape[1:])
        row_bytes = t.element_size() * int(torch.tensor(rest).prod()) if rest else t.element_size()
        if t.numel() == 0:
            b = torch.empty((t.shape[0], row_bytes), dtype=torch.uint8, device=t.device)
        else:
            b = t.contiguous().view(torch.uint8).reshape(t.shape[0], row_bytes)
        out = torch.empty((int(sum(recv_splits)), row_bytes), dtype=torch.uint8, device=t.device)
        dist.all_to_all_single(out, b, [int(c) for c in recv_splits], [int(c) for c in send_splits], group=group)
        return out.view(t.dtype).reshape((out.shape[0],) + rest)

    return exchange


def sharded_lookup(idx: torch.Tensor, W_shard: torch.Tensor, S_shard: torch.Tensor, rows: int, block: int,
                   world: int, exchange, scale_dtype: int | None = None, ops=None) -> torch.Tensor:
    """One rank's part of a row-sharded lookup (engram-first/lookup page, `ParallelEngramEmbedding`,
    world > 1): this rank holds rows [rank * part, ...) of a table of `rows` rows (W_shard, S_shard:
    its shard_part(rows, world) rows, fewer for the last rank) and looks up its own indices idx [n].
    Instead of looking every index up locally, zeroing foreign rows and all-reducing, each request
    goes to the rank that owns its row and only that row comes back:
      pack by owner -> exchange the counts -> exchange the row ids -> look them up in the shard ->
      exchange the rows back -> unpack (+0 rows where no rank owns the index).
    `exchange(t, send_splits, recv_splits)` is the all-to-all (dist_exchange(group) over NCCL).
    `ops` replaces the device steps (pack, lookup, unpack) with others of the same contract; the
    library's kernels when None. Returns bf16 [n, head_dim], equal to engram_lookup on the whole table."""
    if ops is None:
        ops = (engram_shard_pack,
               lambda r, W, S: engram_lookup(r, W, S, block, scale_dtype=scale_dtype),
               engram_shard_unpack)
    pack, lookup, unpack = ops
    D = W_shard.shape[1]
    n = idx.numel()
    counts, local_rows, positions = pack(idx.reshape(-1), rows, world)
    send = [int(c) for c in counts[:world].cpu()]  # split sizes are host values for the exchange
    m = sum(send)
    recv = [int(c) for c in exchange(counts[:world].reshape(world, 1), [1] * world, [1] * world).reshape(-1).cpu()]
    wanted = exchange(local_rows[:m], send, recv)          # row ids other ranks want from this shard
    found = lookup(wanted, W_shard, S_shard).reshape(-1, D)  # this shard's rows for them
    back = exchange(found, recv, send)                      # this rank's rows, in packed order
    return unpack(back, positions, m, D).reshape(tuple(idx.shape) + (D,))


class PreparedHashLookup:
    """A fused hash + lookup call whose arguments are checked and marshalled once, for serving loops
    that call it many times on the same buffers (refill `ids` / `start_pos` / `mask` in place between
    calls). Calling it only enqueues the kernel, without rebuilding pointer arrays or re-checking
    tensors. It runs on the stream given here, or else on the stream current at each call (so it
    also works inside a CUDA-graph capture)."""

    def __init__(self, state: int, ids: torch.Tensor, start_pos: torch.Tensor, W: list, S: list,
                 out: list, mask: torch.Tensor | None = None, hashes: torch.Tensor | None = None,
                 cu_seqlens: torch.Tensor | None = None, max_len: int | None = None, stream=None,
                 cache_rows: torch.Tensor | None = None):
        n = len(W)
        lay = engram_state_layout(state)
        NC = lay["n_layers"] * (lay["max_ngram"] - 1) * lay["n_heads"]
        if cu_seqlens is None:
            B, T = ids.shape
            rows_out = B * T
        else:
            B, T = cu_seqlens.numel() - 1, ids.numel()
            rows_out = T
        _tables(lay, W, S, out, rows_out)
        _size(hashes, rows_out * NC, "hashes")
        _size(mask, rows_out, "mask")
        _size(start_pos, B, "start_pos")
        _size(cache_rows, B, "cache_rows")
        self._keep = (ids, start_pos, W, S, out, mask, hashes, cu_seqlens, cache_rows)  # the buffers stay alive
        self._W = (_P * n)(*[_dev(w.view(torch.uint8), torch.uint8, "W") for w in W])
        sdt = lay["scale_dtype"]
        self._S = (_P * n)(*[_dev_scales(x, sdt) for x in S])
        self._R = (_I64 * n)(*[w.shape[0] for w in W])
        self._O = (_P * n)(*[_dev(o, torch.bfloat16, "out") for o in out])
        m = None if mask is None else _dev(_as_u8(mask), torch.uint8, "mask")
        h = None if hashes is None else _dev(hashes, torch.int64, "hashes")
        sp = _dev(start_pos, torch.int32, "start_pos")
        cr = _rows_ptr(cache_rows)
        self._stream = None if stream is None else _stream(stream)
        L = _lib()
        if cu_seqlens is None:
            self._fn = L.engram_hash_lookup
            self._args = (state, _dev(ids, torch.int64, "ids"), m, sp, cr, B, T, self._W, self._S, self._R, self._O, h)
        else:
            self._fn = L.engram_hash_lookup_varlen
            self._args = (state, _dev(ids, torch.int64, "ids"), m, _dev(cu_seqlens, torch.int32, "cu_seqlens"), sp, cr,
                          B, ids.numel(), _max_len(cu_seqlens, max_len), self._W, self._S, self._R, self._O, h)

    def __call__(self) -> None:
        st = self._stream if self._stream is not None else torch.cuda.current_stream().cuda_stream
        rc = self._fn(*self._args, st)
        if rc != OK:
            raise EngramError(rc, "prepared engram_hash_lookup")


# ----------------------------------------------------------------------------- convenience object
class EngramHash:
    """A state plus the calls that use it (the hash module of the model, with its cache)."""

    def __init__(self, *, n_layers, max_ngram, n_heads, head_dim, block, max_batch, max_seq_len, token_map,
                 multipliers, primes, offsets, dead=-1, pad_id=2, scale_dtype=SCALE_F32):
        self.n_layers, self.max_ngram, self.n_heads = n_layers, max_ngram, n_heads
        self.n_cols = (max_ngram - 1) * n_heads
        self.head_dim, self.block, self.scale_dtype = head_dim, block, int(scale_dtype)
        self.handle = engram_state_create(n_layers=n_layers, max_ngram=max_ngram, n_heads=n_heads, head_dim=head_dim,
                                          block=block, max_batch=max_batch, max_seq_len=max_seq_len,
                                          token_map=token_map, multipliers=multipliers, primes=primes,
                                          offsets=offsets, dead=dead, pad_id=pad_id, scale_dtype=scale_dtype)

    def close(self):
        if self.handle:
            engram_state_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        engram_cache_reset(self.handle)

    def status(self, clear=True) -> int:
        return engram_state_status(self.handle, clear)

    def hash(self, ids, start_pos=0, mask=None, hashes=None, cache_rows=None):
        if hashes is None:
            B, L = ids.shape
            hashes = torch.empty((B, L, self.n_layers, self.n_cols), dtype=torch.int64, device=ids.device)
        return engram_hash(self.handle, ids, start_pos, mask, hashes, cache_rows=cache_rows)

    def hash_lookup(self, ids, W, S, start_pos=0, mask=None, out=None, hashes=None, cache_rows=None):
        if out is None:
            B, L = ids.shape
            out = [torch.empty((B, L, self.n_cols, self.head_dim), dtype=torch.bfloat16, device=ids.device)
                   for _ in range(len(W))]
        return engram_hash_lookup(self.handle, ids, start_pos, W, S, mask, out, hashes, cache_rows=cache_rows)

    def hash_varlen(self, ids, cu_seqlens, start_pos, mask=None, hashes=None, max_len=None, cache_rows=None):
        return engram_hash_varlen(self.handle, ids, cu_seqlens, start_pos, mask, hashes, max_len,
                                  cache_rows=cache_rows)

    def hash_lookup_varlen(self, ids, cu_seqlens, start_pos, W, S, mask=None, out=None, hashes=None, max_len=None,
                           cache_rows=None):
        return engram_hash_lookup_varlen(self.handle, ids, cu_seqlens, start_pos, W, S, mask, out, hashes, max_len,
                                         cache_rows=cache_rows)

    def prepare_hash_lookup(self, ids, start_pos, W, S, out, mask=None, hashes=None, cu_seqlens=None, max_len=None,
                            stream=None, cache_rows=None) -> PreparedHashLookup:
        return PreparedHashLookup(self.handle, ids, start_pos, W, S, out, mask, hashes, cu_seqlens, max_len, stream,
                                  cache_rows)

    def lookup(self, idx, W, S, out=None):
        return engram_lookup(idx, W, S, self.block, out, scale_dtype=self.scale_dtype)
