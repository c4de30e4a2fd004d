#!/usr/bin/env python
"""Benchmark of the fused Engram n-gram hash + fp8 row lookup on GB300.

One step = one pass of the whole hot path over one batch: the n-gram hash
(token_map compression, cache write, lookback with blocking, multiply/XOR,
floored mod by primes, offsets) fused with the gather of 2 x 24 fp8 rows per
token from the two full-scale tables (384,006,168 and 384,016,682 rows x 128,
~98 GB) and their fp32 scales, dequantised to bf16 -- one kernel launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--cfg 3] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is tokens/s over all ranks with inputs
resident in HBM; `e2e` adds the host->device copy of the step's ids and the
device->host copy of its bf16 rows from/to pinned host memory; `roofline`
relates the fused kernel's algorithmic bytes (fp8 row + fp32 scale read +
bf16 row written, 18,624 B per token) to the measured HBM copy bandwidth;
`cpu_baseline` times the CPU oracle on the same workload.

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica on its own batch (weak scaling): the path has no exchange step.
`--impl reference` times the CPU oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_profile_case_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "gram_hash_embedding_gb300", "csrc", f) for f in
                  ("kernels.cu", "engram_internal.cuh", "dequant.cuh")]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--cfg", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8],
                   help="1 prefill B4xL4096, 2 decode B256xL1, 3 full-scale B8xL8192 (default), 4 long chunked, "
                        "5 profiling case (prefill shapes, 1 GB tables), 6 full-scale with head_dim 256, "
                        "7 continuous batching (packed decode + prefill sequences), 8 full-scale with head_dim 256 "
                        "and UE8M0 scales")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=0, help="steps of the end-to-end loop (default min(K, 100))")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mode", choices=["fused", "hash", "lookup"], default="fused",
                   help="fused: engram_hash_lookup (default); hash: engram_hash alone (int64 ids out); "
                        "lookup: engram_lookup alone on the workload's row ids, one launch per layer")
    p.add_argument("--block", action="store_true",
                   help="time the whole Engram block per step: hash + lookup, then per layer the wkv projection "
                        "and the gate, at the released width (dim 5120, 4 copies)")
    p.add_argument("--proj", choices=["fused", "lookahead", "tcgen05", "cublas"], default="fused",
                   help="--block: fused = engram_project_gate (tensor-core projection with the gate's sums in its "
                        "epilogue, keys never written, then the gate's finishing pass); lookahead = the hash alone, "
                        "then per layer engram_lookup_project_gate (the lookup inside that projection, one tile "
                        "group ahead); tcgen05 = engram_project then engram_gate; cublas = torch.matmul (cuBLAS) "
                        "then engram_gate")
    p.add_argument("--shard", type=int, default=0, metavar="W",
                   help="time the device steps of the row-sharded lookup for W ranks on this GPU: engram_shard_pack "
                        "of the workload's layer-0 row ids and engram_shard_unpack of as many head_dim rows (the "
                        "exchange between ranks is the caller's all-to-all and is not timed here)")
    p.add_argument("--graph", action="store_true",
                   help="capture the steps in a CUDA graph and replay it (removes host launch overhead; for the "
                        "small decode / chunk launches, and for --block steps of a few hundred tokens)")
    p.add_argument("--l2", choices=["auto", "flush", "none"], default="auto",
                   help="L2 between timed steps: flush = write 256 MB before every step and time the kernels "
                        "alone; auto (default) = flush when the steps' rows fit in L2 (decode) and launches are "
                        "eager; none = back to back")
    p.add_argument("--l2-fetch", type=int, default=32, choices=[0, 32, 64, 128],
                   help="the context's L2 fetch granularity limit for the run (bytes; 0 leaves the context "
                        "default, 64 on GB300). At 32 a row's random 4-byte scale read costs a 32-byte DRAM "
                        "sector instead of a 128-byte line (engram_set_l2_fetch_granularity)")
    return p.parse_args(argv)


def apply_l2_fetch(geng, nbytes: int):
    """Set the L2 fetch granularity limit of this process's context (0: leave it as it is); returns
    the previous value, or None when it was left."""
    return geng.set_l2_fetch_granularity(nbytes) if nbytes else None


L2_BYTES = 129 * 1000 * 1000  # GB300 L2
DECODE_STEPS = 128  # steps of the decode run (configuration 2)


def l2_working_set(runner) -> int:
    """DRAM bytes the timed steps touch across the cycled id batches: per row of every step a
    128-byte atom for its codes (head_dim bytes, at least 128) and one for its scales, plus the
    bf16 output (written to the same buffers every step)."""
    lay = runner.lay
    rows = runner.tokens_per_step * lay.n_layers * lay.n_cols
    per_row_read = max(128, lay.head_dim) + 128
    return rows * per_row_read * len(runner.ids) + rows * 2 * lay.head_dim


def l2_note(runner, flushed: bool, fits: bool) -> str:
    ws = l2_working_set(runner)
    lay = runner.lay
    tables = sum(lay.rows) * (lay.head_dim + 4 * lay.n_scales)
    if flushed:
        return (f"L2 flushed between timed steps (256 MB written outside the per-launch events; value from the "
                f"event-timed kernels alone): the {len(runner.ids)} cycled id batches touch {ws / 1e6:.0f} MB, "
                f"less than L2")
    if fits:
        return (f"warm: the {len(runner.ids)} cycled id batches touch {ws / 1e6:.0f} MB, which fits in the "
                f"129 MB L2 (back-to-back steps, no flush)")
    return (f"inputs larger than L2: {tables / 1e9:.1f} GB of tables read at random, {ws / 1e6:.0f} MB touched "
            f"over the {len(runner.ids)} cycled id batches")


# ----------------------------------------------------------------------------- distributed plumbing
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29533")
        dist.init_process_group(backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each replica hashes its own batch (different ids); the tables are the same."""
    return base + 1000 * rank


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = self._smi_id(gpu_index)
        self.proc = None
        self.lines = []

    @staticmethod
    def _smi_id(local: int) -> str:
        """nvidia-smi id of the device this process uses (CUDA_VISIBLE_DEVICES may renumber it)."""
        try:
            import torch

            u = str(torch.cuda.get_device_properties(local).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            parts = [v for v in vis.split(",") if v.strip()]
            return parts[local].strip() if local < len(parts) else str(local)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, max_mhz_default=None):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz_default, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(lay, rows_per_launch: int, l2_fetch: int = 0):
    """DRAM bytes per launch of the fused kernel, from the committed one-pass ncu capture of the
    profiling case (about 1 GB of tables: small enough for any capture), scaled to this launch by
    its count of gathered rows (the kernel's DRAM bytes grow with the rows it gathers: a code row,
    a scale sector and a bf16 row each). Returns (bytes, note), or (None, reason) when the kernel
    sources changed since the counters were taken, the row format (head_dim, scale storage) or the
    L2 fetch granularity setting (0: the context default) differs from the capture's."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no capture recorded"
    d = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            d[k.strip()] = v.strip()
    if d.get("source_sha256") != kernel_source_hash():
        return None, "kernel sources changed since the capture"
    if int(d.get("head_dim", -1)) != lay.head_dim or int(d.get("scale_bytes", -1)) != lay.scale_bytes * (
            lay.head_dim // lay.block):
        return None, "another row format than the capture's"
    if int(d.get("l2_fetch_granularity", 0)) != l2_fetch:
        return None, "another L2 fetch granularity than the capture's"
    cap_rows = int(d["rows_per_launch"])
    factor = rows_per_launch / cap_rows
    note = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of the profiling case (cfg {d['cfg']}, "
            f"{cap_rows:,} gathered rows per launch, {float(d['dram_bytes_per_launch']):,.0f} B), scaled by "
            f"{factor:g} to this launch's {rows_per_launch:,} rows ({TRAFFIC_FILE[len(ROOT) + 1:]})")
    return float(d["dram_bytes_per_launch"]) * factor, note


def algo_bytes_per_token(lay) -> int:
    """fp8 row + its scales (of the layout's storage width) read, bf16 row written, per hash column."""
    D, nsc = lay.head_dim, lay.head_dim // lay.block
    return lay.n_layers * lay.n_cols * (D + lay.scale_bytes * nsc + 2 * D)


def scale_torch_dtype(torch, scale_dtype: int):
    """torch dtype of a scale tensor of storage type `scale_dtype` (SCALE_F32, BF16, E8M0, E4M3)."""
    return [torch.float32, torch.bfloat16, torch.float8_e8m0fnu, torch.float8_e4m3fn][scale_dtype]


def scale_bits(torch, t):
    """Host numpy copy of a device scale tensor: fp32 values, or the bits of the other storage types."""
    if t.dtype == torch.float32:
        return t.cpu().numpy()
    if t.element_size() == 2:
        return t.view(torch.int16).cpu().numpy().view("uint16")
    return t.view(torch.uint8).cpu().numpy()


# ----------------------------------------------------------------------------- our arm
class Runner:
    """Device-resident workload and one step of the fused path for configuration `cfg`."""

    def __init__(self, cfg: int, rank: int, device):
        import numpy as np
        import torch

        import gram_hash_embedding_gb300 as geng
        import synth

        self.torch, self.np, self.geng, self.synth = torch, np, geng, synth
        self.cfg = cfg
        self.device = device
        wl = synth.make_workload(cfg)
        self.wl = wl
        lay = wl.layout
        self.lay = lay
        # tables: one replica per GPU, filled by the seeded generator
        self.W, self.S = [], []
        for l, rows in enumerate(lay.rows):
            W = torch.empty((rows, lay.head_dim), dtype=torch.uint8, device=device)
            S = torch.empty((rows, lay.n_scales), dtype=scale_torch_dtype(torch, lay.scale_dtype), device=device)
            synth.fill_table_device(W, S, wl.table_seed, l, lay.scale_dtype)
            self.W.append(W)
            self.S.append(S)
        self.state = geng.EngramHash(n_layers=lay.n_layers, max_ngram=lay.max_ngram, n_heads=lay.n_heads,
                                     head_dim=lay.head_dim, block=lay.block, max_batch=wl.max_batch,
                                     max_seq_len=wl.max_seq_len + (DECODE_STEPS if cfg == 2 else 0),
                                     token_map=lay.token_map,
                                     multipliers=lay.multipliers, primes=lay.primes, offsets=lay.offsets,
                                     dead=lay.dead, pad_id=lay.pad_id, scale_dtype=lay.scale_dtype)
        seed = rank_seed(synth.MASTER_SEED + 17, rank)
        self.varlen = cfg == 7
        # batches: distinct id sets (each with its start positions) cycled step to step
        starts = None
        if cfg == 7:
            ids = [wl.ids]
            masks = [None]
            self.chunks = [(0, wl.ids.size)]
            self.B, self.L = wl.B, wl.L
            self.cu = torch.from_numpy(wl.extra["cu_seqlens"]).to(device)
        elif cfg == 4:
            total = wl.ids.shape[1]
            ids = [wl.ids if rank == 0 else synth.zipf_ids(seed, total).reshape(1, total)]
            masks = [wl.mask]
            self.chunks = [(k * wl.L, (k + 1) * wl.L) for k in range(wl.chunks)]
            self.B, self.L = 1, total
        elif cfg == 2:
            # a decode run: step k gives every row its next Zipf token at position start + k, so the
            # steps gather different rows (about 400 MB of row atoms over the run, three times L2);
            # on rank 0 step 0 is the workload's own decode step
            P = wl.prefill_ids.shape[1]
            base = synth.MASTER_SEED + 2 if rank == 0 else seed
            ids = [synth.zipf_ids(base, wl.B, offset=wl.B * P + k * wl.B).reshape(wl.B, 1) for k in range(DECODE_STEPS)]
            assert rank != 0 or np.array_equal(ids[0], wl.ids)
            starts = [wl.start_pos.astype(np.int32) + k for k in range(DECODE_STEPS)]
            masks = [None] * len(ids)
            self.chunks = [(0, 1)]
            self.B, self.L = wl.B, 1
        else:
            ids = [wl.ids if (k == 0 and rank == 0) else
                   synth.uniform_ids(seed + k, wl.B * wl.L).reshape(wl.B, wl.L) for k in range(4)]
            masks = [wl.mask] * len(ids)
            self.chunks = [(0, wl.L)]
            self.B, self.L = wl.B, wl.L
        self.ids_host = ids
        self.ids = [torch.from_numpy(np.ascontiguousarray(a)).to(device) for a in ids]
        self.masks = [None if m is None else torch.from_numpy(np.ascontiguousarray(m)).to(device) for m in masks]
        if starts is None:
            starts = [wl.start_pos.astype(np.int32)]
        self.starts = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device) for a in starts]
        self.start = self.starts[0]  # the start positions of explicit-ids steps (the end-to-end leg sets them)
        if wl.prefill_ids is not None:  # decode / continuous batching: history first
            self.state.hash(torch.from_numpy(wl.prefill_ids).to(device), 0)
        Lc = self.chunks[0][1] - self.chunks[0][0]
        out_shape = (wl.ids.size, lay.n_cols, lay.head_dim) if self.varlen else (self.B, Lc, lay.n_cols, lay.head_dim)
        self.out = [torch.empty(out_shape, dtype=torch.bfloat16, device=device) for _ in range(lay.n_layers)]
        self.tokens_per_step = wl.ids.size if self.varlen else self.B * self.L
        self.launches_per_step = len(self.chunks)
        # one prepared call per id batch (arguments marshalled once) for the single-launch steps
        self.calls = None
        if len(self.chunks) == 1:
            self.calls = [self.geng.PreparedHashLookup(
                self.state.handle, i, self.starts[j % len(self.starts)], self.W, self.S, self.out, mask=m,
                cu_seqlens=self.cu if self.varlen else None, max_len=self.L if self.varlen else None)
                for j, (i, m) in enumerate(zip(self.ids, self.masks))]
        # chunked steps: one prepared call per (id batch, chunk) with the chunk's start positions already
        # on the device, so nothing but this library's kernels runs between two chunks (an int start
        # position would put a fill kernel before every chunk and end the overlap of consecutive launches)
        self.chunk_calls = None
        if len(self.chunks) > 1:
            chunk_starts = [torch.full((self.B,), c0, dtype=torch.int32, device=device) for c0, _ in self.chunks]
            self.chunk_calls = []
            for i, m in zip(self.ids, self.masks):
                calls = []
                for (c0, c1), sp in zip(self.chunks, chunk_starts):
                    ii = i[:, c0:c1] if i[:, c0:c1].is_contiguous() else i[:, c0:c1].contiguous()
                    mm = None if m is None else (m[:, c0:c1] if m[:, c0:c1].is_contiguous() else m[:, c0:c1].contiguous())
                    calls.append(self.geng.PreparedHashLookup(self.state.handle, ii, sp, self.W, self.S, self.out,
                                                              mask=mm))
                self.chunk_calls.append(calls)
        sname = ["fp32", "bf16", "UE8M0", "E4M3"][lay.scale_dtype]
        self.scale_name = sname
        self.kernel_name = f"hash_kernel<GATHER=true, D={lay.head_dim}, {sname} scales> (hash + gather + dequant)"
        torch.cuda.synchronize(device)

    def step(self, k: int, ids=None, mask=None):
        """Enqueue one step; returns the launches' (start, end) event pairs when timing."""
        if ids is None and mask is None and self.calls is not None:
            self.calls[k % len(self.calls)]()
            return
        if ids is None and mask is None and self.chunk_calls is not None:
            for call in self.chunk_calls[k % len(self.chunk_calls)]:
                call()
            return
        start = self.starts[k % len(self.starts)] if ids is None else self.start
        ids = self.ids[k % len(self.ids)] if ids is None else ids
        mask = self.masks[k % len(self.masks)] if mask is None else mask
        if self.varlen:
            self.geng.engram_hash_lookup_varlen(self.state.handle, ids, self.cu, start, self.W, self.S, mask,
                                                self.out, max_len=self.L)
            return
        for c0, c1 in self.chunks:
            if len(self.chunks) == 1:
                ii, mm, sp = ids, mask, start
            else:
                ii = ids[:, c0:c1]
                mm = None if mask is None else mask[:, c0:c1]
                sp = c0
            self.geng.engram_hash_lookup(self.state.handle, ii if ii.is_contiguous() else ii.contiguous(), sp,
                                         self.W, self.S, mm if (mm is None or mm.is_contiguous()) else mm.contiguous(),
                                         self.out)

    def setup_mode(self, mode: str):
        """Buffers of the hash-only and lookup-only measurements."""
        torch = self.torch
        lay = self.lay
        self.mode = mode
        if mode == "fused":
            return
        self.hash_out = torch.empty((self.B, self.L, lay.n_layers, lay.n_cols), dtype=torch.int64, device=self.device)
        if mode == "lookup":
            # the row ids this workload hashes to, one flat list per layer
            self.geng.engram_hash(self.state.handle, self.ids[0], self.start, self.masks[0], self.hash_out)
            self.idx = [self.hash_out[:, :, l, :].contiguous().view(-1) for l in range(lay.n_layers)]
            self.lookup_out = [torch.empty((self.idx[l].numel(), lay.head_dim), dtype=torch.bfloat16,
                                           device=self.device) for l in range(lay.n_layers)]
            self.launches_per_step = lay.n_layers
            self.kernel_name = f"lookup_kernel<D={lay.head_dim}>"
        else:
            self.kernel_name = "hash_kernel<GATHER=false>"
        torch.cuda.synchronize(self.device)

    def step_mode(self, k: int):
        if self.mode == "hash":
            ids = self.ids[k % len(self.ids)]
            mask = self.masks[k % len(self.masks)]
            self.geng.engram_hash(self.state.handle, ids, self.starts[k % len(self.starts)], mask, self.hash_out)
        elif self.mode == "lookup":
            for l in range(self.lay.n_layers):
                self.geng.engram_lookup(self.idx[l], self.W[l], self.S[l], self.lay.block, self.lookup_out[l])
        else:
            self.step(k)

    def mode_bytes_per_token(self) -> int:
        lay = self.lay
        if self.mode == "hash":  # ids in, cache entry out, int64 hash ids out (mask byte if any)
            return 8 + 4 + 8 * lay.n_layers * lay.n_cols + (1 if self.masks[0] is not None else 0)
        if self.mode == "lookup":  # the fused bytes plus the int64 row id read per row
            return algo_bytes_per_token(lay) + 8 * lay.n_layers * lay.n_cols
        return algo_bytes_per_token(lay)

    def e2e_buffers(self):
        torch = self.torch
        self.ids_pinned = [torch.from_numpy(self.np.ascontiguousarray(a)).pin_memory() for a in self.ids_host]
        self.mask_pinned = [None if m is None else m.cpu().pin_memory() for m in self.masks]
        self.start_pinned = [s.cpu().pin_memory() for s in self.starts]
        self.ids_dev = torch.empty_like(self.ids[0])
        self.mask_dev = None if self.masks[0] is None else torch.empty_like(self.masks[0])
        self.start_dev = torch.empty_like(self.start)
        self.out_pinned = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.out]
        if self.varlen:
            self.cu_pinned = self.cu.cpu().pin_memory()
            self.cu_dev = torch.empty_like(self.cu)
        # groups of batch rows for the pipelined copy-out: at most 8, each of at least 4096 tokens
        n = max(1, min(self.B, 8, self.B * self.L // 4096))
        per = -(-self.B // n)
        self.e2e_pieces = [(b, min(self.B, b + per)) for b in range(0, self.B, per)]
        self.e2e_events = [torch.cuda.Event() for _ in self.e2e_pieces]
        self.e2e_rows = torch.arange(self.B, dtype=torch.int32, device=self.device)
        self.copy_stream = torch.cuda.Stream()
        # the pipelined leg alternates two sets of buffers, so a step's calls overlap the previous
        # step's copies; set s may be refilled once the copies of the step that used it are done
        self.e2e_sets = [(self.ids_dev, self.start_dev, self.mask_dev, self.out, self.out_pinned)]
        self.e2e_sets.append((torch.empty_like(self.ids_dev), torch.empty_like(self.start_dev),
                              None if self.mask_dev is None else torch.empty_like(self.mask_dev),
                              [torch.empty_like(o) for o in self.out],
                              [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.out]))
        self.e2e_done = [None, None]

    def e2e_step(self, k: int, drain: bool = True):
        """Host ids -> device, fused hash + lookup through the C ABI, bf16 rows -> host. `drain`: the
        current stream waits for the step's copies (the last step of a timed run, always outside the
        pipelined leg)."""
        if not self.varlen and len(self.chunks) == 1 and len(self.e2e_pieces) > 1:
            self.e2e_pipelined(k, drain)
            return
        j = k % len(self.ids_pinned)
        self.ids_dev.copy_(self.ids_pinned[j], non_blocking=True)
        if self.mask_dev is not None:
            self.mask_dev.copy_(self.mask_pinned[j % len(self.mask_pinned)], non_blocking=True)
        self.start_dev.copy_(self.start_pinned[j % len(self.start_pinned)], non_blocking=True)
        saved, saved_cu = self.start, getattr(self, "cu", None)
        self.start = self.start_dev
        if self.varlen:
            self.cu_dev.copy_(self.cu_pinned, non_blocking=True)
            self.cu = self.cu_dev
        try:
            if self.varlen or len(self.chunks) == 1:
                self.step(k, self.ids_dev, self.mask_dev)
                for o, h in zip(self.out, self.out_pinned):
                    h.copy_(o, non_blocking=True)
            else:  # chunked: copy each chunk's rows out after its launch
                for c0, c1 in self.chunks:
                    mm = None if self.mask_dev is None else self.mask_dev[:, c0:c1].contiguous()
                    self.geng.engram_hash_lookup(self.state.handle, self.ids_dev[:, c0:c1].contiguous(), c0, self.W,
                                                 self.S, mm, self.out)
                    for o, h in zip(self.out, self.out_pinned):
                        h.copy_(o, non_blocking=True)
        finally:
            self.start = saved
            if self.varlen:
                self.cu = saved_cu

    def e2e_pipelined(self, k: int, drain: bool):
        """One call per group of batch rows, each on its rows' own cache rows (rows never interact,
        so hash ids, rows and cache equal one call's): group g's rows leave for the host on a copy
        stream while group g+1 is computed, and step k uses buffer set k % 2, so its calls also
        overlap the copies of step k - 1."""
        torch = self.torch
        cur = torch.cuda.current_stream()
        s = k % 2
        ids_dev, start_dev, mask_dev, out, out_pinned = self.e2e_sets[s]
        if self.e2e_done[s] is not None:  # the copies of step k - 2 have left set s
            cur.wait_event(self.e2e_done[s])
        j = k % len(self.ids_pinned)
        ids_dev.copy_(self.ids_pinned[j], non_blocking=True)
        if mask_dev is not None:
            mask_dev.copy_(self.mask_pinned[j % len(self.mask_pinned)], non_blocking=True)
        start_dev.copy_(self.start_pinned[j % len(self.start_pinned)], non_blocking=True)
        for (b0, b1), ev in zip(self.e2e_pieces, self.e2e_events):
            mm = None if mask_dev is None else mask_dev[b0:b1]
            self.geng.engram_hash_lookup(self.state.handle, ids_dev[b0:b1], start_dev[b0:b1], self.W,
                                         self.S, mm, [o[b0:b1] for o in out], cache_rows=self.e2e_rows[b0:b1])
            ev.record(cur)
            self.copy_stream.wait_event(ev)
            with torch.cuda.stream(self.copy_stream):
                for o, h in zip(out, out_pinned):
                    h[b0:b1].copy_(o[b0:b1], non_blocking=True)
        done = torch.cuda.Event()
        done.record(self.copy_stream)
        self.e2e_done[s] = done
        if drain:
            cur.wait_stream(self.copy_stream)

    def e2e_bytes(self):
        h2d = self.ids_pinned[0].numel() * 8 + self.start_pinned[0].numel() * 4 + (4 * self.cu.numel() if self.varlen else 0)
        if self.mask_dev is not None:
            h2d += self.mask_dev.numel()
        d2h = sum(o.numel() * 2 for o in self.out) * len(self.chunks)
        return h2d, d2h


def link_bandwidth(torch, runner, reps: int = 5):
    """The CPU-GPU link alone, in the same run as the end-to-end leg: one step's output rows (device
    to pinned host) and one step's ids (pinned host to device) copied with no kernel running, CUDA
    events, best of `reps`. The end-to-end step cannot beat its device-to-host copy at this rate."""
    out = runner.e2e_sets[0][3]
    out_pinned = runner.e2e_sets[0][4]
    d2h_bytes = sum(o.numel() * o.element_size() for o in out)
    ids_dev, ids_host = runner.e2e_sets[0][0], runner.ids_pinned[0]
    h2d_bytes = ids_dev.numel() * ids_dev.element_size()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best_d2h = best_h2d = float("inf")
    torch.cuda.synchronize()
    for _ in range(reps):
        a.record()
        for o, h in zip(out, out_pinned):
            h.copy_(o, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best_d2h = min(best_d2h, a.elapsed_time(b) / 1e3)
        a.record()
        ids_dev.copy_(ids_host, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best_h2d = min(best_h2d, a.elapsed_time(b) / 1e3)
    return {"d2h_bytes": d2h_bytes, "d2h_ms": best_d2h * 1e3, "d2h_gbs": d2h_bytes / best_d2h / 1e9,
            "h2d_bytes": h2d_bytes, "h2d_ms": best_h2d * 1e3, "h2d_gbs": h2d_bytes / best_h2d / 1e9,
            "how": "the step's rows device->pinned host and its ids pinned host->device, no kernel running, "
                   f"best of {reps}"}


def time_region(torch, dist, dev_index, fn, steps, stream, per_launch_events=False, between=None):
    """Run `fn(k)` `steps` times between barriers and synchronisations; returns (total seconds, per-step
    seconds between the events around each `fn(k)`, or None) from CUDA events on `stream`.
    `between(k)`, when given, runs before each step outside its events (an L2 flush)."""
    torch.cuda.synchronize()
    barrier(dist, dev_index)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    pairs = []
    start.record(stream)
    for k in range(steps):
        if between is not None:
            between(k)
        if per_launch_events:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(k)
            b.record(stream)
            pairs.append((a, b))
        else:
            fn(k)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev_index)
    total = start.elapsed_time(end) / 1e3
    per_step = [a.elapsed_time(b) / 1e3 for a, b in pairs] if pairs else None
    return total, per_step


def cpu_baselines(runner, n_tokens: int):
    """Time the CPU oracle (as it stands) on the first n_tokens of the workload: hash of those tokens,
    then the lookup of every row they touch, single-threaded and on every host core; plus the
    torch-CPU restatement on the same sample. The touched rows are copied out of the
    generator-filled device tables into compact host tables (not timed).
    Returns (single-thread oracle, all-cores oracle, torch CPU) baseline dicts."""
    import numpy as np

    import oracle

    torch = runner.torch
    wl, lay = runner.wl, runner.lay
    ids = runner.ids_host[0]
    B, L = ids.shape
    rows_used = max(1, min(B, -(-n_tokens // L)))
    cut = min(L, n_tokens)
    sub = np.ascontiguousarray(ids[:rows_used, :cut])
    mask = None if wl.mask is None else np.ascontiguousarray(wl.mask[:rows_used, :cut])
    orc = oracle.OracleState.from_layout(lay, rows_used, max(cut, 1))
    t0 = time.perf_counter()
    hashes, _ = orc.hash(sub, 0, mask)
    t_hash = time.perf_counter() - t0
    t_lookup = 0.0
    compact = []
    for l in range(lay.n_layers):
        flat = hashes[:, :, l, :].reshape(-1)
        uniq, inv = np.unique(flat, return_inverse=True)
        inv = inv.astype(np.int64)
        sel = torch.from_numpy(uniq).to(runner.device)
        Wc = runner.W[l][sel].cpu().numpy()
        Sc = scale_bits(torch, runner.S[l][sel])
        compact.append((inv, Wc, Sc, int(uniq.size)))
        t0 = time.perf_counter()
        oracle.engram_lookup(inv, Wc, Sc, uniq.size, lay.head_dim, lay.block, scale_dtype=lay.scale_dtype)
        t_lookup += time.perf_counter() - t0
    tokens = sub.size
    what = (f"first {tokens} tokens of the same workload ({rows_used} sequence(s) x {cut}); hash + lookup of their "
            f"{tokens * lay.n_layers * lay.n_cols} rows")
    single = {"value": tokens / (t_hash + t_lookup), "unit": "tokens/s", "cores": 1, "kind": "oracle",
              "sample": f"{what}; single-threaded C; hash {t_hash:.3f} s + lookup {t_lookup:.3f} s"}
    ph, pl, cores = cpu_baseline_all_cores(lay, sub, mask, compact)
    allc = {"value": tokens / (ph + pl), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}; the same C oracle in {cores} spawned processes (hash split by sequence, lookup "
                      f"in index chunks); hash {ph:.3f} s + lookup {pl:.3f} s"}
    threads = torch.get_num_threads()
    tables = [(inv, Wc, Sc) for inv, Wc, Sc, _ in compact]
    torch_cpu_hash_lookup(torch, lay, sub[:, :min(cut, 64)], None if mask is None else mask[:, :min(cut, 64)],
                          [(inv[:64], Wc, Sc) for inv, Wc, Sc in tables])  # warm-up
    t0 = time.perf_counter()
    torch_cpu_hash_lookup(torch, lay, sub, mask, tables)
    tt = time.perf_counter() - t0
    tcpu = {"value": tokens / tt, "unit": "tokens/s", "cores": threads, "kind": "torch-cpu restatement",
            "sample": f"{what}; vectorised torch CPU ops (int64 hash, fp8 gather, fp32 multiply, bf16 cast) on "
                      f"{threads} threads; {tt:.3f} s"}
    return single, allc, tcpu


def _oracle_task(task):
    """Worker of the all-cores oracle timing (a spawned process): one slice of the oracle's work on
    arrays memory-mapped from the parent's staging directory. Returns the seconds it computed."""
    import numpy as np

    import oracle

    kind, d = task[0], task[1]
    ld = lambda n: np.load(os.path.join(d, n + ".npy"), mmap_mode="r")
    if kind == "warm":
        oracle.lib()
        return 0.0
    if kind == "hash":
        _, _, b, lay_args = task
        ids = np.ascontiguousarray(ld("ids")[b:b + 1])
        mask = None if not os.path.exists(os.path.join(d, "mask.npy")) else np.ascontiguousarray(ld("mask")[b:b + 1])
        n_layers, max_ngram, n_heads, mult, primes, offsets, dead, pad_id = lay_args
        orc = oracle.OracleState(n_layers, max_ngram, n_heads, ld("token_map"), mult, primes, offsets, dead, pad_id,
                                 1, ids.shape[1])
        t0 = time.perf_counter()
        orc.hash(ids, 0, mask)
        return time.perf_counter() - t0
    _, _, l, a, b, n_uniq, D, block, sdt = task
    idx = np.ascontiguousarray(ld(f"inv{l}")[a:b])
    W, S = ld(f"W{l}"), ld(f"S{l}")
    t0 = time.perf_counter()
    oracle.engram_lookup(idx, W, S, n_uniq, D, block, scale_dtype=sdt)
    return time.perf_counter() - t0


def cpu_baseline_all_cores(lay, sub, mask, compact):
    """The same oracle, as it stands, on every host core: a spawned process pool splits the hash by
    sequence and the lookup into index chunks (rows never interact, lookups are independent). The
    inputs are staged once as memory-mapped files; the timed region is the two parallel passes
    (the second of two runs, so page mapping is not timed)."""
    import multiprocessing as mp
    import shutil
    import tempfile

    import numpy as np

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    base = "/dev/shm" if os.path.isdir("/dev/shm") else None
    d = tempfile.mkdtemp(prefix="engram_oracle_", dir=base)
    try:
        np.save(os.path.join(d, "ids.npy"), sub)
        if mask is not None:
            np.save(os.path.join(d, "mask.npy"), mask)
        np.save(os.path.join(d, "token_map.npy"), np.ascontiguousarray(lay.token_map, dtype=np.int64))
        for l, (inv, Wc, Sc, n_uniq) in enumerate(compact):
            np.save(os.path.join(d, f"inv{l}.npy"), inv)
            np.save(os.path.join(d, f"W{l}.npy"), Wc)
            np.save(os.path.join(d, f"S{l}.npy"), Sc)
        lay_args = (lay.n_layers, lay.max_ngram, lay.n_heads, lay.multipliers, lay.primes, lay.offsets, lay.dead,
                    lay.pad_id)
        tasks_h = [("hash", d, b, lay_args) for b in range(sub.shape[0])]
        tasks_l = []
        for l, (inv, _, _, n_uniq) in enumerate(compact):
            step = max(1, -(-inv.size // (4 * cores)))
            tasks_l += [("lookup", d, l, a, min(inv.size, a + step), n_uniq, lay.head_dim, lay.block,
                         lay.scale_dtype)
                        for a in range(0, inv.size, step)]
        with mp.get_context("spawn").Pool(cores) as pool:
            pool.map(_oracle_task, [("warm", d)] * cores)
            for _ in range(2):
                t0 = time.perf_counter()
                pool.map(_oracle_task, tasks_h)
                t1 = time.perf_counter()
                pool.map(_oracle_task, tasks_l, chunksize=1)
                t2 = time.perf_counter()
        return t1 - t0, t2 - t1, cores
    finally:
        shutil.rmtree(d, ignore_errors=True)


def torch_cpu_hash_lookup(torch, lay, ids, mask, tables):
    """A vectorised torch-CPU restatement of the path, for a second CPU number (not the oracle, and
    not on the product path): the n-gram hash of sequences that start at position 0 with no
    history, then the lookup of every row from compact host tables.
    ids int64 [B, L]; mask bool [B, L] or None; tables[l] = (inv, W fp8 codes, S fp32) with inv the
    compact index of each of layer l's B*L*C row ids. Returns (hashes [B, L, Λ, C], [bf16 rows])."""
    import numpy as np

    N, H, NL, C = lay.max_ngram, lay.n_heads, lay.n_layers, lay.n_cols
    dead, pad = int(lay.dead), int(lay.pad_id)
    ids_t = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int64))
    V = int(lay.token_map.size)
    tm = torch.from_numpy(np.ascontiguousarray(lay.token_map, dtype=np.int64))
    valid = (ids_t >= 0) & (ids_t < V)
    c = torch.where(valid, tm[ids_t.clamp(0, V - 1)], torch.full_like(ids_t, dead))
    if mask is not None:
        c = torch.where(torch.from_numpy(np.ascontiguousarray(mask, dtype=bool)), c, torch.full_like(c, dead))
    B, L = c.shape
    pos = torch.arange(L)
    blocked = torch.zeros((B, L), dtype=torch.bool)
    toks = []
    for sft in range(N):  # slot sft holds the token sft positions back; blocking latches
        src = torch.full_like(c, dead)
        if sft < L:
            src[:, sft:] = c[:, :L - sft]
        blocked = blocked | (pos < sft)[None, :] | (src == dead)
        toks.append(torch.where(blocked, torch.full_like(src, pad), src))
    tok = torch.stack(toks, -1)  # [B, L, N]
    mult = torch.from_numpy(np.ascontiguousarray(lay.multipliers, dtype=np.int64).reshape(NL, N))
    prod = tok[:, :, None, :] * mult[None, None]  # int64 products wrap mod 2^64
    P = torch.from_numpy(np.ascontiguousarray(lay.primes, dtype=np.int64).reshape(NL, N - 1, H))
    O = torch.from_numpy(np.ascontiguousarray(lay.offsets, dtype=np.int64).reshape(NL, N - 1, H))
    r = prod[..., 0]
    cols = []
    for i in range(1, N):
        r = r ^ prod[..., i]
        cols.append(torch.remainder(r[..., None], P[None, None, :, i - 1, :]) + O[None, None, :, i - 1, :])
    hashes = torch.stack(cols, 3).reshape(B, L, NL, C)
    rows = []
    for inv, Wc, Sc in tables:
        it = torch.from_numpy(np.ascontiguousarray(inv, dtype=np.int64))
        w = torch.from_numpy(np.ascontiguousarray(Wc))[it].view(torch.float8_e4m3fn).float()  # gather codes, then widen
        sc = torch.from_numpy(np.ascontiguousarray(Sc))[it]
        if lay.scale_dtype != 0:  # the stored bits, widened as `.float()` widens them
            sc = sc.view(scale_torch_dtype(torch, lay.scale_dtype))
        sc = sc.float()
        D = w.shape[-1]
        blk = D // sc.shape[-1]
        rows.append((w.view(-1, sc.shape[-1], blk) * sc[:, :, None]).view(-1, D).to(torch.bfloat16))
    return hashes, rows


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    if rank == 0:
        import __graft_entry__

        __graft_entry__.build()
    barrier(dist, local)
    import gram_hash_embedding_gb300 as geng

    geng._lib()
    l2_default = apply_l2_fetch(geng, args.l2_fetch)
    runner = Runner(args.cfg, rank, device)
    runner.setup_mode(args.mode)
    stream = torch.cuda.current_stream(device)
    K, W = args.steps, args.warmup
    fits_l2 = l2_working_set(runner) < L2_BYTES
    flush_l2 = args.l2 == "flush" or (args.l2 == "auto" and fits_l2 and not args.graph)
    if flush_l2 and args.graph:
        raise SystemExit("--l2 flush times each kernel between flushes; use eager launches (no --graph)")
    for k in range(W):
        runner.step_mode(k)
    torch.cuda.synchronize()
    flags = runner.state.status()

    clocks = ClockSampler(local)
    if args.graph:
        # one graph holds many steps (cycling the distinct id batches), so the replay launch itself
        # is amortised: the time per step is that of back-to-back kernels, as in a serving loop
        n_batches = len(runner.ids)
        per_graph = max(n_batches, (64 // (n_batches * runner.launches_per_step)) * n_batches)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(per_graph):
                runner.step_mode(k)
        for _ in range(3):
            graph.replay()
        replays = max(1, -(-K // per_graph))
        K = replays * per_graph
        stream = torch.cuda.current_stream(device)
        clocks.start()
        total, _ = time_region(torch, dist, local, lambda k: graph.replay(), replays, stream)
        clocks.stop()
        mean_launch = median_launch = total / K
    else:
        flush = None
        if flush_l2:
            l2_scratch = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # twice the 129 MB L2
            flush = lambda k: l2_scratch.fill_(k & 0xFF)  # noqa: E731
        clocks.start()
        total, per_step = time_region(torch, dist, local, runner.step_mode, K, stream, per_launch_events=True,
                                      between=flush)
        clocks.stop()
        mean_launch, median_launch = statistics.mean(per_step), statistics.median(per_step)
        if flush_l2:  # the timed work is the kernels alone; the flushes between them are not counted
            total = sum(per_step)
    total_max = max_over_ranks(dist, total, device)
    tokens = runner.tokens_per_step * K * world
    value = tokens / total_max

    # end to end: host ids in, host bf16 rows out, every step (the fused call)
    runner.e2e_buffers()
    Ke = args.e2e_steps or max(3, min(K, 100))
    for k in range(3):
        runner.e2e_step(k)
    e_total, _ = time_region(torch, dist, local, lambda k: runner.e2e_step(k, drain=k == Ke - 1), Ke, stream)
    e_total = max_over_ranks(dist, e_total, device)
    e_value = runner.tokens_per_step * Ke * world / e_total
    link = link_bandwidth(torch, runner) if rank == 0 else None
    h2d, d2h = runner.e2e_bytes()

    lay = runner.lay
    bpt = runner.mode_bytes_per_token()
    per_launch_tokens = runner.tokens_per_step // runner.launches_per_step
    algo_bytes = per_launch_tokens * bpt
    launch_s = mean_launch / runner.launches_per_step
    peak, peak_kind = measured_peaks()
    achieved = algo_bytes / launch_s / 1e9
    traffic, traffic_note = (recorded_traffic(lay, per_launch_tokens * lay.n_layers * lay.n_cols, args.l2_fetch)
                             if args.mode == "fused" else (None, "recorded for the fused kernel only"))

    cpu = cpu_all = cpu_torch = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not runner.varlen and args.mode == "fused":
        cpu, cpu_all, cpu_torch = cpu_baselines(runner, runner.tokens_per_step)
    csum = clocks.summary()
    wl = runner.wl
    line = {
        "metric": "Engram hash+fp8-gather tokens/s (B8×L8192); gathered HBM GB/s vs peak" if args.mode == "fused"
        else f"Engram {args.mode}-only tokens/s (entry point engram_{args.mode})",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": total_max / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": wl.name if args.cfg != 2 else f"{wl.name}, a run of {DECODE_STEPS} consecutive steps",
            "cfg": args.cfg,
            "B": runner.B,
            "L": runner.L,
            "engram_layers": lay.n_layers,
            "hash_cols": lay.n_cols,
            "head_dim": lay.head_dim,
            "fp8_block": lay.block,
            "table_rows": lay.rows,
            "arithmetic": "hash int64 (wrapping multiply, XOR, floored mod); fp8 E4M3 x "
                          f"{runner.scale_name} scale widened to fp32, one fp32 multiply, RNE to bf16",
            "parallelism": f"replicas x{world} (no exchange step)",
            "l2": l2_note(runner, flush_l2, fits_l2),
            "status_flags_after_warmup": flags,
            "l2_fetch_granularity": (f"{args.l2_fetch} B (context default {l2_default} B)" if args.l2_fetch
                                     else "context default"),
            "launch": "CUDA graph replay" if args.graph else "eager launches from Python",
        },
        "gathered_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "traffic_source": traffic_note, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": algo_bytes, "launch_us": launch_s * 1e6,
                     "launch_us_median": median_launch / runner.launches_per_step * 1e6,
                     "kernel": runner.kernel_name},
        "e2e": {"value": e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": Ke, "ms_per_step": e_total / Ke * 1e3, "call": "engram_hash_lookup",
                "link": link,
                "copy_out": (f"pipelined: {len(runner.e2e_pieces)} calls on groups of batch rows, each group's rows "
                             "copied to the host on a second stream while the next group is computed; steps "
                             "alternate two sets of buffers, so a step's calls overlap the previous step's copies")
                if not runner.varlen and len(runner.chunks) == 1 and len(runner.e2e_pieces) > 1
                else "after the call"},
        "gpu_launches": K * runner.launches_per_step,
        "clocks": csum,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "cpu_torch_restatement": cpu_torch,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- the whole Engram block
def run_block(args):
    """Engram block per step on workload args.cfg: the fused hash + lookup, then for each engram layer
    the wkv projection and the gate (in place on the residual copies), by the path --proj names.
    Weights are seeded synthetic values; dims are the released model's (dim 5120, hc_mult 4)."""
    import numpy as np
    import torch

    import gram_hash_embedding_gb300 as geng

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        import __graft_entry__

        __graft_entry__.build()
    l2_default = apply_l2_fetch(geng, args.l2_fetch)
    runner = Runner(args.cfg, rank, device)
    lay = runner.lay
    T = runner.tokens_per_step
    dim, hc = 5120, 4
    K = lay.n_cols * lay.head_dim
    g = torch.Generator(device="cpu").manual_seed(20261202)
    wkv = [(torch.randn((dim * (hc + 1), K), generator=g) * K ** -0.5).to(torch.bfloat16).to(device)
           for _ in range(lay.n_layers)]
    qw = [torch.rand((hc, dim), generator=g).add_(0.5).to(torch.bfloat16).to(device) for _ in range(lay.n_layers)]
    kw = [torch.rand((hc, dim), generator=g).add_(0.5).to(torch.bfloat16).to(device) for _ in range(lay.n_layers)]
    x = torch.randn((T, hc, dim), generator=g).to(torch.bfloat16).to(device)
    lookahead = args.proj == "lookahead"
    kv = (None if args.proj in ("fused", "lookahead")
          else torch.empty((T, dim * (hc + 1)), dtype=torch.bfloat16, device=device))
    ws = None
    if args.proj == "fused":
        ws = torch.empty(geng.engram_project_gate_workspace(T, hc, dim), dtype=torch.uint8, device=device)
    elif lookahead:
        ws = torch.empty(geng.engram_lookup_project_gate_workspace(T, lay.n_cols, lay.head_dim, hc, dim),
                         dtype=torch.uint8, device=device)
        runner.setup_mode("hash")  # the step hashes only; each layer's rows are looked up inside its projection
        hashes = runner.hash_out.view(T, lay.n_layers, lay.n_cols)
    mask = None if runner.masks[0] is None else runner.masks[0].reshape(-1)
    stream = torch.cuda.current_stream(device)
    if args.proj == "fused":
        names = ["hash+lookup"] + [f"wkv+gate{l}" for l in range(lay.n_layers)]
    elif lookahead:
        names = ["hash"] + [f"lookup+wkv+gate{l}" for l in range(lay.n_layers)]
    else:
        names = ["hash+lookup"] + [f"{n}{l}" for l in range(lay.n_layers) for n in ("wkv", "gate")]

    def step(k, ev=None):
        if ev is not None:
            ev[0].record(stream)
        if lookahead:
            runner.step_mode(k)
        else:
            runner.step(k)
        i = 1
        for l in range(lay.n_layers):
            if ev is not None:
                ev[i].record(stream)
            if lookahead:
                geng.engram_lookup_project_gate(x, hashes[:, l, :], runner.W[l], runner.S[l], wkv[l], qw[l], kw[l],
                                                lay.block, mask, workspace=ws, out=x)
                i += 1
                continue
            emb = runner.out[l].view(T, K)
            if args.proj == "fused":
                geng.engram_project_gate(x, emb, wkv[l], qw[l], kw[l], mask, workspace=ws, out=x)
                i += 1
                continue
            if args.proj == "tcgen05":
                geng.engram_project(emb, wkv[l], out=kv)
            else:
                torch.matmul(emb, wkv[l].t(), out=kv)
            if ev is not None:
                ev[i + 1].record(stream)
            geng.engram_gate(x, kv, qw[l], kw[l], mask, out=x)
            i += 2
        if ev is not None:
            ev[i].record(stream)

    for k in range(max(3, args.warmup // 10)):
        step(k)
    torch.cuda.synchronize()
    K_steps = max(3, min(args.steps, 50))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K_steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    t0.record(stream)
    for k in range(K_steps):
        step(k, evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    total = t0.elapsed_time(t1) / 1e3
    comp = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) * 1e3 for i, n in enumerate(names)}
    eager_ms = total / K_steps * 1e3
    if args.graph:
        # the same steps captured in one CUDA graph and replayed back to back: no host launch gaps
        # (the per-component times above stay those of the eager pass, whose events split the step)
        per_graph = 16
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(per_graph):
                step(k)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        replays = max(1, -(-K_steps // per_graph))
        clocks = ClockSampler(local)
        clocks.start()
        t0.record(stream)
        for _ in range(replays):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        clocks.stop()
        K_steps = replays * per_graph
        total = t0.elapsed_time(t1) / 1e3
    peak_hbm, _ = measured_peaks()
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peaks = json.load(f)
    gemm_flops = 2.0 * T * K * dim * (hc + 1)
    gate_bytes = T * 2.0 * dim * (3 * hc + 1)
    lookup_bytes = T * algo_bytes_per_token(lay)
    if lookahead:  # the hash-only kernel: ids in, cache entries and int64 hash ids out
        roof = {"hash": {"bound": "hbm", "achieved": T * runner.mode_bytes_per_token() / comp["hash"] / 1e3,
                         "peak": peak_hbm, "unit": "GB/s"}}
    else:
        roof = {"hash+lookup": {"bound": "hbm", "achieved": lookup_bytes / comp["hash+lookup"] / 1e3,
                                "peak": peak_hbm, "unit": "GB/s"}}
    proj_kernel = {"fused": "engram_project_gate: tcgen05 projection (CTA pairs) with the gate's sums in its "
                            "epilogue + the gate's finishing pass",
                   "lookahead": "engram_lookup_project_gate: the lookup (warps of every CTA, one tile group ahead) "
                                "inside the tcgen05 projection with the gate's sums in its epilogue + the gate's "
                                "finishing pass",
                   "tcgen05": "engram_project: tcgen05 projection (CTA pairs)",
                   "cublas": "cuBLAS bf16 GEMM (library)"}[args.proj]
    for l in range(lay.n_layers):
        if args.proj in ("fused", "lookahead"):
            name = f"wkv+gate{l}" if args.proj == "fused" else f"lookup+wkv+gate{l}"
            roof[name] = {"bound": "tensor", "achieved": gemm_flops / comp[name] / 1e6,
                          "peak": float(peaks["bf16_tflops_sustained"]), "unit": "TFLOP/s", "kernel": proj_kernel}
            continue
        roof[f"wkv{l}"] = {"bound": "tensor", "achieved": gemm_flops / comp[f"wkv{l}"] / 1e6,
                           "peak": float(peaks["bf16_tflops_sustained"]), "unit": "TFLOP/s", "kernel": proj_kernel}
        roof[f"gate{l}"] = {"bound": "hbm", "achieved": gate_bytes / comp[f"gate{l}"] / 1e3, "peak": peak_hbm,
                            "unit": "GB/s"}
    for r in roof.values():
        r["frac"] = r["achieved"] / r["peak"]
    line = {
        "metric": "Engram block (hash + fp8 lookup + wkv projection + gate) tokens/s",
        "value": T * K_steps / total, "unit": "tokens/s", "n_gpus": 1, "steps": K_steps,
        "ms_per_step": total / K_steps * 1e3, "higher_is_better": True, "dtype": "bf16/f32", "data": "synthetic",
        "config": {"workload": runner.wl.name, "dim": dim, "hc_mult": hc, "wkv": [dim * (hc + 1), K],
                   "projection": args.proj,
                   "l2_fetch_granularity": (f"{args.l2_fetch} B (context default {l2_default} B)" if args.l2_fetch
                                            else "context default"),
                   "launch": ("CUDA graph replay (16 steps per graph); component times from an eager pass"
                              if args.graph else "eager launches from Python")},
        "eager_ms_per_step": eager_ms,
        "component_us": comp, "roofline": roof, "clocks": clocks.summary(),
        # ours per step: the fused hash + lookup, and per layer projection + finishing pass (fused), projection +
        # gate (tcgen05), or the gate alone (cublas: the projection is cuBLAS's)
        "gpu_launches": K_steps * (runner.launches_per_step +
                                   lay.n_layers * {"cublas": 1, "lookahead": 3}.get(args.proj, 2)),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- sharded lookup's device steps
def run_shard(args):
    """engram_shard_pack and engram_shard_unpack on the row ids of one engram layer of workload
    args.cfg (the hash is computed once, untimed), for args.shard ranks, CUDA events over the launches."""
    import numpy as np
    import torch

    import gram_hash_embedding_gb300 as geng
    import synth

    torch.cuda.set_device(0)
    import __graft_entry__

    __graft_entry__.build()
    wl = synth.make_workload(args.cfg)
    lay = wl.layout
    st = geng.EngramHash(n_layers=lay.n_layers, max_ngram=lay.max_ngram, n_heads=lay.n_heads, head_dim=lay.head_dim,
                         block=lay.block, max_batch=wl.max_batch, max_seq_len=wl.max_seq_len, token_map=lay.token_map,
                         multipliers=lay.multipliers, primes=lay.primes, offsets=lay.offsets, dead=lay.dead,
                         pad_id=lay.pad_id)
    ids = torch.from_numpy(np.ascontiguousarray(wl.ids.reshape(wl.B, -1)[:, :wl.L])).cuda()
    idx = st.hash(ids, 0)[:, :, 0, :].contiguous().reshape(-1)
    n, world, rows, D = idx.numel(), int(args.shard), int(lay.rows[0]), lay.head_dim
    L = geng._lib()
    s = torch.cuda.current_stream().cuda_stream
    counts = torch.empty(world + 1, dtype=torch.int64, device="cuda")
    local = torch.empty(n, dtype=torch.int64, device="cuda")
    pos = torch.empty(n, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(int(L.engram_shard_pack_workspace(n, world)), 16), dtype=torch.uint8, device="cuda")
    recv = torch.zeros((n, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((n, D), dtype=torch.bfloat16, device="cuda")

    def pack():
        L.engram_shard_pack(idx.data_ptr(), n, rows, world, counts.data_ptr(), local.data_ptr(), pos.data_ptr(),
                            ws.data_ptr(), ws.numel(), s)

    def unpack():
        L.engram_shard_unpack(recv.data_ptr(), pos.data_ptr(), n, n, D, out.data_ptr(), s)

    def timed(fn, k):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(k):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / k * 1e3

    K = max(3, min(args.steps, 200))
    t_pack, t_unpack = timed(pack, K), timed(unpack, K)
    pack_bytes = n * (8 + 8 + 16)  # two passes over the ids, local row + position written
    unpack_bytes = n * (8 + 4 * D)  # position read, row read and written
    peak, peak_kind = measured_peaks()
    line = {"metric": "sharded lookup device steps (us per launch pair)", "workload": wl.name, "indices": n,
            "world": world, "head_dim": D, "steps": K,
            "pack_us": t_pack, "pack_gbs": pack_bytes / t_pack / 1e3,
            "unpack_us": t_unpack, "unpack_gbs": unpack_bytes / t_unpack / 1e3,
            "unpack_frac_of_hbm": unpack_bytes / t_unpack / 1e3 / peak, "peak_kind": peak_kind,
            "counts": [int(c) for c in counts.cpu()]}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as it stands, timed on the host cores: each step hashes a bounded sample of
    the workload (the first T tokens of one of its sequences, in turn) and looks up every row
    those tokens touch."""
    import numpy as np

    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    import synth

    oracle.build()
    wl = synth.make_workload(args.cfg)
    lay = wl.layout
    K, W = args.steps, args.warmup
    # size each step so the whole run stays within about two minutes of oracle time
    est_tok_s = 6000.0
    T = int(max(8, min(wl.L if args.cfg != 4 else 8192, est_tok_s * 120.0 / max(1, K + W))))
    ids_all = wl.ids
    B = ids_all.shape[0]
    samples = []
    for b in range(min(B, 8)):
        sub = np.ascontiguousarray(ids_all[b:b + 1, :T])
        msk = None if wl.mask is None else np.ascontiguousarray(wl.mask[b:b + 1, :T])
        orc = oracle.OracleState.from_layout(lay, 1, T)
        h, _ = orc.hash(sub, 0, msk)
        tabs = []
        for l in range(lay.n_layers):
            flat = h[:, :, l, :].reshape(-1)
            uniq, inv = np.unique(flat, return_inverse=True)
            Wc = synth.table_rows(wl.table_seed, l, uniq, lay.head_dim)
            Sc = synth.table_scales(wl.table_seed, l, uniq, lay.n_scales, lay.scale_dtype)
            tabs.append((uniq, Wc, Sc))
        samples.append((sub, msk, orc, tabs))

    def one(k):
        sub, msk, orc, tabs = samples[k % len(samples)]
        orc.reset()
        t0 = time.perf_counter()
        h, _ = orc.hash(sub, 0, msk)
        el = time.perf_counter() - t0
        for l, (uniq, Wc, Sc) in enumerate(tabs):
            local_idx = np.searchsorted(uniq, h[:, :, l, :].reshape(-1))
            t0 = time.perf_counter()
            oracle.engram_lookup(local_idx, Wc, Sc, uniq.size, lay.head_dim, lay.block, scale_dtype=lay.scale_dtype)
            el += time.perf_counter() - t0
        return el

    for k in range(W):
        one(k)
    total = sum(one(k) for k in range(K))
    value = T * K / total
    sample = (f"each step: the first {T} tokens of one sequence of the workload (cycling over {len(samples)}), "
              f"hash + lookup of their {T * lay.n_layers * lay.n_cols} rows from compact host tables; "
              "single-threaded C oracle")
    line = {
        "impl": "reference",
        "metric": "Engram hash+fp8-gather tokens/s (B8×L8192); gathered HBM GB/s vs peak" if args.mode == "fused"
        else f"Engram {args.mode}-only tokens/s (entry point engram_{args.mode})",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "cfg": args.cfg, "sample_tokens_per_step": T},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.block:
        run_block(args)
    elif args.shard:
        run_shard(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
