"""Host-side pieces of bench.py (no GPU): argument defaults, the byte model, the traffic record,
the clock-sample parser."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_defaults_run_the_full_scale_workload():
    a = bench.parse_args([])
    assert a.cfg == 3 and a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"


def test_algorithmic_bytes_per_token():
    lay = synth.make_layout("full", 1)
    assert bench.algo_bytes_per_token(lay) == 18_624  # 2 x 24 x (128 + 4 + 256)
    assert bench.algo_bytes_per_token(synth.make_layout("tiny", 1)) == 6 * (32 + 4 + 64)


def test_traffic_record_matches_the_kernel_sources():
    # the committed ncu record (profiling case) is only used for the kernel and row format it was
    # taken on, at the fetch limit it was taken at, and scales with the gathered rows
    full = synth.make_layout("full", 1)
    rows = 65_536 * 48
    t, note = bench.recorded_traffic(full, rows, 32)
    assert t is None or (1.0e9 < t < 1.45e9 and "scaled" in note), (t, note)
    if t is not None:
        t2, _ = bench.recorded_traffic(full, rows // 4, 32)
        assert abs(t2 * 4 - t) < 1.0
    assert bench.recorded_traffic(full, rows, 64)[0] is None
    assert bench.recorded_traffic(synth.make_layout("tiny", 1), rows, 32)[0] is None  # head_dim 32


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1900, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1985 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def _compact_tables(lay, hashes, seed):
    import numpy as np

    out = []
    for l in range(lay.n_layers):
        uniq, inv = np.unique(hashes[:, :, l, :].reshape(-1), return_inverse=True)
        W = synth.table_rows(seed, l, uniq, lay.head_dim)
        S = synth.table_scales(seed, l, uniq, lay.n_scales)
        out.append((inv.astype(np.int64), W, S, int(uniq.size)))
    return out


def test_torch_cpu_restatement_equals_the_oracle():
    """The second CPU number comes from a vectorised torch restatement; it must compute exactly what
    the oracle computes (hash ids and bf16 rows), including masks, invalid ids, full 64-bit
    multipliers (negative running values) and two scale blocks per row."""
    import numpy as np
    import torch

    import oracle

    rng = np.random.default_rng(5)
    lays = [synth.make_layout("tiny", 3, full64=True), synth.make_layout("tiny", 4)]
    p = synth.distinct_primes_in(9, 997, 2003, (2, 3, 4))
    lays.append(synth.Layout(2, 4, 4, 64, 32, 500, 90, synth.uniform_int(9, synth.TAG_TOKEN_MAP, 500, 0, 90),
                             synth.multipliers(9, 2, 4, full64=True), p, synth.column_offsets(p)))
    for i, lay in enumerate(lays):
        B, L = 3, 70
        ids = rng.integers(-2, lay.raw_vocab + 2, size=(B, L))
        mask = rng.random((B, L)) > 0.2 if i != 1 else None
        exp_h, _ = oracle.OracleState.from_layout(lay, B, L).hash(ids, 0, mask)
        compact = _compact_tables(lay, exp_h, 40 + i)
        h, rows = bench.torch_cpu_hash_lookup(torch, lay, ids, mask, [(a, W, S) for a, W, S, _ in compact])
        assert np.array_equal(h.numpy(), exp_h), i
        for l, (inv, W, S, n) in enumerate(compact):
            exp = oracle.engram_lookup(inv, W, S, n, lay.head_dim, lay.block)
            got = rows[l].view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got, exp.reshape(got.shape)), (i, l)


def test_all_cores_oracle_timing_runs():
    import numpy as np

    import oracle

    lay = synth.make_layout("tiny", 6)
    ids = np.random.default_rng(6).integers(0, lay.raw_vocab, size=(2, 300))
    h, _ = oracle.OracleState.from_layout(lay, 2, 300).hash(ids, 0)
    th, tl, cores = bench.cpu_baseline_all_cores(lay, ids, None, _compact_tables(lay, h, 6))
    assert th > 0 and tl > 0 and cores >= 1


def test_l2_working_set_decides_the_flush():
    """Decode steps touch a few MB of rows (they fit in L2, so the bench flushes L2 between them by
    default); the prefill and full-scale steps touch far more than L2."""
    from types import SimpleNamespace

    lay = synth.make_layout("prefill", 1)
    decode = SimpleNamespace(lay=lay, tokens_per_step=256, ids=[0] * 4)
    full = SimpleNamespace(lay=synth.make_layout("full", 1), tokens_per_step=65536, ids=[0] * 4)
    assert bench.l2_working_set(decode) < bench.L2_BYTES < bench.l2_working_set(full)
    assert "flushed" in bench.l2_note(decode, True, True) and "warm" in bench.l2_note(decode, False, True)
    assert "larger than L2" in bench.l2_note(full, False, False)
    assert bench.parse_args([]).l2 == "auto"
