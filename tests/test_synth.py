"""Host-side checks of the seeded input generators (CPU only)."""
import numpy as np

import synth


def test_generator_is_counter_based_and_deterministic():
    a = synth.words(1, 2, np.arange(10, dtype=np.uint64))
    b = synth.words(1, 2, np.arange(5, 10, dtype=np.uint64))
    assert np.array_equal(a[5:], b)
    assert not np.array_equal(a, synth.words(2, 2, np.arange(10, dtype=np.uint64)))
    # splitmix64 reference values (Vigna's splitmix64.c seeded with 0: first outputs)
    z = np.array([0x9E3779B97F4A7C15, (2 * 0x9E3779B97F4A7C15) % 2 ** 64], dtype=np.uint64)
    assert [int(v) for v in synth.mix64(z)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_fp8_lut_is_normal_and_nan_free():
    lut = synth.fp8_normal_lut()
    assert lut.shape == (65536,) and lut.dtype == np.uint8
    assert not np.isin(lut, [0x7F, 0xFF]).any()
    import torch

    vals = torch.from_numpy(lut.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1.0) < 0.05
    assert np.all(np.diff(vals) >= 0)  # monotone in the uniform


def test_table_rows_and_scales():
    rows = np.array([0, 1, 5, 10 ** 8 + 3])
    W = synth.table_rows(3, 1, rows, 128)
    assert W.shape == (4, 128) and W.dtype == np.uint8
    assert np.array_equal(W[2], synth.table_rows(3, 1, [5], 128)[0])
    assert not np.array_equal(W[0], synth.table_rows(3, 0, [0], 128)[0])  # layers differ
    S = synth.table_scales(3, 1, rows, 2)
    assert S.dtype == np.float32 and (S >= 0.01).all() and (S < 1.0).all()


def test_workloads_shapes():
    w0 = synth.make_workload(0)
    assert w0.ids.shape == (1, 64) and w0.layout.rows[0] == int(w0.layout.primes.sum())
    assert (w0.layout.primes >= 997).all() and (w0.layout.primes <= 2003).all()
    assert len(set(w0.layout.primes.reshape(-1).tolist())) == 6
    m = w0.layout.multipliers
    assert (m % 2 == 1).all() and (m >= 1).all() and (m < 2 ** 31).all()
    w1 = synth.make_workload(1)
    assert w1.ids.shape == (4, 4096) and abs((~w1.mask).mean() - 0.10) < 0.01
    assert (w1.ids[~w1.mask] == synth.IMAGE_TOKEN_ID).all()
    assert w1.layout.n_cols == 24 and 23e6 < w1.layout.rows[0] < 25e6
    w4 = synth.make_workload(4)
    frac = (~w4.mask[0, :8192]).mean()
    assert abs(frac - 0.15) < 0.01 and w4.mask[0, 8192:].all()
    # Zipf ids repeat
    assert len(np.unique(w4.ids)) < 0.5 * w4.ids.size


def test_scale_codes_of_the_other_storage_types():
    """bf16 / UE8M0 / E4M3 scale patterns: the documented ranges, finite and positive, and the
    released head_dim workload with UE8M0 scales."""
    rows = np.arange(4000)
    bf = synth.table_scales(5, 0, rows, 2, synth.SCALE_BF16)
    e8 = synth.table_scales(5, 0, rows, 2, synth.SCALE_E8M0)
    e4 = synth.table_scales(5, 0, rows, 2, synth.SCALE_E4M3)
    assert bf.dtype == np.uint16 and e8.dtype == np.uint8 and e4.dtype == np.uint8
    bfv = (bf.astype(np.uint32) << 16).view(np.float32)
    assert (bfv >= 2.0 ** -7).all() and (bfv < 2.0).all() and len(np.unique(bf)) > 500
    assert set(np.unique(e8).tolist()) == set(range(120, 128))
    e4_exp = (e4 >> 3) & 0xF
    assert (e4 < 0x80).all() and set(np.unique(e4_exp).tolist()) == {4, 5, 6, 7}
    # the same counters as the fp32 scales: row r, scale j is one word whatever the storage type
    assert np.array_equal(synth.table_scales(5, 0, [7, 9], 2, synth.SCALE_E8M0), e8[[7, 9]])
    w8 = synth.make_workload(8)
    assert w8.layout.head_dim == 256 and w8.layout.scale_dtype == synth.SCALE_E8M0 and w8.layout.scale_bytes == 1
    assert w8.layout.rows == synth.make_workload(6).layout.rows
