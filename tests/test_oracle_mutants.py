"""The pins must catch plausible mistakes in the oracle.

Each case copies the oracle's C source to a temporary directory, plants one
mistake (a dropped term, a wrong sign or index, a transposed operand),
compiles it, and checks that at least one pin fails on that build. Mistakes
are planted only in these CPU copies.
"""
import os
import shutil
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "engram_oracle.c")

MUTANTS = {
    "lookback_forward": ("pos - shift < 0 ? 0 : pos - shift", "pos + shift"),
    "no_position_block": ("blocked || (pos < shift) || (source == dead)", "blocked || (source == dead)"),
    "no_dead_block": ("blocked || (pos < shift) || (source == dead)", "blocked || (pos < shift)"),
    "non_cumulative_block": ("blocked = blocked || (pos < shift)", "blocked = (pos < shift)"),
    "pad_swapped": ("tokens[shift] = blocked ? pad_id : source;", "tokens[shift] = blocked ? source : pad_id;"),
    "mask_to_pad": ("if (mask != NULL && !mask[t]) c = dead;", "if (mask != NULL && !mask[t]) c = pad_id;"),
    "mask_ignored": ("if (mask != NULL && !mask[t]) c = dead;", ""),
    "xor_as_add": ("rolling ^= products[i];", "rolling += products[i];"),
    "first_product_dropped": ("uint64_t rolling = products[0];", "uint64_t rolling = 0;"),
    "multiplier_index": ("multipliers[l * max_ngram + k]", "multipliers[k]"),
    "prime_head_dropped": ("primes[(l * (max_ngram - 1) + (i - 1)) * n_heads + h]",
                           "primes[(l * (max_ngram - 1) + (i - 1)) * n_heads]"),
    "column_transposed": ("const int64_t col = (i - 1) * n_heads + h;", "const int64_t col = h * (max_ngram - 1) + (i - 1);"),
    "offset_dropped": ("oracle_floor_mod(x, p) + offsets[l * C + col]", "oracle_floor_mod(x, p)"),
    "truncated_mod": ("if (r != 0 && ((r < 0) != (p < 0))) r += p;", ""),
    "mod_sign_flipped": ("if (r != 0 && ((r < 0) != (p < 0))) r += p;", "if (r != 0 && ((r < 0) != (p < 0))) r -= p;"),
    "unsigned_mod": ("const int64_t x = (int64_t)rolling;", "const int64_t x = (int64_t)(rolling >> 1);"),
    "cache_write_shift": ("cache_row[s + t] = c;", "cache_row[t] = c;"),
    "varlen_offset_dropped": ("ids + begin, mask ? mask + begin : NULL", "ids, mask"),
    "varlen_cache_row": ("offsets, cache + r * cache_len, cache_len, ids + begin", "offsets, cache, cache_len, ids + begin"),
    "dense_cache_row": ("offsets, cache + r * cache_len, cache_len, ids + b * L", "offsets, cache + b * cache_len, cache_len, ids + b * L"),
    "cache_rows_ignored": ("const int64_t r = cache_rows ? cache_rows[b] : b;", "const int64_t r = b;"),
    "bad_row_not_flagged": ("      fl |= ORACLE_FLAG_BAD_ROW;\n      continue;", "      continue;"),
    "fp8_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e8m0_bias": ("return (float)ldexp(1.0, (int)e - 127);", "return (float)ldexp(1.0, (int)e - 128);"),
    "e8m0_nan_dropped": ("  if (e == 0xFF) return NAN;\n", ""),
    "bf16_widen_shift": ("const uint32_t u = (uint32_t)h << 16;", "const uint32_t u = (uint32_t)h << 15;"),
    "scale_dtype_ignored": ("    case ORACLE_SCALE_E8M0: return oracle_e8m0_to_f32(((const uint8_t*)S)[i]);\n", ""),
    "fp8_subnormal": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "fp8_mantissa": ("1.0 + (double)m / 8.0", "1.0 + (double)m / 16.0"),
    "fp8_sign": ("return (float)(sign ? -v : v);", "return (float)v;"),
    "bf16_truncate": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) {", "if (0) {"),
    "bf16_ties_away": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "scale_block_index": ("scale_at(S, scale_dtype, local * n_scales + k / block)",
                          "scale_at(S, scale_dtype, local * n_scales + k % n_scales)"),
    "scale_row_index": ("scale_at(S, scale_dtype, local * n_scales + k / block)", "scale_at(S, scale_dtype, k / block)"),
    "masked_rows_read": ("const int64_t local = out_of_range ? 0 : r;", "const int64_t local = out_of_range ? 0 : r;\n    const int dummy_ = out_of_range; (void)dummy_;"),
}
# the last one is a no-op control: it must *survive* (proves the harness can pass)
CONTROL = "masked_rows_read"


def _build_variant(name, old, new, tmp):
    src = open(SRC).read()
    assert old in src, f"mutation {name}: pattern not found"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    return oracle.load_variant(oracle.build(force=True, src=path, out=os.path.join(tmp, f"lib{name}.so")))


def _pins_fail(L):
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(L)
        except (AssertionError, ValueError, IndexError, OverflowError):
            return pin.__name__
    return None


@pytest.fixture(scope="module")
def tmpdir_mut():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmpdir_mut):
    old, new = MUTANTS[name]
    L = _build_variant(name, old, new, tmpdir_mut)
    caught = _pins_fail(L)
    if name == CONTROL:
        assert caught is None, f"control build failed pin {caught}"
    else:
        assert caught is not None, f"planted mistake {name} passed every pin"


# ----------------------------------------------------------------------------- the float64 gate oracle
GATE_MUTANTS = {
    "norm_over_copies": ("(h * h).mean(-1)", "(h * h).mean(-2, keepdims=True).squeeze(-2)[:, None].repeat(h.shape[1], 1)"),
    "weight_dropped": ("(h * weight[None] * key)", "(h * key)"),
    "no_dim_scale": (" * rstd * dim ** -0.5", " * rstd"),
    "sign_lost": ("np.copysign(np.sqrt(np.maximum(np.abs(dot), clamp)), dot)", "np.sqrt(np.maximum(np.abs(dot), clamp))"),
    "sigmoid_flipped": ("1.0 / (1.0 + np.exp(-signed_sqrt))", "1.0 / (1.0 + np.exp(signed_sqrt))"),
    "mask_inverted": ("np.where(np.asarray(mask, dtype=bool)[:, None], gate, 0.0)",
                      "np.where(np.asarray(mask, dtype=bool)[:, None], 0.0, gate)"),
    "value_per_copy": ("h + gate[..., None] * value[:, None, :]", "h + gate[..., None] * key"),
    "key_shifted": ("key, value = kv[:, :hc, :], kv[:, hc, :]", "key, value = kv[:, 1:, :], kv[:, 0, :]"),
    "sqrt_dropped": ("np.sqrt(np.maximum(np.abs(dot), clamp))", "np.maximum(np.abs(dot), clamp)"),
}


@pytest.mark.parametrize("name", sorted(GATE_MUTANTS))
def test_planted_gate_mistake_is_caught(name):
    import inspect

    src = inspect.getsource(oracle.engram_gate)
    old, new = GATE_MUTANTS[name]
    assert old in src, f"gate mutation {name}: pattern not found"
    ns = dict(vars(oracle))
    exec(src.replace(old, new, 1), ns)
    with pytest.raises((AssertionError, ValueError, IndexError)):
        oracle_pins.pin_gate(ns["engram_gate"])
    oracle_pins.pin_gate(oracle.engram_gate)  # the real one passes
