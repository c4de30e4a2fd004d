"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import synth
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_released_table_rows_from_prime_search():
    """The released row counts equal the sums of consecutive primes above engram_vocab_size,
    dealt 24 per layer in ascending order; the column offsets then tile [0, rows)."""
    cfg = {}
    with open(__file__.replace("test_oracle_pins.py", "golden/released_config.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                cfg[k] = [int(x) for x in v]
    n_layers = len(cfg["engram_layer_ids"])
    primes = synth.layered_primes(cfg["engram_vocab_size"][0], n_layers, cfg["engram_max_ngram_size"][0],
                                  cfg["engram_n_heads"][0])
    rows = [int(primes[l].sum()) for l in range(n_layers)]
    assert rows == cfg["engram_num_embeddings"]
    off = synth.column_offsets(primes)
    flat = primes.reshape(n_layers, -1)
    assert (off[:, 0] == 0).all() and ((off + flat)[:, -1] == np.array(rows)).all()
    assert (off[:, 1:] == (off + flat)[:, :-1]).all()


def test_oracle_hash_rejects_bad_shapes():
    lay = synth.make_layout("tiny", 1)
    st = oracle.OracleState.from_layout(lay, 1, 8)
    with pytest.raises(ValueError):
        st.hash(np.zeros((2, 4), np.int64), 0)  # B > cache rows


@pytest.mark.parametrize("pin", [oracle_pins.pin_bf16_from_f64, oracle_pins.pin_linear, oracle_pins.pin_gate],
                         ids=lambda f: f.__name__)
def test_gate_pin(pin):
    pin()
