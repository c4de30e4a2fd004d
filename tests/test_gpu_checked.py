"""The checked build (-DENGRAM_CHECKED=1: every global access of the hash and fused kernels is tested
against the call's sizes, and one outside them is skipped and raises STATUS_CHECK) runs random
parity cases, packed calls and the grid-limit batch: results equal the oracle's and no access was
out of bounds (GPU only). Built beside the release library, in its own file."""
import os

import pytest

import gram_hash_embedding_gb300 as geng
from gram_hash_embedding_gb300 import _build
from tests import gpu_helpers as H
from tests import test_gpu_parity, test_gpu_random_sweep, test_gpu_varlen

pytestmark = pytest.mark.gpu

CHECKED = os.path.join(os.path.dirname(_build.LIB), "libengram_checked.so")


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    H.build_all()
    _build.build(extra_flags=["-DENGRAM_CHECKED=1"], lib_path=CHECKED)
    saved = geng._LIB_PATH, geng._lib_handle
    geng._LIB_PATH, geng._lib_handle = CHECKED, None
    try:
        yield
    finally:
        geng._LIB_PATH, geng._lib_handle = saved


def test_the_checked_library_is_loaded():
    geng._lib()
    assert geng._lib_handle._name == CHECKED


@pytest.mark.parametrize("seed", range(0, 48, 2))
def test_random_cases(seed):
    # each case asserts that the state's status equals the oracle's flags, so a STATUS_CHECK fails it
    test_gpu_random_sweep.test_random_case(seed)


@pytest.mark.parametrize("lens", [[5, 0, 17, 1, 40, 3, 16, 33], [0, 0, 0, 7]])
def test_packed(lens):
    test_gpu_varlen.test_packed_matches_oracle(lens)


def test_grid_limit_batch():
    test_gpu_parity.test_batch_at_the_grid_limit()
