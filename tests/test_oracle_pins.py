"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import pins

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def test_philox_matches_triton_philox(orc, philox_ref):
    pins.pin_philox_matches_reference(orc, *philox_ref)


def test_element_counter_word_mapping(orc, philox_ref):
    pins.pin_element_mapping(orc, *philox_ref)


def test_philox_fill_layout(orc, philox_ref):
    pins.pin_philox_fill_layout(orc, *philox_ref)


def test_philox_statistics(orc):
    pins.pin_philox_statistics(orc)


def test_sr_exhaustive_unbiased(orc):
    pins.pin_sr_exhaustive(orc)


def test_sr_inf_nan(orc):
    pins.pin_sr_inf_nan(orc)


def test_sr_mean_with_philox_bits(orc):
    pins.pin_sr_mean_with_philox(orc)


def test_rne_matches_torch(orc):
    pins.pin_rne_matches_torch(orc)


def test_adamw_tracks_textbook_fp64(orc):
    pins.pin_adamw_textbook(orc)


def test_adamw_tracks_torch(orc):
    pins.pin_adamw_torch(orc)


def test_adamw_special_cases(orc):
    pins.pin_adamw_special_cases(orc)


def test_adamw_one_step_tight(orc):
    pins.pin_adamw_one_step_tight(orc)


def test_adamw_dtype_paths(orc):
    pins.pin_adamw_dtype_paths(orc)


def test_scalars(orc):
    pins.pin_scalars(orc)


def test_subulp_demo_increment(orc):
    pins.pin_demo_increment(orc)


def test_subulp_demo_adamw(orc):
    pins.pin_demo_adamw(orc)


def test_shard_invariance(orc):
    pins.pin_shard_invariance(orc)


def test_no_fp_contraction(orc):
    pins.pin_no_contraction(orc)


def test_gemm_exact_small(orc):
    pins.pin_gemm_exact_small(orc)


def test_gemm_closed_forms(orc):
    pins.pin_gemm_closed_forms(orc)
