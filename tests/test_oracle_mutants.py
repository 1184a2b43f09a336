"""The oracle's pins catch plausible mistakes.

Each mutant is the oracle compiled with one deliberate mistake planted in it
(K6O_MUTANT in oracle/k6_oracle.c): a wrong rotation sign, a dropped factor in
the rotary frequency, swapped grid axes, the wrong softmax scale, a merge
weighted by the maximum instead of the log-sum-exp, transposed relayout
indices, a log-sum-exp without its maximum, joint keys read from the video
tensor, a backward pass without its D_i term.  Every mutant must fail at
least one pin; the oracle itself passes all.
"""
import numpy as np
import pytest

from oracle import oracle as O

from . import test_oracle_pins as pins

CHECKS = {
    "decimal brute force": lambda: pins.test_attention_matches_decimal_brute_force(8, 3, 2.0),
    "torch sdpa": pins.test_attention_matches_torch_sdpa_fp64,
    "identical keys": pins.test_identical_keys_give_mean_of_values,
    "unequal chunks": pins.test_unequal_chunks_merge_equals_unchunked,
    "merge decimal": pins.test_merge_matches_decimal_definition,
    "rope norm": pins.test_rope_preserves_each_pair_norm,
    "rope relative t": lambda: pins.test_rope_relative_position_property(0),
    "rope frequency ladder": pins.test_rope_frequency_ladder_and_axis_segments,
    "rope 1-d complex": pins.test_rope_1d_joint_equals_complex_product,
    "relayout transpose": lambda: pins.test_relayout_matches_transpose_and_round_trips(1, 40, 24, 8, 8, np.uint16),
    "backward differences": pins.test_backward_matches_central_differences_of_the_forward,
}


def run_checks():
    failed = []
    for name, check in CHECKS.items():
        try:
            check()
        except AssertionError:
            failed.append(name)
    return failed


@pytest.fixture
def restore_oracle():
    yield
    O.use_mutant(0)


def test_oracle_itself_passes_every_check(restore_oracle):
    O.use_mutant(0)
    assert run_checks() == []


@pytest.mark.parametrize("mutant", range(1, 10))
def test_pins_catch_a_planted_mistake(mutant, restore_oracle):
    O.use_mutant(mutant)
    failed = run_checks()
    assert failed, f"planted mistake {mutant} passed every pin"
    print(mutant, failed)
