"""Plant one mistake at a time in the oracle (a CPU rebuild of its C source) and
check that the pins catch every one of them."""
import os

import pytest

import oracle
import test_layouts as layouts
import test_oracle_bwd_pins as bwd_pins
import test_oracle_pins as pins

PINS = [
    pins.test_worked_example_ring_simulator,
    lambda: pins.test_zero_query_gives_mean_of_visible_values(True),
    pins.test_single_visible_key,
    pins.test_dominant_key_selects_its_value,
    lambda: pins.test_matches_torch_float64_softmax(True),
    pins.test_lse_gradient_is_attention_over_keys,
    lambda: pins.test_shard_partials_merge_to_unsharded(True),
    pins.test_fanout_equals_per_branch_attention_over_prefix_plus_suffix,
    lambda: layouts.test_oracle_on_stored_layout_equals_sequence_order("zigzag"),
    pins.test_fanout_prefill_equals_causal_attention_over_prefix_plus_suffix,
    lambda: bwd_pins.test_bwd_finite_differences(True),
    lambda: bwd_pins.test_bwd_matches_torch_float64_autograd(True, 6, 2),
]

MUTANTS = {
    1: "softmax scale 1/d instead of 1/sqrt(d)",
    2: "causal mask drops the diagonal",
    3: "lse in log2 instead of ln",
    4: "interleaved GQA head map",
    5: "scores against V instead of K",
    6: "last visible key dropped",
    7: "merge forgets to normalise",
    8: "causal mask on the stored order instead of sequence positions",
    9: "backward: softmax Jacobian's row term dropped",
    10: "backward: dK without the softmax scale",
    11: "fan-out prefill: a row does not see its own suffix token",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    path = oracle.build(mutant=mutant, out=os.path.join(tmp_path, f"liboracle_m{mutant}.so"))
    caught = []
    oracle.use_library(path)
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin)
    finally:
        oracle.use_library(None)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"
