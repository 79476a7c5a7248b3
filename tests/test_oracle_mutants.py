"""Mutation check of the oracle's pins: each test-only oracle build with one
planted, plausible mistake (a wrong ape row, swapped kv halves, a missing
first-group mask, buffer_len off by one, a short write set, a decode slot off
by one, a ragged id without its request offset, a wrong read page, a dropped
term, a sign error, an input row off by one; in the SWA-paged planner: no
page-end writes, the ring offset taken modulo the page size, records without
state reads translated; in norm + RoPE: a rotation sign, the position, the
rotated channels; in the online state: no reset at a group start, the sum not
rescaled, an ape row off by one) must fail at least one pin."""
import pytest

from tests import test_oracle_norm_rope as N
from tests import test_oracle_online as L
from tests import test_oracle_paged as Q
from tests import test_oracle_pins as P

MUTANTS = {
    1: "ape row off by one",
    2: "C4 overlap entries read the main kv half",
    3: "first-group mask missing",
    4: "buffer_len off by one",
    5: "C4 write set without the overlap group",
    6: "decode write slot off by one",
    7: "ragged id without the request offset",
    8: "read_page_0 of the current group",
    9: "a dropped denominator term",
    10: "sign error in the exponent",
    11: "input row off by one",
    12: "paged C4 write set without the SWA page ends",
    13: "paged ring offset modulo the SWA page size",
    14: "paged records without state reads translated",
    15: "RoPE rotation sign",
    16: "RoPE position seq_len instead of seq_len - ratio",
    17: "RoPE on the first rope_dim channels",
    18: "online state not reset at a group start",
    19: "online sum not rescaled on a new maximum",
    20: "online ape row off by one",
}


def pins(o):
    yield lambda: P.test_plan_worked_examples(o)
    for ratio in (4, 128):
        yield lambda ratio=ratio: P.test_plan_bruteforce(o, ratio, 1)
        yield lambda ratio=ratio: P.test_equal_scores_give_window_mean(o, ratio)
        yield lambda ratio=ratio: P.test_dominant_ape_selects_entry_and_column(o, ratio)
    yield lambda: P.test_c4_first_group_masks_previous_group(o)
    yield lambda: P.test_pool_matches_float64_torch_softmax(o, 4, 0, 0)
    yield lambda: P.test_pool_matches_float64_torch_softmax(o, 128, 1, 0)
    yield lambda: P.test_decode_nonboundary_rows_are_zero(o)
    for ratio in (4, 128):
        yield lambda ratio=ratio: P.test_modes_equal_history(o, ratio, 0)
    for ratio in (4, 128):
        yield lambda ratio=ratio: Q.test_identity_mapping_gives_legacy_plans(o, ratio, 0)
    yield lambda: Q.test_page_end_positions_are_written_before_first_write(o)
    yield lambda: Q.test_paged_schedules_equal_history(o, 0)
    yield lambda: N.test_constant_row_normalises_to_the_weight(o)
    yield lambda: N.test_matches_float64_torch(o, 1)
    yield lambda: N.test_rotation_keeps_pair_lengths_and_relative_positions(o)
    yield lambda: N.test_position_is_seq_len_minus_ratio(o)
    yield lambda: L.test_online_plan_worked_example(o)
    yield lambda: L.test_online_closed_forms(o)
    yield lambda: L.test_online_schedules_equal_window_definition(o, 0)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(oracle_mod, mutant):
    o = oracle_mod
    path = o.build(mutant=mutant)
    o.use_library(path)
    try:
        caught = None
        for pin in pins(o):
            try:
                pin()
            except Exception as e:  # an assertion, an oracle error code, a numpy error
                caught = e
                break
        assert caught is not None, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
    finally:
        o.use_library(None)


def test_unmutated_oracle_passes_the_same_pins(oracle_mod):
    for pin in pins(oracle_mod):
        pin()
