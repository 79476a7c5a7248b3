"""Mutation check of the oracle's pins: a copy of the oracle's C source with one
planted, plausible mistake (a wrong ape row, swapped kv halves, a missing
first-group mask, buffer_len off by one, a short write set, a decode slot off
by one, a ragged id without its request offset, a wrong read page, a dropped
term, a sign error, an input row off by one; in the SWA-paged planner: no
page-end writes, the ring offset taken modulo the page size, records without
state reads translated; in norm + RoPE: a rotation sign, the position, the
rotated channels; in the online state: no reset at a group start, the sum not
rescaled, an ape row off by one; and bf16 rounding by truncation, a decode
page of the previous group, a write set a group too long, a decode that pools
before it writes the new token, RMSNorm's eps outside the root, RoPE's cos and
sin swapped, padding with zero bytes, token-layout rows in plan order) is
compiled on its own and must fail at least one pin.  The mistakes are textual patches of the source (the first n
occurrences of a fragment replaced), so the oracle itself carries no hooks."""
import pytest

from tests import test_oracle_norm_rope as N
from tests import test_oracle_online as L
from tests import test_oracle_paged as Q
from tests import test_oracle_pins as P

# mutant -> (what it plants, [(fragment of the oracle source, its replacement, occurrences replaced)])
MUTANTS = {
    1: ('ape row off by one', [
        ('int arow = i;',
         'int arow = (i + 1) % W;', 1),
    ]),
    2: ('C4 overlap entries read the main kv half', [
        ('int kv_col = (ratio == 4) ? (i < 4 ? 0 : hd) + c : c;',
         'int kv_col = (ratio == 4) ? (i < 4 ? hd : hd) + c : c;', 1),
    ]),
    3: ('first-group mask missing', [
        ('if (ratio == 4 && seq_len == 4 && i < 4) { /* first group: no previous group */',
         'if (0) {', 1),
        ('if (ratio == 4 && P->seq_len == 4 && i < 4) {',
         'if (0) {', 1),
    ]),
    4: ('buffer_len off by one', [
        ('const int64_t bl = W - (j + 1 < W ? j + 1 : W);',
         'const int64_t bl = W - (j + 1 < W ? j + 1 : W) - (j + 1 < W ? 1 : 0);', 1),
    ]),
    5: ('C4 write set without the overlap group', [
        ('const int64_t first_w = (sl / ratio) * ratio - overlap;',
         'const int64_t first_w = (sl / ratio) * ratio - 0;', 1),
    ]),
    6: ('decode write slot off by one', [
        ('int64_t loc = legacy_loc(ratio, rid[b], p1);',
         'int64_t loc = legacy_loc(ratio, rid[b], p1 + 1);', 1),
    ]),
    7: ('ragged id without the request offset', [
        ('const uint64_t ragged = token_base + (uint64_t)j;',
         'const uint64_t ragged = 0 + (uint64_t)j;', 1),
    ]),
    8: ('read_page_0 of the current group', [
        ('const int64_t p0 = p - ratio > 0 ? p - ratio : 0;',
         'const int64_t p0 = p;', 1),
    ]),
    9: ('a dropped denominator term', [
        ('den += w;',
         'if (i != W - 1) den += w;', 1),
    ]),
    10: ('sign error in the exponent', [
        ('double w = exp((double)s[i] - (double)m);',
         'double w = exp((double)m - (double)s[i]);', 1),
    ]),
    11: ('input row off by one', [
        ('int64_t irow = ragged - (W - 1) + i;',
         'int64_t irow = ragged - (W - 1) + i - 1;', 1),
    ]),
    12: ('paged C4 write set without the SWA page ends', [
        ('if (p >= first_w || (ratio == 4 && p % sps >= sps - ratio)) {',
         'if (p >= first_w) {', 1),
    ]),
    13: ('paged ring offset modulo the SWA page size', [
        ('return (swa / sps) * ring + swa % ring;',
         'return (swa / sps) * ring + swa % sps;', 1),
    ]),
    14: ('paged records without state reads translated', [
        ('if (bl > 0) {',
         'if (1) {', 1),
    ]),
    15: ('RoPE rotation sign', [
        ('y[base + 2 * i] = a * cs - b * sn;',
         'y[base + 2 * i] = a * cs + b * sn;', 1),
    ]),
    16: ('RoPE position seq_len instead of seq_len - ratio', [
        ('pos = (int64_t)P->seq_len - ratio;',
         'pos = (int64_t)P->seq_len - 0;', 2),
    ]),
    17: ('RoPE on the first rope_dim channels', [
        ('const int base = hd - rope_dim;',
         'const int base = 0;', 1),
    ]),
    18: ('online state not reset at a group start', [
        ('if (first) {',
         'if (0) {', 1),
    ]),
    19: ('online sum not rescaled on a new maximum', [
        ('*l = *l * c + e;',
         '*l = *l + e;', 1),
    ]),
    20: ('online ape row off by one', [
        ('const float bias = load_elem(ape, (size_t)(p % 128) * hd + c, in_dtype);',
         'const float bias = load_elem(ape, (size_t)((p + 1) % 128) * hd + c, in_dtype);', 1),
    ]),
    21: ('bf16 rounding by truncation', [
        ('double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);', 'double r = ldexp(floor(ldexp(a, -qexp)), qexp);', 1),
    ]),
    22: ('decode read_page_1 of the previous group', [
        ('plan[b].read_page_1 = (int32_t)legacy_page(ratio, rid[b], p1);',
         'plan[b].read_page_1 = (int32_t)legacy_page(ratio, rid[b], p0);', 1),
    ]),
    23: ('prefill write set a group too long', [
        ('const int64_t first_w = (sl / ratio) * ratio - overlap;',
         'const int64_t first_w = (sl / ratio - 1) * ratio - overlap;', 1),
    ]),
    24: ('decode pools before writing the new token', [
        ('    memcpy((char*)state + (size_t)P->write_loc * row_bytes, row_ptr(input, b, width, in_dtype), row_bytes);\n'
         '    if (P->seq_len % (uint32_t)ratio != 0) continue;',
         '    if (P->seq_len % (uint32_t)ratio != 0) {\n'
         '      memcpy((char*)state + (size_t)P->write_loc * row_bytes, row_ptr(input, b, width, in_dtype), row_bytes);\n'
         '      continue;\n'
         '    }', 1),
        ('    pool_window(ratio, hd, in_dtype, out_dtype, (const void* const*)entries, ape,\n'
         '                (char*)out + (size_t)b * (size_t)hd * elem_size(out_dtype));\n  }\n  free(entries);\n  return ORC_OK;',
         '    pool_window(ratio, hd, in_dtype, out_dtype, (const void* const*)entries, ape,\n'
         '                (char*)out + (size_t)b * (size_t)hd * elem_size(out_dtype));\n'
         '    memcpy((char*)state + (size_t)P->write_loc * row_bytes, row_ptr(input, b, width, in_dtype), row_bytes);\n'
         '  }\n  free(entries);\n  return ORC_OK;', 1),
    ]),
    25: ('RMSNorm eps outside the root', [
        ('const double r = 1.0 / sqrt(ss / hd + (double)eps);', 'const double r = 1.0 / (sqrt(ss / hd) + (double)eps);', 1),
    ]),
    27: ('padding with zero bytes instead of the invalid record', [
        ('if (cap_c > nc) memset(pc + nc, 0xFF, sizeof(orc_plan_c) * (cap_c - nc));',
         'if (cap_c > nc) memset(pc + nc, 0x00, sizeof(orc_plan_c) * (cap_c - nc));', 1),
    ]),
    28: ('token layout rows in plan order', [
        ('size_t orow = out_layout == ORC_OUT_TOKEN ? (size_t)ragged : (size_t)e;', 'size_t orow = (size_t)e;', 1),
    ]),
    26: ('RoPE cos and sin swapped', [
        ('const double cs = freqs[((size_t)pos * (rope_dim / 2) + i) * 2];',
         'const double cs = freqs[((size_t)pos * (rope_dim / 2) + i) * 2 + 1];', 1),
        ('const double sn = freqs[((size_t)pos * (rope_dim / 2) + i) * 2 + 1];',
         'const double sn = freqs[((size_t)pos * (rope_dim / 2) + i) * 2];', 1),
    ]),
}


def pins(o):
    yield lambda: P.test_plan_worked_examples(o)
    yield lambda: P.test_bf16_round_once(o)
    yield lambda: P.test_plan_padding_capacity_and_validation(o)
    yield lambda: P.test_prefill_token_layout_zero_rows_and_compact_order(o)
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
    yield lambda: N.test_eps_sits_inside_the_root(o)
    yield lambda: N.test_matches_float64_torch(o, 1)
    yield lambda: N.test_rotation_keeps_pair_lengths_and_relative_positions(o)
    yield lambda: N.test_position_is_seq_len_minus_ratio(o)
    yield lambda: L.test_online_plan_worked_example(o)
    yield lambda: L.test_online_closed_forms(o)
    yield lambda: L.test_online_schedules_equal_window_definition(o, 0)


def mutated_source(o, mutant):
    text = o.source()
    for fragment, replacement, n in MUTANTS[mutant][1]:
        assert text.count(fragment) >= n, f"mutant {mutant}: {fragment!r} not in the oracle source"
        text = text.replace(fragment, replacement, n)
    return text


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(oracle_mod, mutant):
    o = oracle_mod
    path = o.build_variant(mutated_source(o, mutant), f"mutant{mutant}")
    o.use_library(path)
    try:
        caught = None
        for pin in pins(o):
            try:
                pin()
            except Exception as e:  # an assertion, an oracle error code, a numpy error
                caught = e
                break
        assert caught is not None, f"mutant {mutant} ({MUTANTS[mutant][0]}) passed every pin"
    finally:
        o.use_library(None)


def test_unmutated_oracle_passes_the_same_pins(oracle_mod):
    for pin in pins(oracle_mod):
        pin()
