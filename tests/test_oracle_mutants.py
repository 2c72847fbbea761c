"""Each planted oracle mistake is caught by at least one pin.

The mutants are the tinyllm page's pitfall list where it applies to a two-pass
oracle (s03 logical block index as block id, s04 KV-head offset dropped, s05
round-robin GQA, s06 a window of w + 1, s07 query at n instead of n - 1, s08 V
read from the K pool, s13 empty context accepted, s14 max_blocks trusted, s15
block ids trusted) and further plausible slips in the scatter, gather, score,
split-KV reduction and merge arithmetic, and in the attention-sink term (s60 the sink
left out of the exp-sum, s61 its term taken as 1 instead of e^(sink - m)) and the fp8 pools
(s70 a wrong exponent bias, s71 truncation instead of rounding, s72 / s73 a dequantisation
scale ignored), the per kv head scales (s74 the query head's index taken for the kv
head's, s75 the first head's scale used for every head) and the per-block scales (s76 the
block's factor of kv head 0 used for every head).
"""
import pytest

import oracle
from tests import oracle_pins as P

KILLERS = {
    3: ["hand_example", "brute_force", "block_permutation"],
    4: ["brute_force"],
    5: ["brute_force"],
    6: ["brute_force"],
    7: ["hand_example", "brute_force"],
    8: ["hand_example", "closed_forms"],
    13: ["validation"],
    14: ["validation"],
    15: ["validation"],
    20: ["hand_example_via_cache", "scatter_gather_roundtrip"],
    21: ["hand_example_via_cache", "scatter_gather_roundtrip"],
    22: ["scatter_gather_roundtrip"],
    30: ["brute_force"],
    31: ["brute_force"],
    32: ["hand_example", "closed_forms"],
    40: ["splitkv_masked_partition"],
    41: ["splitkv_all_masked"],
    42: ["splitkv_matches_full"],
    50: ["merge_edge_cases"],
    51: ["merge_edge_cases"],
    52: ["merge_identity"],
    60: ["sinks_closed_forms", "sinks_brute_force"],
    61: ["sinks_closed_forms", "sinks_brute_force"],
    70: ["fp8_codec", "fp8_attention_brute_force"],
    71: ["fp8_codec", "fp8_scatter"],
    72: ["fp8_attention_brute_force", "dequant_scales", "splitkv_fp8_scaled"],
    73: ["fp8_attention_brute_force", "dequant_scales", "splitkv_fp8_scaled"],
    74: ["per_head_attention"],
    75: ["per_head_scatter", "per_head_attention"],
    76: ["per_block_attention"],
}


@pytest.mark.parametrize("mutant", sorted(KILLERS))
def test_mutant_is_killed(mutant):
    oracle.set_mutant(mutant)
    try:
        caught = []
        for name in KILLERS[mutant]:
            try:
                P.ALL_PINS[name]()
            except AssertionError:
                caught.append(name)
        assert caught, f"mutant {mutant} survived {KILLERS[mutant]}"
    finally:
        oracle.set_mutant(0)
