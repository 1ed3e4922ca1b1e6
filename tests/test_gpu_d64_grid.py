"""GPU parity of the head_dim-64 backward on grids of more CTAs than the GPU
has SMs (one CTA per (sequence, key/value head, key block)).  Between them
the cases put in one launch: key blocks past a short sequence's end (CTAs
that exit at once), empty sequences, key blocks no query sees (CTAs with
no sweep, whose dK / dV rows are written as zeros), ragged tails of both
query and key blocks, NaN padding rows, grouped-query heads, and each mask.
Every element is compared with the fp64 oracle."""
import pytest
import torch

import seeded_inputs as si
from parity import Prepared, check_case

pytestmark = pytest.mark.gpu


def n_ctas(case):
    return -(-max(case.kv_lens) // 128) * case.kv_heads * case.batch


CASES = [
    si.Case("grid_d64_varlen_causal_nan", 16, 64, [700, 1, 0, 1300, 513], [700, 1, 0, 1300, 513], True, 81,
            pad_q=11, pad_kv=7),
    si.Case("grid_d64_bottom_right_keys_unseen", 12, 64, [200, 77], [1500, 1300], True, 82, bottom_right=True),
    si.fixed("grid_d64_window", 2, 8, 64, 1500, 1500, True, 83, window=300),
    si.fixed("grid_d64_gqa_16_4", 4, 16, 64, 1200, 1200, False, 84, heads_kv=4),
    si.Case("grid_d64_cross_ragged", 16, 64, [513, 129, 1000], [2000, 700, 1111], False, 85, pad_kv=3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_d64_grid_parity(case):
    assert n_ctas(case) > 152
    check_case(Prepared(case))


def test_d64_grid_deterministic_repeats_bitwise():
    """Deterministic mode on the same grid: oracle parity, bitwise repeats,
    and dK / dV bits equal to the atomic mode's (the same per-block products
    in the same order)."""
    import attention_backward_sm_gb300 as fab
    case = CASES[0]
    prep = Prepared(case)
    first = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    check_case(prep, out=first)
    again = prep.run(dq_mode=fab.FA_DQ_DETERMINISTIC)
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    anyorder = prep.run(dq_mode=fab.FA_DQ_ATOMIC)
    assert torch.equal(first[1], anyorder[1]) and torch.equal(first[2], anyorder[2])
