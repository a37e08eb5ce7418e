"""Host-side schedule of the verify pass (no GPU): where the layer chain joins the paging stream."""
import pytest

from speculative_decode_verify_attn_gb300.passes import is_full_layer, join_points


@pytest.mark.parametrize("n_full", [1, 2, 3, 4, 5, 9, 10, 16, 33])
def test_every_full_layer_waits_for_its_own_page_in(n_full):
    joins = join_points(n_full)
    covered = -1
    for j in range(n_full):
        if j in joins:
            assert joins[j] >= covered          # page-ins complete in order: waits only move forward
            covered = joins[j]
        assert covered >= j, f"full layer {j} could start before its page-in"
    assert covered == n_full - 1


def test_joins_are_few():
    # ten full layers (the 40-layer 3-in-4 pattern) join four times, not ten
    assert join_points(10) == {0: 0, 1: 2, 3: 6, 7: 9}
    assert len(join_points(64)) == 7


def test_three_in_four_pattern():
    full = [l for l in range(40) if is_full_layer(l)]
    assert full == list(range(3, 40, 4))
