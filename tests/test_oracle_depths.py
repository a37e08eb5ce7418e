"""Pins of the oracle's confidence-gated depth policy: brute force over every depth vector on
small cases, the closed form of the expected committed tokens, and special cases."""
import itertools

import numpy as np
import pytest

from oracle import vfy_oracle as O


def test_expected_committed_closed_form():
    for c in (0.0, 0.3, 0.56, 0.9, 1.0):
        for d in range(0, 12):
            want = d + 1 if c == 1.0 else (1 - c ** (d + 1)) / (1 - c)
            assert abs(O.expected_committed(c, d) - want) < 1e-12


@pytest.mark.parametrize("seed", range(12))
def test_gate_depths_is_the_brute_force_optimum(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 5))
    conf = rng.uniform(0, 1, n).round(3).tolist()
    max_depth = int(rng.integers(0, 5))
    budget = int(rng.integers(n, n * (max_depth + 1) + 3))
    got = O.gate_depths(conf, budget, max_depth)
    assert all(0 <= d <= max_depth for d in got) and sum(got) + n <= max(budget, n)
    best = max(sum(O.expected_committed(c, d) for c, d in zip(conf, ds))
               for ds in itertools.product(range(max_depth + 1), repeat=n) if sum(ds) + n <= budget)
    assert abs(sum(O.expected_committed(c, d) for c, d in zip(conf, got)) - best) < 1e-12


def test_gate_depths_special_cases():
    assert O.gate_depths([0.5, 0.5, 0.5], 3, 16) == [0, 0, 0]            # budget = one row each
    assert O.gate_depths([0.9, 0.1], 6, 3) == [3, 1]                     # the confident one saturates
    assert O.gate_depths([0.5, 0.5], 5, 16) == [2, 1]                    # ties go to the lower index
    assert O.gate_depths([0.7, 0.7, 0.7], 30, 4) == [4, 4, 4]            # budget beyond every max
    assert O.gate_depths([], 4, 2) == []


@pytest.mark.parametrize("seed", range(20))
def test_library_gate_depths_matches_the_oracle(seed):
    """vfy_gate_depths (host code of libvfy.so, no device needed) gives the oracle's depths."""
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import vfy
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 12))
    conf = rng.uniform(0, 1, n).astype(np.float32)
    if n > 2:
        conf[1] = conf[0]                                  # a tie
    max_depth = int(rng.integers(0, 17))
    budget = int(rng.integers(0, n * 18 + 2))
    assert vfy.vfy_gate_depths(conf, budget, max_depth) == O.gate_depths([float(c) for c in conf], budget, max_depth)


def test_library_gate_depths_rejects_bad_confidence():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import vfy
    for bad in ([0.5, float("nan")], [1.5], [-0.1]):
        with pytest.raises(vfy.VfyError):
            vfy.vfy_gate_depths(bad, 10, 4)
