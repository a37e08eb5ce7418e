"""Pins of the oracle's residency selection, page-in and greedy acceptance.

Residency ('Laguna XS 2.1 33B on a RTX 3090' (lucebox), 'Three optimizations', item 1):
  * hand-worked cases (tests/golden/select_cases.json);
  * numpy.argsort(-scores, kind='stable') on NaN-free inputs;
  * brute force on n <= 8: the chosen set is the unique k-subset every member of which beats
    every non-member (higher score, or equal score and lower index; NaN loses to all numbers);
  * slot invariants over random multi-step histories.
Acceptance ('The model, fast MoE with a drafter in the box'; 'The Death of the Compute-Moat',
'DFlash Drafters and the End of Speculative Loss'):
  * hand-worked cases (tests/golden/accept_cases.json);
  * torch.argmax on CPU as the library routine for ties, signed zeros, infinities and NaN;
  * planted prefixes: drafts equal to the greedy tokens for exactly n positions.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32(values):
    return np.array([float(v) for v in values], dtype=np.float32)


# ---------------------------------------------------------------------------------------------
# Residency
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", load("select_cases.json")["cases"], ids=lambda c: c["name"])
def test_select_golden(case):
    ids, slots, pagein, new_slot = O.select_resident_one(
        f32(case["scores"]), case["k"], case["prev_slot"], case["slot_base"])
    assert ids == case["ids"]
    assert slots == case["slots"]
    assert [list(p) for p in pagein] == case["pagein"]
    assert new_slot.tolist() == case["new_slot"]


def beats(scores, a, b):
    sa, sb = float(scores[a]), float(scores[b])
    if math.isnan(sa) or math.isnan(sb):
        if math.isnan(sa) and math.isnan(sb):
            return a < b
        return math.isnan(sb)
    return sa > sb or (sa == sb and a < b)


def brute_force_topk(scores, k):
    n = len(scores)
    k = min(k, n)
    found = []
    for subset in itertools.combinations(range(n), k):
        rest = [j for j in range(n) if j not in subset]
        if all(beats(scores, a, b) for a in subset for b in rest):
            found.append(list(subset))
    assert len(found) == 1
    return found[0]


def test_select_brute_force_small():
    rng = np.random.default_rng(0)
    pool = np.array([-np.inf, -1.0, -0.0, 0.0, 0.5, 0.5, 2.0, np.inf, np.nan], dtype=np.float32)
    for trial in range(300):
        n = int(rng.integers(1, 9))
        scores = rng.choice(pool, n)
        k = int(rng.integers(1, n + 2))
        ids, _, _, _ = O.select_resident_one(scores, k, [-1] * n, 0)
        assert ids == brute_force_topk(scores, k), (scores, k)


def test_select_matches_stable_argsort():
    rng = np.random.default_rng(1)
    for trial in range(20):
        n = int(rng.integers(50, 600))
        scores = np.round(rng.standard_normal(n) * 3).astype(np.float32)   # many ties
        k = int(rng.integers(1, n))
        ids, _, _, _ = O.select_resident_one(scores, k, [-1] * n, 0)
        ref = np.sort(np.argsort(-scores, kind="stable")[:k])
        assert ids == ref.tolist()


def test_select_multi_step_invariants():
    """Over a random history: kept chunks keep their slot, slots stay distinct and in range,
    the page-in list is exactly the newly chosen chunks, evicted chunks get -1."""
    rng = np.random.default_rng(2)
    cu = [0, 300, 310, 700]
    k = 64
    slot_map = np.full(cu[-1], -1)
    for step in range(12):
        scores = synth.gumbel_scores(rng, cu[-1])
        res = O.select_resident(scores, cu, k, slot_map)
        for b in range(3):
            c0, c1 = cu[b], cu[b + 1]
            r0, r1 = res["cu_resident"][b], res["cu_resident"][b + 1]
            ids = res["resident_ids"][r0:r1]
            slots = res["resident_slots"][r0:r1]
            assert r1 - r0 == min(k, c1 - c0)
            assert list(ids) == sorted(ids)
            assert len(set(slots.tolist())) == len(slots)
            assert all(b * k <= s < (b + 1) * k for s in slots)
            paged = {c for c, s in res["pagein"][b]}
            for c, s in zip(ids, slots):
                if slot_map[c0 + c] >= 0:
                    assert s == slot_map[c0 + c] and (c0 + c) not in paged
                else:
                    assert (c0 + c) in paged
            new = res["slot_of_chunk"][c0:c1]
            assert (new >= 0).sum() == len(ids)
            assert all(new[c] == s for c, s in zip(ids, slots))
        slot_map = res["slot_of_chunk"]


def test_rotating_residency_plants_its_winners():
    """The planted score schedule makes exactly `rotate` new chunks enter at each step."""
    rng = np.random.default_rng(3)
    rot = synth.rotating_residency(rng, 4096, 128, 16, 262144, 17)
    slot_map = np.full(4096, -1)
    for step in range(4):
        res = O.select_resident(rot.scores(step), [0, 4096], 128, slot_map)
        assert np.array_equal(res["resident_ids"], rot.winners(step))
        if step > 0:
            assert len(res["pagein"][0]) == 16
        slot_map = res["slot_of_chunk"]


SELECT_MUTATIONS = {
    "ties to the higher index": lambda scores: sorted(
        range(len(scores)), key=lambda j: (math.isnan(float(scores[j])),
                                           -float(scores[j]) if not math.isnan(float(scores[j])) else 0, -j)),
    "NaN ranks first": lambda scores: sorted(
        range(len(scores)), key=lambda j: (not math.isnan(float(scores[j])),
                                           -float(scores[j]) if not math.isnan(float(scores[j])) else 0, j)),
    "ascending scores": lambda scores: sorted(
        range(len(scores)), key=lambda j: (math.isnan(float(scores[j])),
                                           float(scores[j]) if not math.isnan(float(scores[j])) else 0, j)),
}


@pytest.mark.parametrize("name", sorted(SELECT_MUTATIONS))
def test_select_planted_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(O, "rank_chunks", SELECT_MUTATIONS[name])
    caught = False
    for case in load("select_cases.json")["cases"]:
        ids, *_ = O.select_resident_one(f32(case["scores"]), case["k"], case["prev_slot"],
                                         case["slot_base"])
        caught |= ids != case["ids"]
    assert caught


def test_page_in_is_bit_exact():
    rng = np.random.default_rng(4)
    hk = rng.integers(0, 65536, (20, 2, 64, 8), dtype=np.uint16)
    hv = rng.integers(0, 65536, (20, 2, 64, 8), dtype=np.uint16)
    pk = np.zeros((6, 2, 64, 8), np.uint16)
    pv = np.zeros((6, 2, 64, 8), np.uint16)
    pairs = [(3, 5), (19, 0), (7, 2)]
    nk, nv = O.page_in(hk, hv, pk, pv, pairs)
    for c, s in pairs:
        assert nk[s].tobytes() == hk[c].tobytes() and nv[s].tobytes() == hv[c].tobytes()
    untouched = [s for s in range(6) if s not in (5, 0, 2)]
    assert not nk[untouched].any() and not nv[untouched].any()


# ---------------------------------------------------------------------------------------------
# Acceptance
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", load("accept_cases.json")["cases"], ids=lambda c: c["name"])
def test_accept_golden(case):
    logits = np.array([[float(v) for v in row] for row in case["logits"]], dtype=np.float32)
    assert [O.argmax_row(r) for r in logits] == case["argmax"]
    n, bonus, committed = O.accept_seq(logits, case["drafts"])
    assert (n, bonus, committed) == (case["n"], case["bonus"], case["committed"])


def test_argmax_matches_torch_argmax():
    """torch.argmax on CPU: ties to the first index, NaN is the maximum (first NaN)."""
    rng = np.random.default_rng(5)
    specials = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 1.0, 1.0], dtype=np.float32)
    for trial in range(400):
        n = int(rng.integers(1, 40))
        row = np.round(rng.standard_normal(n)).astype(np.float32)
        m = int(rng.integers(0, 4))
        row[rng.integers(0, n, m)] = rng.choice(specials, m)
        assert O.argmax_row(row) == int(torch.argmax(torch.from_numpy(row))), row


def test_accept_planted_prefix_lengths():
    """Drafts equal to the greedy tokens for exactly n positions give accepted length n."""
    rng = np.random.default_rng(6)
    vocab = 1024
    logits = synth.normal_logits(rng, 17, vocab)
    a = [O.argmax_row(r) for r in logits]
    for n_match in range(0, 17):
        drafts = synth.drafts_prefix(rng, a, n_match, vocab)
        n, bonus, committed = O.accept_seq(logits, drafts)
        assert n == n_match and bonus == a[n_match]
        assert committed[:n_match] == a[:n_match] and committed[n_match] == a[n_match]
        assert committed[n_match + 1:] == [-1] * (16 - n_match)


def test_accept_ragged_batch():
    rng = np.random.default_rng(7)
    vocab = 300
    depths = [2, 16, 0, 11, 4]
    cu = np.concatenate([[0], np.cumsum([d + 1 for d in depths])])
    targets = rng.integers(0, vocab, cu[-1])
    logits = synth.planted_logits(rng, targets, vocab)
    want = [min(d, int(rng.integers(0, d + 1))) for d in depths]
    drafts = np.concatenate([synth.drafts_prefix(rng, targets[cu[b]:cu[b + 1]], want[b], vocab)
                             for b in range(len(depths))]).astype(np.int32)
    ns, bonus, committed = O.accept(logits, drafts, cu)
    assert ns.tolist() == want
    assert bonus.tolist() == [int(targets[cu[b] + want[b]]) for b in range(len(depths))]
    assert len(committed) == cu[-1]


def test_planted_logits_argmax_is_target():
    rng = np.random.default_rng(8)
    targets = rng.integers(0, 5000, 17)
    logits = synth.planted_logits(rng, targets, 5000)
    assert [O.argmax_row(r) for r in logits] == targets.tolist()


def test_accept_planted_mistake_is_caught(monkeypatch):
    """Comparing draft r with the greedy token of row r+1 (an off-by-one) fails the golden cases."""
    def shifted(logits, drafts):
        a = [O.argmax_row(r) for r in logits]
        n = 0
        while n < len(drafts) and a[n + 1] == int(drafts[n]):
            n += 1
        return n, a[n], [int(x) for x in drafts[:n]] + [a[n]] + [-1] * (len(drafts) - n)
    monkeypatch.setattr(O, "accept_seq", shifted)
    bad = 0
    for case in load("accept_cases.json")["cases"]:
        logits = np.array([[float(v) for v in row] for row in case["logits"]], dtype=np.float32)
        bad += O.accept_seq(logits, case["drafts"]) != (case["n"], case["bonus"], case["committed"])
    assert bad > 0
