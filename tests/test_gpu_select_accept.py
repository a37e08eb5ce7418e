"""GPU parity of vfy_select_resident, vfy_page_in and vfy_accept against the oracle, bit-exact.

Residency and page-in: 'Laguna XS 2.1 33B on a RTX 3090' (lucebox), 'Three optimizations',
item 1. Acceptance: same page, 'The model, fast MoE with a drafter in the box', and 'The Death of
the Compute-Moat', 'DFlash Drafters and the End of Speculative Loss'.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def H():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import harness
    return harness


@pytest.fixture(scope="module")
def vfy():
    from speculative_decode_verify_attn_gb300 import vfy
    return vfy


@pytest.fixture(scope="module")
def ctx(vfy, H):
    c = vfy.vfy_create(16, 4, 128, max_seqs=8, max_queries_per_seq=17, device=0)
    yield c
    c.close()


def check_select(H, vfy, ctx, scores, cu, k, prev):
    got = H.select_resident(ctx, scores, cu, k, prev)
    ref = O.select_resident(scores, cu, k, prev)
    assert np.array_equal(got["resident_ids"], ref["resident_ids"])
    assert np.array_equal(got["resident_slots"], ref["resident_slots"])
    assert np.array_equal(got["cu_resident"], ref["cu_resident"])
    assert np.array_equal(got["slot_of_chunk"], ref["slot_of_chunk"])
    for b in range(len(cu) - 1):
        cnt = int(got["pagein_count"][b])
        pairs = got["pagein_list"][b * k: b * k + cnt].tolist()
        assert pairs == [list(p) for p in ref["pagein"][b]]
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    return ref["slot_of_chunk"]


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "select_cases.json")))["cases"],
                         ids=lambda c: c["name"])
def test_select_golden(H, vfy, ctx, case):
    scores = np.array([float(v) for v in case["scores"]], np.float32)
    n = len(scores)
    k = case["k"]
    # the golden slot_base is b * k: place the case at sequence b = slot_base / k
    b = case["slot_base"] // k
    cu = [0] * (b + 1) + [n]
    prev = np.array(case["prev_slot"], np.int32)
    got = H.select_resident(ctx, scores, cu, k, prev)
    assert got["resident_ids"].tolist() == case["ids"]
    assert got["resident_slots"].tolist() == case["slots"]
    assert got["slot_of_chunk"].tolist() == case["new_slot"]
    cnt = int(got["pagein_count"][b])
    assert got["pagein_list"][b * k: b * k + cnt].tolist() == case["pagein"]


@pytest.mark.parametrize("n,k", [(512, 128), (4096, 128), (4096, 4096), (32768, 128), (100, 7), (1, 1)])
def test_select_random_ties_and_specials(H, vfy, ctx, n, k):
    rng = np.random.default_rng(n + k)
    scores = np.round(rng.standard_normal(n) * 4).astype(np.float32)          # many ties
    m = max(1, n // 50)
    scores[rng.integers(0, n, m)] = rng.choice(np.array([np.nan, np.inf, -np.inf, -0.0, 0.0], np.float32), m)
    prev = np.full(n, -1, np.int32)
    held = rng.permutation(n)[: min(k, n) // 2]
    prev[held] = rng.permutation(k)[: len(held)]
    check_select(H, vfy, ctx, scores, [0, n], k, prev)


def test_select_multi_sequence_history(H, vfy, ctx):
    """Several steps, three sequences, the slot map carried from step to step on the device."""
    rng = np.random.default_rng(3)
    cu = [0, 300, 310, 3000]
    k = 64
    prev = np.full(cu[-1], -1, np.int32)
    for step in range(6):
        scores = synth.gumbel_scores(rng, cu[-1])
        prev = check_select(H, vfy, ctx, scores, cu, k, prev).astype(np.int32)


def test_select_rotating_schedule_pages_16(H, vfy, ctx):
    """The 256K schedule: 4096 chunks, top-128, exactly 16 newcomers per step."""
    rng = np.random.default_rng(4)
    rot = synth.rotating_residency(rng, 4096, 128, 16, 262144, 17)
    prev = np.full(4096, -1, np.int32)
    for step in range(4):
        got = H.select_resident(ctx, rot.scores(step), [0, 4096], 128, prev)
        assert np.array_equal(got["resident_ids"], rot.winners(step))
        if step:
            assert int(got["pagein_count"][0]) == 16
        prev = check_select(H, vfy, ctx, rot.scores(step), [0, 4096], 128, prev).astype(np.int32)


@pytest.mark.parametrize("ctas", [0, 1, 3, 4])
def test_page_in_bit_exact(H, vfy, ctx, ctas):
    """Every CTAs-per-chunk setting (0 = the default 2) copies the chosen chunks bit-exactly and
    touches no other slot."""
    rng = np.random.default_rng(5)
    n_host, n_slots, k = 40, 12, 12
    hk = rng.integers(0, 65536, (n_host, 4, 64, 128), dtype=np.uint16)
    hv = rng.integers(0, 65536, (n_host, 4, 64, 128), dtype=np.uint16)
    host_k = H.host_bf16(hk)
    host_v = H.host_bf16(hv)
    pk = torch.zeros((n_slots, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    pv = torch.zeros_like(pk)
    pairs = [(3, 5), (39, 0), (7, 11), (0, 2)]
    plist = np.full((k, 2), -1, np.int32)
    plist[: len(pairs)] = pairs
    vfy.vfy_set_pagein_ctas(ctx, ctas)
    try:
        vfy.vfy_page_in(ctx, host_k, host_v, n_host, pk, pv, n_slots, H.dev_i32(plist), H.dev_i32([len(pairs)]),
                        1, k)
    finally:
        vfy.vfy_set_pagein_ctas(ctx, 0)
    torch.cuda.synchronize()
    gk, gv = H.bits_of(pk), H.bits_of(pv)
    nk, nv = O.page_in(hk, hv, np.zeros_like(gk), np.zeros_like(gv), pairs)
    assert gk.tobytes() == nk.tobytes() and gv.tobytes() == nv.tobytes()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


def test_page_in_ctas_bounds(vfy, ctx):
    for bad in (-1, 5):
        with pytest.raises(vfy.VfyError) as e:
            vfy.vfy_set_pagein_ctas(ctx, bad)
        assert e.value.status == vfy.VFY_EINVAL


def test_page_in_rejects_pageable_memory(H, vfy, ctx):
    hk = torch.zeros((2, 4, 64, 128), dtype=torch.bfloat16)           # not pinned
    pk = torch.zeros((2, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vfy.VfyError) as e:
        vfy.vfy_page_in(ctx, hk, hk, 2, pk, pk, 2, H.dev_i32(np.zeros((1, 2))), H.dev_i32([0]), 1, 1)
    assert e.value.status == vfy.VFY_EINVAL


# ---------------------------------------------------------------------------------------------
# Acceptance
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "accept_cases.json")))["cases"],
                         ids=lambda c: c["name"])
def test_accept_golden(H, vfy, ctx, case):
    logits = np.array([[float(v) for v in row] for row in case["logits"]], np.float32)
    n, bonus, committed = H.accept(ctx, logits, np.array(case["drafts"], np.int32), [0, len(logits)])
    assert (int(n[0]), int(bonus[0]), committed.tolist()) == (case["n"], case["bonus"], case["committed"])


def test_accept_tiny_config(H, vfy, ctx):
    """17 x 1024 logits ~ N(0,1); drafts = the greedy tokens for 7 positions, then random: n = 7."""
    rng = np.random.default_rng(0)
    logits = synth.normal_logits(rng, 17, 1024)
    a = [O.argmax_row(r) for r in logits]
    drafts = synth.drafts_prefix(rng, a, 7, 1024)
    n, bonus, committed = H.accept(ctx, logits, drafts, [0, 17])
    rn, rb, rc = O.accept(logits, drafts, [0, 17])
    assert n.tolist() == rn.tolist() == [7]
    assert bonus.tolist() == rb.tolist() and committed.tolist() == rc.tolist()


@pytest.mark.parametrize("n_match", [0, 1, 8, 15, 16])
def test_accept_full_vocab(H, vfy, ctx, n_match):
    """17 x 131072 fp32 logits, the vocabulary of the 256K workload."""
    rng = np.random.default_rng(n_match)
    logits = synth.normal_logits(rng, 17, synth.VOCAB)
    a = [O.argmax_row(r) for r in logits]
    drafts = synth.drafts_prefix(rng, a, n_match, synth.VOCAB)
    n, bonus, committed = H.accept(ctx, logits, drafts, [0, 17])
    rn, rb, rc = O.accept(logits, drafts, [0, 17])
    assert n.tolist() == rn.tolist() == [n_match]
    assert bonus.tolist() == rb.tolist() and committed.tolist() == rc.tolist()


def test_accept_ties_nan_and_odd_vocab(H, vfy, ctx):
    """Ties, signed zeros, infinities and NaN across CTA boundaries, vocab not a multiple of 4."""
    rng = np.random.default_rng(7)
    V = 100003
    logits = np.round(rng.standard_normal((6, V)) * 2).astype(np.float32)
    logits[0, [5, 70000]] = 50.0                       # tie in different CTAs -> 5
    logits[1, [99999, 100002]] = np.inf                # -> 99999
    logits[2, [12345, 80000]] = np.nan                 # first NaN -> 12345
    logits[3] = -0.0
    logits[3, 77] = 0.0                                # all zero: -> 0
    logits[4] = -np.inf                                # -> 0
    drafts = np.array([5, 99999, 12345, 0, 0], np.int32)
    n, bonus, committed = H.accept(ctx, logits, drafts, [0, 6])
    rn, rb, rc = O.accept(logits, drafts, [0, 6])
    assert n.tolist() == rn.tolist() and bonus.tolist() == rb.tolist()
    assert committed.tolist() == rc.tolist()
    torch_a = torch.argmax(torch.from_numpy(logits), dim=1).tolist()
    assert [O.argmax_row(r) for r in logits] == torch_a


def test_accept_ties_nan_vectorised_path(H, vfy, ctx):
    """Vocabulary a multiple of 4 (16-byte loads): ties inside one 16-byte word, inside one thread's
    round of loads and across CTAs, signed zeros, infinities, NaN and a maximum in the last entry."""
    V = 131072
    rows = 10
    logits = np.full((rows, V), -1.0, np.float32)
    logits[0, [9, 10]] = 50.0                          # one 16-byte word -> 9
    logits[1, [1 + 4 * 256 * 3, 1, 70001]] = 50.0      # one thread's round and another CTA -> 1
    logits[2, [40, 41]] = [-0.0, 0.0]                  # signed zeros tie -> 40
    logits[3, [50, 51]] = [0.0, -0.0]                  # -> 50
    logits[4, [7 + 1024, 7, 100]] = [np.nan, np.nan, np.inf]   # first NaN -> 7
    logits[5, [3, 131000]] = [np.inf, np.inf]          # -> 3
    logits[6] = -np.inf                                # -> 0
    logits[7, 131071] = 2.0                            # the last entry -> 131071
    logits[8] = -0.0                                   # all -0 -> 0
    logits[9, [23, 24, 131068]] = [np.nan, 5.0, np.nan]   # NaN in a word's last lane -> 23
    want = [9, 1, 40, 50, 7, 3, 0, 131071, 0, 23]
    assert [O.argmax_row(r) for r in logits] == want
    drafts = np.array(want[:-1], np.int32)
    drafts[4] = 8                                      # the first mismatch is draft 4
    n, bonus, committed = H.accept(ctx, logits, drafts, [0, rows])
    rn, rb, rc = O.accept(logits, drafts, [0, rows])
    assert n.tolist() == rn.tolist() == [4]
    assert bonus.tolist() == rb.tolist() == [7]
    assert committed.tolist() == rc.tolist()


def test_accept_ragged_batch_and_repeat_calls(H, vfy, ctx):
    """Eight sequences, depths from {2,4,8,11,16} and one depth 0; the second call must not see the
    first call's state."""
    rng = np.random.default_rng(8)
    V = 131072
    depths = [2, 4, 8, 11, 16, 16, 0, 2]
    cu = np.concatenate([[0], np.cumsum([d + 1 for d in depths])]).astype(np.int32)
    for trial in range(2):
        targets = rng.integers(0, V, int(cu[-1]))
        logits = synth.planted_logits(rng, targets, V)
        drafts = np.concatenate([synth.drafts_matching(rng, targets[cu[b]:cu[b + 1]], 0.56, V)
                                 for b in range(len(depths))]).astype(np.int32)
        n, bonus, committed = H.accept(ctx, logits, drafts, cu)
        rn, rb, rc = O.accept(logits, drafts, cu)
        assert n.tolist() == rn.tolist() and bonus.tolist() == rb.tolist()
        assert committed.tolist() == rc.tolist()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
