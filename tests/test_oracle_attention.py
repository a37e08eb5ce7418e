"""Pins of the oracle's attention (full-layer pool attention and ring-window attention).

The oracle gathers an explicit key list from a chunk pool or a ring and loops over queries.
These tests check it against formulations that share nothing with that code:
  * dense attention over the logical (unpaged, unrotated) K/V arrays with a mask built by
    numpy.tril / numpy.triu, GQA by numpy.repeat, softmax and LSE by scipy.special;
  * closed forms (a single key, identical keys, Q = 0, a two-key LSE);
  * one-hot probes at the window edge and just past the causal boundary.
A last group plants mistakes in the oracle's small definitions and checks that a pin fails.
Sources: 'Laguna XS 2.1 33B on a RTX 3090' (lucebox), 'Three optimizations', items 1 and 3.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

C = 64


def logical_from_store(store):
    """[chunk][Hkv][64][d] -> [pos][Hkv][d]"""
    n, hkv, t, d = store.shape
    return store.transpose(0, 2, 1, 3).reshape(n * t, hkv, d)


def dense_attention(q_bits, k_log_bits, v_log_bits, mask, scale=None):
    """Dense masked attention: q [q][Hq][d], K/V [P][Hkv][d], mask [q][P] bool."""
    q = O.bf16_to_f64(q_bits)
    k = O.bf16_to_f64(k_log_bits)
    v = O.bf16_to_f64(v_log_bits)
    hq, hkv, d = q.shape[1], k.shape[1], q.shape[2]
    k = np.repeat(k, hq // hkv, axis=1)
    v = np.repeat(v, hq // hkv, axis=1)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    s = np.einsum("qhd,phd->hqp", q, k) * scale
    s = np.where(mask[None, :, :], s, -np.inf)
    empty = ~mask.any(axis=1)
    s_safe = np.where(empty[None, :, None], 0.0, s)
    p = softmax(s_safe, axis=-1)
    p = np.where(empty[None, :, None], 0.0, p)
    out = np.einsum("hqp,phd->qhd", p, v)
    lse = logsumexp(s_safe, axis=-1).T
    lse = np.where(empty[:, None], -np.inf, lse)
    return out, lse


def causal_mask_last(L, q):
    """Rows = the last q positions of a length-L causal (lower-triangular) mask."""
    return np.tril(np.ones((L, L), dtype=bool))[L - q:]


def band_mask_last(L, q, w):
    """Causal band of width w (self included), last q rows."""
    full = np.tril(np.ones((L, L), dtype=bool)) & ~np.tril(np.ones((L, L), dtype=bool), -w)
    return full[L - q:]


def make_paged(rng, shape, L, n_chunks, q, std=0.5):
    hkv, d = shape.num_kv_heads, shape.head_dim
    store_k = synth.normal_bf16(rng, (n_chunks, hkv, C, d), std)
    store_v = synth.normal_bf16(rng, (n_chunks, hkv, C, d), std)
    qb = synth.normal_bf16(rng, (q, shape.num_q_heads, d), std)
    return qb, store_k, store_v


def pool_with_permuted_slots(rng, store_k, store_v, ids, num_slots):
    slots = rng.permutation(num_slots)[: len(ids)]
    pk = synth.normal_bf16(rng, (num_slots,) + store_k.shape[1:])
    pv = synth.normal_bf16(rng, (num_slots,) + store_v.shape[1:])
    pk[slots] = store_k[ids]
    pv[slots] = store_v[ids]
    return pk, pv, slots


# ---------------------------------------------------------------------------------------------
# Paged full-layer attention
# ---------------------------------------------------------------------------------------------

def check_paged_vs_dense(seed=0, shape=synth.TINY, L=1024, q=17, resident=None, tol=1e-11):
    rng = np.random.default_rng(seed)
    n = (L + C - 1) // C
    qb, sk, sv = make_paged(rng, shape, L, n, q)
    ids = np.arange(n) if resident is None else np.array(sorted(resident))
    pk, pv, slots = pool_with_permuted_slots(rng, sk, sv, ids, n + 3)
    out, lse, rsum = O.attend_full_seq(qb, pk, pv, ids, slots, L, return_rowsum=True)
    k_log = logical_from_store(sk)[:L]
    v_log = logical_from_store(sv)[:L]
    mask = causal_mask_last(L, q)
    if resident is not None:
        in_pool = np.zeros(L, dtype=bool)
        for c in ids:
            in_pool[c * C:(c + 1) * C] = True
        mask = mask & in_pool[None, :]
    ref, ref_lse = dense_attention(qb, k_log, v_log, mask)
    ok_rows = mask.any(axis=1)
    assert np.allclose(rsum[ok_rows], 1.0, atol=1e-12)
    same_empty = np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    return bool(same_empty and np.max(np.abs(out - ref)) <= tol
                and np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= tol)


def test_paged_all_resident_equals_dense_causal():
    """The identity: paged attention with every chunk resident == dense causal attention."""
    assert check_paged_vs_dense(seed=0, shape=synth.TINY, L=1024, q=17)


def test_paged_ragged_tail_and_gqa():
    shape = synth.Shape(4, 2, 32)
    assert check_paged_vs_dense(seed=1, shape=shape, L=300, q=17)      # 5 chunks, 44-token tail


def test_paged_subset_equals_dense_restricted():
    """Only the resident chunks' positions are attended."""
    shape = synth.Shape(4, 2, 32)
    assert check_paged_vs_dense(seed=2, shape=shape, L=700, q=9, resident=[0, 3, 4, 7, 10])


def test_paged_row_without_keys_is_zero():
    """If no resident position is <= p_i, the row outputs 0 and LSE = -inf."""
    rng = np.random.default_rng(3)
    shape = synth.Shape(2, 1, 16)
    L, q = 200, 5
    qb, sk, sv = make_paged(rng, shape, L, 4, q)
    # resident: chunk 3 only (positions 192..199); queries sit at 195..199 -> query 0 sees 192..195
    out, lse = O.attend_full_seq(qb, sk, sv, [3], [3], L)
    assert np.isfinite(lse).all()
    out2, lse2 = O.attend_full_seq(qb, sk, sv, [3], [3], 190 + q)   # L=195: chunk 3 starts at 192
    # queries at 190..194: query 0 (190) and 1 (191) see nothing in chunk 3
    assert np.all(out2[:2] == 0) and np.all(np.isneginf(lse2[:2]))
    assert np.all(np.isfinite(lse2[2:]))


# ---------------------------------------------------------------------------------------------
# Ring-window attention
# ---------------------------------------------------------------------------------------------

def check_ring_vs_dense(seed=0, shape=synth.Shape(4, 2, 32), L=1000, q=17, W=64, R=256, tol=1e-11):
    rng = np.random.default_rng(seed)
    hkv, d = shape.num_kv_heads, shape.head_dim
    k_log = synth.normal_bf16(rng, (L, hkv, d), 0.7)
    v_log = synth.normal_bf16(rng, (L, hkv, d), 0.7)
    qb = synth.normal_bf16(rng, (q, shape.num_q_heads, d), 0.7)
    phi = synth.wrapping_ring_offset(rng, L, W + q - 1, R)
    # The ring holds positions L-R .. L-1; position p sits at slot (p + phi) mod R.
    # Build it with numpy.roll from the last R logical positions (slot j of the unrotated ring
    # holds position L - R + j; rolling by (L - R + phi) mod R moves it to its slot).
    tail_k = np.transpose(k_log[L - R:], (1, 0, 2))       # [Hkv][R][d]
    tail_v = np.transpose(v_log[L - R:], (1, 0, 2))
    ring_k = np.roll(tail_k, (L - R + phi) % R, axis=1)
    ring_v = np.roll(tail_v, (L - R + phi) % R, axis=1)
    out, lse, rsum = O.attend_ring_seq(qb, ring_k, ring_v, phi, L, W, return_rowsum=True)
    mask = band_mask_last(L, q, W)
    ref, ref_lse = dense_attention(qb, k_log, v_log, mask)
    assert np.allclose(rsum, 1.0, atol=1e-12)
    return np.max(np.abs(out - ref)) <= tol and np.max(np.abs(lse - ref_lse)) <= tol


def test_ring_equals_dense_window():
    assert check_ring_vs_dense()


def test_ring_real_sizes_wraps():
    """Window 512 in a 2048-slot ring with a write head that forces wraparound."""
    assert check_ring_vs_dense(seed=5, shape=synth.Shape(2, 1, 16), L=5000, q=17, W=512, R=2048)


def test_ring_short_sequence():
    """Context shorter than the window: every earlier position is attended."""
    assert _ring_short()


def _ring_short():
    rng = np.random.default_rng(6)
    L, q, W, R = 300, 17, 512, 2048
    k_log = synth.normal_bf16(rng, (L, 1, 16))
    v_log = synth.normal_bf16(rng, (L, 1, 16))
    qb = synth.normal_bf16(rng, (q, 2, 16))
    phi = 1900
    ring_k = np.zeros((1, R, 16), dtype=np.uint16)
    ring_v = np.zeros((1, R, 16), dtype=np.uint16)
    ring_k[0] = np.roll(np.concatenate([k_log[:, 0], np.zeros((R - L, 16), np.uint16)]), phi, axis=0)
    ring_v[0] = np.roll(np.concatenate([v_log[:, 0], np.zeros((R - L, 16), np.uint16)]), phi, axis=0)
    out, lse = O.attend_ring_seq(qb, ring_k, ring_v, phi, L, W)
    ref, ref_lse = dense_attention(qb, k_log, v_log, causal_mask_last(L, q))
    return np.max(np.abs(out - ref)) <= 1e-11 and np.max(np.abs(lse - ref_lse)) <= 1e-11


# ---------------------------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------------------------

def test_single_key_returns_its_value():
    rng = np.random.default_rng(7)
    qb = synth.normal_bf16(rng, (1, 2, 16))
    sk = synth.normal_bf16(rng, (1, 1, C, 16))
    sv = synth.normal_bf16(rng, (1, 1, C, 16))
    out, lse = O.attend_full_seq(qb, sk, sv, [0], [0], 1)     # L = 1: one position, one query
    v0 = O.bf16_to_f64(sv[0, 0, 0])
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)
    s = O.bf16_to_f64(qb[0]) @ O.bf16_to_f64(sk[0, 0, 0]) / 4.0
    assert np.allclose(lse[0], s, atol=1e-14)


def test_identical_keys_give_mean_value():
    rng = np.random.default_rng(8)
    L, q = 200, 3
    sk = np.tile(synth.normal_bf16(rng, (1, 1, 1, 16)), (4, 1, C, 1))
    sv = synth.normal_bf16(rng, (4, 1, C, 16))
    qb = synth.normal_bf16(rng, (q, 2, 16))
    out, lse = O.attend_full_seq(qb, sk, sv, range(4), range(4), L)
    vlog = O.bf16_to_f64(logical_from_store(sv)[:L, 0])
    for i in range(q):
        p = L - q + i
        assert np.allclose(out[i, 0], vlog[: p + 1].mean(axis=0), atol=1e-12)


def test_zero_query_gives_mean_value_and_log_count():
    rng = np.random.default_rng(9)
    L, q = 130, 2
    sk = synth.normal_bf16(rng, (3, 1, C, 8))
    sv = synth.normal_bf16(rng, (3, 1, C, 8))
    qb = np.zeros((q, 1, 8), dtype=np.uint16)
    out, lse = O.attend_full_seq(qb, sk, sv, range(3), range(3), L)
    vlog = O.bf16_to_f64(logical_from_store(sv)[:L, 0])
    for i in range(q):
        p = L - q + i
        assert np.allclose(out[i, 0], vlog[: p + 1].mean(axis=0), atol=1e-12)
        assert abs(lse[i, 0] - math.log(p + 1)) < 1e-12


def test_two_key_lse_and_weights():
    """Scores a, b -> weights e^a/(e^a+e^b), LSE = log(e^a + e^b); scale 1/sqrt(64) = 1/8."""
    d = 64
    qv = np.zeros(d, np.float32); qv[0] = 8.0
    k0 = np.zeros(d, np.float32); k0[0] = 1.5
    k1 = np.zeros(d, np.float32); k1[0] = -0.5
    v0 = np.zeros(d, np.float32); v0[1] = 1.0
    v1 = np.zeros(d, np.float32); v1[2] = 1.0
    sk = np.zeros((1, 1, C, d), np.uint16); sv = np.zeros((1, 1, C, d), np.uint16)
    sk[0, 0, 0], sk[0, 0, 1] = synth.bf16_bits(k0), synth.bf16_bits(k1)
    sv[0, 0, 0], sv[0, 0, 1] = synth.bf16_bits(v0), synth.bf16_bits(v1)
    qb = synth.bf16_bits(qv).reshape(1, 1, d)
    out, lse = O.attend_full_seq(qb, sk, sv, [0], [0], 2)        # query at position 1
    a, b = 1.5, -0.5
    assert abs(lse[0, 0] - math.log(math.exp(a) + math.exp(b))) < 1e-14
    assert abs(out[0, 0, 1] - math.exp(a) / (math.exp(a) + math.exp(b))) < 1e-14
    assert abs(out[0, 0, 2] - math.exp(b) / (math.exp(a) + math.exp(b))) < 1e-14


def onehot_ring_probe(offset_from_query):
    """Q = 0 (uniform weights), V one-hot at position p_last - offset; returns that coordinate."""
    L, q, W, R, d = 3000, 1, 512, 2048, 8
    ring_k = np.zeros((1, R, d), np.uint16)
    ring_v = np.zeros((1, R, d), np.uint16)
    phi = 777
    p = L - 1 - offset_from_query
    if p >= 0:
        ring_v[0, (p + phi) % R, 3] = synth.bf16_bits(np.float32([1.0]))[0]
    qb = np.zeros((q, 1, d), np.uint16)
    out, _ = O.attend_ring_seq(qb, ring_k, ring_v, phi, L, W)
    return out[0, 0, 3]


def test_window_edge_onehot():
    assert abs(onehot_ring_probe(511) - 1 / 512) < 1e-15     # p - 511: inside the window
    assert onehot_ring_probe(512) == 0.0                      # p - 512: outside
    assert abs(onehot_ring_probe(0) - 1 / 512) < 1e-15        # itself


def test_causality_onehot():
    """A value one position after query i never reaches query i."""
    L, q, d = 256, 4, 8
    sk = np.zeros((4, 1, C, d), np.uint16)
    sv = np.zeros((4, 1, C, d), np.uint16)
    qb = np.zeros((q, 1, d), np.uint16)
    p1 = L - q + 1                                 # position of query 1
    sv[(p1 + 1) // C, 0, (p1 + 1) % C, 5] = synth.bf16_bits(np.float32([1.0]))[0]
    out, _ = O.attend_full_seq(qb, sk, sv, range(4), range(4), L)
    assert out[1, 0, 5] == 0.0 and out[0, 0, 5] == 0.0
    assert abs(out[2, 0, 5] - 1.0 / (p1 + 2)) < 1e-15


def test_gqa_head_map_by_value():
    """KV head h holds the constant value h+1; q-head g must read KV head g // G."""
    L, q, d = 64, 2, 8
    hq, hkv = 6, 3
    sk = np.zeros((1, hkv, C, d), np.uint16)
    sv = np.zeros((1, hkv, C, d), np.uint16)
    for h in range(hkv):
        sv[0, h] = synth.bf16_bits(np.full((C, d), h + 1, np.float32))
    qb = synth.normal_bf16(np.random.default_rng(0), (q, hq, d))
    out, _ = O.attend_full_seq(qb, sk, sv, [0], [0], L)
    expect = np.repeat(np.arange(1, hkv + 1), hq // hkv)
    assert np.allclose(out[0, :, 0], expect, atol=1e-12, rtol=0)


# ---------------------------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------------------------

def all_attention_pins_pass():
    try:
        ok = (check_paged_vs_dense(seed=0, shape=synth.Shape(4, 2, 16), L=300, q=17)
              and check_ring_vs_dense(seed=0, shape=synth.Shape(4, 2, 16), L=600, q=17, W=64, R=256))
        test_window_edge_onehot()
        test_causality_onehot()
        test_gqa_head_map_by_value()
        test_two_key_lse_and_weights()
        return bool(ok)
    except AssertionError:
        return False


MUTATIONS = {
    "query position off by one": ("_query_position", lambda L, q, i: L - q + i + 1),
    "query position from the front": ("_query_position", lambda L, q, i: i),
    "GQA interleaved": ("_kv_head_of", lambda g, G: g % G),
    "window one too wide": ("_window_start", lambda p, w: max(0, p - w)),
    "window one too narrow": ("_window_start", lambda p, w: max(0, p - w + 2)),
    "ring offset sign": ("_ring_slot", lambda p, phi, R: (p - phi) % R),
    "scale 1/d": ("_default_scale", lambda d: 1.0 / d),
}


def test_pins_pass_on_the_oracle():
    assert all_attention_pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    assert not all_attention_pins_pass(), name


def test_dropped_normalisation_is_caught(monkeypatch):
    def unnormalised(q, keys, values, scale):
        if keys.shape[0] == 0:
            return np.zeros(values.shape[1]), -math.inf, 0.0
        s = scale * (keys @ q)
        w = np.exp(s - s.max())
        return w @ values, s.max() + math.log(w.sum()), 1.0
    monkeypatch.setattr(O, "softmax_attend", unnormalised)
    assert not all_attention_pins_pass()
