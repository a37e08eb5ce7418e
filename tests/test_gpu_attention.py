"""GPU parity of vfy_attend_full / vfy_attend_swa against the fp64 oracle, through the C ABI.

Workloads follow 'Laguna XS 2.1 33B on a RTX 3090' (lucebox): 16 drafts + 1 verified together
('The model ...'), a pool of 64-token chunks with a resident subset ('Three optimizations',
item 1), a 512-token window in a 2048-slot ring (item 3). Tolerance: elementwise
|gpu - oracle| <= 2e-2 + 1e-2 |oracle| and normwise <= 1e-2 (bf16 in, fp32 accumulate).
"""
import numpy as np
import pytest

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

C = 64


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


def make_ctx(vfy, shape, max_seqs=1, max_q=17, **kw):
    return vfy.vfy_create(shape.num_q_heads, shape.num_kv_heads, shape.head_dim, max_seqs=max_seqs,
                          max_queries_per_seq=max_q, device=0, **kw)


def paged_case(rng, shape, L, q, n_slots=None, resident=None, std=1.0):
    n = (L + C - 1) // C
    ids = np.arange(n) if resident is None else np.array(sorted(resident))
    n_slots = n_slots or n + 5
    slots = rng.permutation(n_slots)[: len(ids)].astype(np.int32)
    kp = synth.normal_bf16(rng, (n_slots, shape.num_kv_heads, C, shape.head_dim), std)
    vp = synth.normal_bf16(rng, (n_slots, shape.num_kv_heads, C, shape.head_dim), std)
    qb = synth.normal_bf16(rng, (q, shape.num_q_heads, shape.head_dim), std)
    return qb, kp, vp, ids.astype(np.int32), slots


def run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, L, what):
    q = qb.shape[0]
    got, lse = H.attend_full(ctx, qb, [0, q], kp, vp, ids, slots, [0, len(ids)], [L])
    ref, rlse = O.attend_full_seq(qb, kp, vp, ids, slots, L)
    assert_attn_close(got, ref, what)
    assert_lse_close(lse, rlse, what)
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


def test_full_tiny_config(H, vfy):
    """1 sequence, 17 queries, 4 q-heads / 1 KV head, d = 64, 1024 tokens = 16 chunks all resident
    in permuted slots, Q/K/V ~ 0.5 N(0,1), seed 0."""
    rng = np.random.default_rng(0)
    ctx = make_ctx(vfy, synth.TINY)
    qb, kp, vp, ids, slots = paged_case(rng, synth.TINY, 1024, 17, std=0.5)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, 1024, "tiny")


@pytest.mark.parametrize("splits", [1, 3, 16, 64])
def test_full_split_counts(H, vfy, splits):
    """Any split count gives the same answer (the combine is exact up to rounding)."""
    rng = np.random.default_rng(1)
    ctx = make_ctx(vfy, synth.LAGUNA)
    vfy.vfy_set_splits(ctx, splits, 0)
    qb, kp, vp, ids, slots = paged_case(rng, synth.LAGUNA, 3000, 17)      # 47 chunks, ragged tail
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, 3000, f"splits={splits}")


@pytest.mark.parametrize("L", [1, 17, 63, 64, 65, 129, 1000])
def test_full_short_and_ragged_lengths(H, vfy, L):
    rng = np.random.default_rng(L)
    q = min(17, L)
    ctx = make_ctx(vfy, synth.LAGUNA)
    qb, kp, vp, ids, slots = paged_case(rng, synth.LAGUNA, L, q)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, L, f"L={L}")


def test_full_32k_top128_pool(H, vfy):
    """32K context = 512 chunks; the resident pool is the top-128 by Gumbel scores (block chunk
    forced), held in shuffled slots."""
    rng = np.random.default_rng(2)
    s = synth.LAGUNA
    L, q, n, k = 32768, 17, 512, 128
    scores = synth.force_block_resident(synth.gumbel_scores(rng, n), L, q)
    ids = np.array(O.select_resident_one(scores, k, [-1] * n, 0)[0], dtype=np.int32)
    slots = rng.permutation(k).astype(np.int32)
    store_k = synth.normal_bf16(rng, (n, s.num_kv_heads, C, s.head_dim))
    store_v = synth.normal_bf16(rng, (n, s.num_kv_heads, C, s.head_dim))
    kp = np.zeros((k,) + store_k.shape[1:], np.uint16)
    vp = np.zeros_like(kp)
    kp[slots] = store_k[ids]
    vp[slots] = store_v[ids]
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, L, "32K top-128")


def test_full_rows_without_keys(H, vfy):
    """Resident set = only the last chunk; early queries of the block see no key: O = 0, LSE = -inf."""
    rng = np.random.default_rng(3)
    s = synth.LAGUNA
    L, q = 64 * 10 + 5, 17             # last chunk holds positions 640..644; queries at 628..644
    qb, kp, vp, _, _ = paged_case(rng, s, L, q)
    ids = np.array([10], np.int32)
    slots = np.array([4], np.int32)
    ctx = make_ctx(vfy, s)
    got, lse = H.attend_full(ctx, qb, [0, q], kp, vp, ids, slots, [0, 1], [L])
    ref, rlse = O.attend_full_seq(qb, kp, vp, ids, slots, L)
    assert np.all(np.isneginf(rlse[:12])) and np.all(O.bf16_to_f64(got[:12]) == 0)
    assert_attn_close(got, ref, "empty rows")
    assert_lse_close(lse, rlse, "empty rows")


def test_full_rescale_path(H, vfy):
    """Keys grow in magnitude along the context, so the running maximum rises by far more than
    the rescale threshold several times within one split."""
    rng = np.random.default_rng(4)
    s = synth.LAGUNA
    L, q, n = 1024, 17, 16
    q_f = rng.standard_normal((q, s.num_q_heads, s.head_dim)).astype(np.float32)
    k_f = rng.standard_normal((n, s.num_kv_heads, C, s.head_dim)).astype(np.float32)
    k_f *= np.linspace(0.2, 6.0, n, dtype=np.float32)[:, None, None, None]
    qb = synth.bf16_bits(q_f)
    kp = synth.bf16_bits(k_f)
    vp = synth.normal_bf16(rng, kp.shape)
    ids = np.arange(n, dtype=np.int32)
    ctx = make_ctx(vfy, s)
    vfy.vfy_set_splits(ctx, 1, 0)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, ids.copy(), L, "rescale")


def test_full_nan_poison_outside_the_attended_set(H, vfy):
    """NaN in every pool slot that is not resident, and in the unused tail of the last chunk,
    must not reach the output."""
    rng = np.random.default_rng(5)
    s = synth.LAGUNA
    L, q = 1000, 17                     # 16 chunks; chunk 15 holds 960..999, tail 1000..1023
    qb, kp, vp, ids, slots = paged_case(rng, s, L, q, n_slots=24, resident=[0, 2, 5, 9, 14, 15])
    nan = np.uint16(0x7FC0)
    for sl in set(range(24)) - set(slots.tolist()):
        kp[sl] = nan
        vp[sl] = nan
    tail_slot = slots[-1]
    kp[tail_slot, :, 1000 - 960:] = nan
    vp[tail_slot, :, 1000 - 960:] = nan
    ctx = make_ctx(vfy, s)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, L, "NaN poison")


def test_full_ragged_batch(H, vfy):
    """Several sequences with different depths (q = D + 1) and lengths in one call."""
    rng = np.random.default_rng(6)
    s = synth.LAGUNA
    depths = [2, 16, 4, 11, 8]
    lens = [300, 5000, 64, 2049, 777]
    qs = [d + 1 for d in depths]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    n_per = [(L + C - 1) // C for L in lens]
    total_slots = sum(n_per) + 7
    perm = rng.permutation(total_slots)
    kp = synth.normal_bf16(rng, (total_slots, s.num_kv_heads, C, s.head_dim))
    vp = synth.normal_bf16(rng, (total_slots, s.num_kv_heads, C, s.head_dim))
    qb = synth.normal_bf16(rng, (int(cu_q[-1]), s.num_q_heads, s.head_dim))
    ids, slots, cu_res = [], [], [0]
    off = 0
    for n in n_per:
        ids += list(range(n))
        slots += perm[off:off + n].tolist()
        off += n
        cu_res.append(len(ids))
    ids = np.array(ids, np.int32)
    slots = np.array(slots, np.int32)
    ctx = make_ctx(vfy, s, max_seqs=8)
    got, lse = H.attend_full(ctx, qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    ref, rlse = O.attend_full(qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    assert_attn_close(got, ref, "ragged")
    assert_lse_close(lse, rlse, "ragged")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


# Splits over at least 8 resident chunks take tiles of two chunks. 150 chunks over 17 or 19 splits
# give splits of 7 to 9 chunks, so some tiles hold one chunk only; 64 splits stay on 1-chunk tiles.
@pytest.mark.parametrize("splits", [17, 19, 64])
def test_full_wide_tiles(H, vfy, splits):
    rng = np.random.default_rng(21)
    ctx = make_ctx(vfy, synth.LAGUNA)
    vfy.vfy_set_splits(ctx, splits, 0)
    L = 150 * C - 37                                                      # ragged last chunk
    qb, kp, vp, ids, slots = paged_case(rng, synth.LAGUNA, L, 17)
    run_full_and_check(H, vfy, ctx, qb, kp, vp, ids, slots, L, f"wide splits={splits}")


def test_full_wide_tiles_ragged_batch(H, vfy):
    """Sequences of 150, 37 and 1 resident chunks with 17 splits: the long one takes two-chunk
    tiles, and so does every sequence in the launch, down to one tile with a single chunk."""
    rng = np.random.default_rng(22)
    s = synth.LAGUNA
    lens = [150 * C, 37 * C - 5, 50]
    qs = [17, 9, 17]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    n_per = [(L + C - 1) // C for L in lens]
    total_slots = sum(n_per) + 3
    perm = rng.permutation(total_slots)
    kp = synth.normal_bf16(rng, (total_slots, s.num_kv_heads, C, s.head_dim))
    vp = synth.normal_bf16(rng, (total_slots, s.num_kv_heads, C, s.head_dim))
    qb = synth.normal_bf16(rng, (int(cu_q[-1]), s.num_q_heads, s.head_dim))
    ids, slots, cu_res = [], [], [0]
    off = 0
    for n in n_per:
        ids += list(range(n))
        slots += perm[off:off + n].tolist()
        off += n
        cu_res.append(len(ids))
    ids = np.array(ids, np.int32)
    slots = np.array(slots, np.int32)
    ctx = make_ctx(vfy, s, max_seqs=4)
    vfy.vfy_set_splits(ctx, 17, 0)
    got, lse = H.attend_full(ctx, qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    ref, rlse = O.attend_full(qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    assert_attn_close(got, ref, "wide ragged")
    assert_lse_close(lse, rlse, "wide ragged")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


def test_full_wide_tiles_bad_slot_is_reported(H, vfy):
    rng = np.random.default_rng(23)
    s = synth.LAGUNA
    qb, kp, vp, ids, slots = paged_case(rng, s, 150 * C, 17)
    slots = slots.copy()
    slots[77] = 10_000_000
    ctx = make_ctx(vfy, s)
    vfy.vfy_set_splits(ctx, 17, 0)
    H.attend_full(ctx, qb, [0, 17], kp, vp, ids, slots, [0, len(ids)], [150 * C])
    assert vfy.vfy_get_status(ctx) == vfy.VFY_EDEVICE_INPUT


def test_full_bad_slot_is_reported_not_faulted(H, vfy):
    rng = np.random.default_rng(7)
    s = synth.LAGUNA
    qb, kp, vp, ids, slots = paged_case(rng, s, 500, 17)
    slots = slots.copy()
    slots[2] = 10_000_000
    ctx = make_ctx(vfy, s)
    H.attend_full(ctx, qb, [0, 17], kp, vp, ids, slots, [0, len(ids)], [500])
    assert vfy.vfy_get_status(ctx) == vfy.VFY_EDEVICE_INPUT
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK      # the word was cleared


# ---------------------------------------------------------------------------------------------
# Window layers
# ---------------------------------------------------------------------------------------------

def ring_case(rng, shape, B, R=2048, std=1.0):
    k = synth.normal_bf16(rng, (B, shape.num_kv_heads, R, shape.head_dim), std)
    v = synth.normal_bf16(rng, (B, shape.num_kv_heads, R, shape.head_dim), std)
    return k, v


def test_swa_32k_wrapping(H, vfy):
    """Same heads, 2048-slot ring with the write head placed so the 528-position span wraps."""
    rng = np.random.default_rng(10)
    s = synth.LAGUNA
    L, q = 32768, 17
    rk, rv = ring_case(rng, s, 1)
    phi = synth.wrapping_ring_offset(rng, L, 512 + q - 1, 2048)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s)
    got, lse = H.attend_swa(ctx, qb, [0, q], rk, rv, [phi], [L])
    ref, rlse = O.attend_ring_seq(qb, rk[0], rv[0], phi, L, 512)
    assert_attn_close(got, ref, "swa wrap")
    assert_lse_close(lse, rlse, "swa wrap")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


# Up to 16 splits merge inside the attention kernel (one cluster per KV head); 17 and 40 go through
# the combine kernel. 16 and 40 leave some splits without a tile.
@pytest.mark.parametrize("splits", [1, 2, 5, 10, 16, 17, 40])
@pytest.mark.parametrize("phi", [0, 63, 64, 1500, 2047])
def test_swa_offsets_and_splits(H, vfy, phi, splits):
    rng = np.random.default_rng(11 + phi)
    s = synth.LAGUNA
    L, q = 9000, 17
    rk, rv = ring_case(rng, s, 1)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s)
    vfy.vfy_set_splits(ctx, 0, splits)
    got, lse = H.attend_swa(ctx, qb, [0, q], rk, rv, [phi], [L])
    ref, rlse = O.attend_ring_seq(qb, rk[0], rv[0], phi, L, 512)
    assert_attn_close(got, ref, f"phi={phi} splits={splits}")
    assert_lse_close(lse, rlse, f"phi={phi} splits={splits}")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


@pytest.mark.parametrize("splits,kernels", [(10, 1), (16, 1), (17, 2)])
def test_swa_kernels_per_call(H, vfy, splits, kernels):
    """Splits that fit one cluster merge in the attention kernel; more add the combine kernel."""
    rng = np.random.default_rng(31)
    s = synth.LAGUNA
    rk, rv = ring_case(rng, s, 1)
    qb = synth.normal_bf16(rng, (17, s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s)
    vfy.vfy_set_splits(ctx, 0, splits)
    n0 = vfy.vfy_launch_count(ctx)
    H.attend_swa(ctx, qb, [0, 17], rk, rv, [5], [9000])
    assert vfy.vfy_launch_count(ctx) - n0 == kernels


@pytest.mark.parametrize("L", [1, 17, 100, 511, 512, 528, 529, 2000])
def test_swa_short_sequences(H, vfy, L):
    rng = np.random.default_rng(100 + L)
    s = synth.TINY
    q = min(17, L)
    rk, rv = ring_case(rng, s, 1, std=0.5)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim), 0.5)
    ctx = make_ctx(vfy, s)
    got, lse = H.attend_swa(ctx, qb, [0, q], rk, rv, [700], [L])
    ref, rlse = O.attend_ring_seq(qb, rk[0], rv[0], 700, L, 512)
    assert_attn_close(got, ref, f"L={L}")
    assert_lse_close(lse, rlse, f"L={L}")


def test_swa_nan_poison_outside_the_window(H, vfy):
    rng = np.random.default_rng(12)
    s = synth.LAGUNA
    L, q, R = 20000, 17, 2048
    rk, rv = ring_case(rng, s, 1)
    phi = synth.wrapping_ring_offset(rng, L, 512 + q - 1, R)
    live = {(p + phi) % R for p in range(L - 528, L)}
    dead = np.array(sorted(set(range(R)) - live))
    rk[0][:, dead] = np.uint16(0x7FC0)
    rv[0][:, dead] = np.uint16(0x7FC0)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s)
    got, _ = H.attend_swa(ctx, qb, [0, q], rk, rv, [phi], [L])
    ref, _ = O.attend_ring_seq(qb, rk[0], rv[0], phi, L, 512)
    assert_attn_close(got, ref, "swa poison")


def test_swa_ragged_batch(H, vfy):
    rng = np.random.default_rng(13)
    s = synth.LAGUNA
    depths = [2, 4, 8, 11, 16, 16, 2, 8]
    lens = [4000, 200000, 513, 99999, 17, 60000, 3, 1234]
    qs = [min(d + 1, L) for d, L in zip(depths, lens)]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    rk, rv = ring_case(rng, s, len(lens))
    phis = rng.integers(0, 2048, len(lens)).astype(np.int32)
    qb = synth.normal_bf16(rng, (int(cu_q[-1]), s.num_q_heads, s.head_dim))
    ctx = make_ctx(vfy, s, max_seqs=8)
    got, lse = H.attend_swa(ctx, qb, cu_q, rk, rv, phis, lens)
    ref, rlse = O.attend_ring(qb, cu_q, rk, rv, phis, lens, 512)
    assert_attn_close(got, ref, "swa ragged")
    assert_lse_close(lse, rlse, "swa ragged")


@pytest.mark.parametrize("tiles_per_split", [1, 2, 3])
def test_repeated_short_splits_are_stable(H, vfy, tiles_per_split):
    """Splits of one to three tiles, repeated: the epilogue must wait for the last P.V MMA even
    when the previous one is still running."""
    rng = np.random.default_rng(20 + tiles_per_split)
    s = synth.LAGUNA
    L, q, R = 9000, 17, 2048
    rk, rv = ring_case(rng, s, 1)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    phi = 1500                                     # 10 slot-aligned tiles
    ctx = make_ctx(vfy, s)
    vfy.vfy_set_splits(ctx, 0, 10 // tiles_per_split)
    ref, _ = O.attend_ring_seq(qb, rk[0], rv[0], phi, L, 512)
    for rep in range(25):
        got, _ = H.attend_swa(ctx, qb, [0, q], rk, rv, [phi], [L])
        assert_attn_close(got, ref, f"rep {rep}")
