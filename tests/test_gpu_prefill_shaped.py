"""Prefill-shaped verify: a block of up to 1024 queries through the same paged and ring kernels
('Laguna XS 2.1 33B on a RTX 3090', 'Three optimizations' item 1: the prefill runs through the
pool in 1024-token batches with CUDA-graph replay). Query i of a q-token block sits at position
L - q + i and attends causally, so the block's q * G rows split into row tiles of 128, each with
CTAs of its own. Checked against the fp64 oracle on every row: the full layer for automatic and
few splits (two-chunk tiles and the combine), many splits (one-chunk tiles and the combine) and
16 splits (4 chunks each: the cluster merge); the window layer; a ragged batch."""
import numpy as np
import pytest

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

C = 64
QB = 1024


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


def ctx_for(vfy, max_seqs=1, max_splits=48):
    s = synth.LAGUNA
    return vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=max_seqs, max_queries_per_seq=QB,
                          max_splits=max_splits, device=0)


@pytest.mark.parametrize("splits", [0, 40, 3, 16])
def test_prefill_shaped_full_layer(H, vfy, splits):
    rng = np.random.default_rng(60 + splits)
    s = synth.LAGUNA
    L = 4096 + 37
    n = (L + C - 1) // C
    slots = rng.permutation(n + 3)[:n].astype(np.int32)
    ids = np.arange(n, dtype=np.int32)
    kp = synth.normal_bf16(rng, (n + 3, s.num_kv_heads, C, s.head_dim))
    vp = synth.normal_bf16(rng, (n + 3, s.num_kv_heads, C, s.head_dim))
    qb = synth.normal_bf16(rng, (QB, s.num_q_heads, s.head_dim))
    ctx = ctx_for(vfy)
    vfy.vfy_set_splits(ctx, splits, 0)
    got, lse = H.attend_full(ctx, qb, [0, QB], kp, vp, ids, slots, [0, n], [L])
    ref, rlse = O.attend_full_seq(qb, kp, vp, ids, slots, L)
    assert_attn_close(got, ref, f"prefill-shaped full splits={splits}")
    assert_lse_close(lse, rlse, f"prefill-shaped full splits={splits}")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


@pytest.mark.parametrize("splits", [0, 17])
def test_prefill_shaped_window_layer(H, vfy, splits):
    rng = np.random.default_rng(70 + splits)
    s = synth.LAGUNA
    L = 9000
    k = synth.normal_bf16(rng, (1, s.num_kv_heads, synth.RING, s.head_dim))
    v = synth.normal_bf16(rng, (1, s.num_kv_heads, synth.RING, s.head_dim))
    phi = synth.wrapping_ring_offset(rng, L, synth.WINDOW + QB - 1, synth.RING)
    qb = synth.normal_bf16(rng, (QB, s.num_q_heads, s.head_dim))
    ctx = ctx_for(vfy)
    vfy.vfy_set_splits(ctx, 0, splits)
    got, lse = H.attend_swa(ctx, qb, [0, QB], k, v, [phi], [L])
    ref, rlse = O.attend_ring_seq(qb, k[0], v[0], phi, L, synth.WINDOW)
    assert_attn_close(got, ref, f"prefill-shaped window splits={splits}")
    assert_lse_close(lse, rlse, f"prefill-shaped window splits={splits}")


def test_prefill_shaped_ragged_batch(H, vfy):
    """A 1000-query block next to a 17-query verify block and a 300-query block in one call."""
    rng = np.random.default_rng(80)
    s = synth.LAGUNA
    lens = [3000, 1500, 777]
    qs = [1000, 17, 300]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    n_per = [(L + C - 1) // C for L in lens]
    total = sum(n_per) + 4
    perm = rng.permutation(total)
    kp = synth.normal_bf16(rng, (total, s.num_kv_heads, C, s.head_dim))
    vp = synth.normal_bf16(rng, (total, s.num_kv_heads, C, s.head_dim))
    qb = synth.normal_bf16(rng, (int(cu_q[-1]), s.num_q_heads, s.head_dim))
    ids, slots, cu_res, off = [], [], [0], 0
    for n in n_per:
        ids += list(range(n))
        slots += perm[off:off + n].tolist()
        off += n
        cu_res.append(len(ids))
    ids, slots = np.array(ids, np.int32), np.array(slots, np.int32)
    ctx = ctx_for(vfy, max_seqs=3)
    got, lse = H.attend_full(ctx, qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    ref, rlse = O.attend_full(qb, cu_q, kp, vp, ids, slots, cu_res, lens)
    assert_attn_close(got, ref, "prefill-shaped ragged")
    assert_lse_close(lse, rlse, "prefill-shaped ragged")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
