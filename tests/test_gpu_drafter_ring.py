"""The drafter's context-KV ring through the window-attention kernel ('Laguna XS 2.1 33B on a RTX
3090', 'Three optimizations' item 2: the drafter's K/V sit in a position-indexed ring over a
feature window of up to 4K tokens; 'The model ...': 16 proposals per step). The 16 proposal
positions attend the last 4096 positions of a ring of 8192 slots, with the write head placed so
that the block's span wraps. The pages give no drafter head counts: the target's 16 q / 4 KV x
128 are reused. Checked against the fp64 oracle on every row, for automatic split counts (the
combine path), for 16 and fewer splits (the cluster merge, several tiles per split), short
contexts and a ragged batch."""
import numpy as np
import pytest

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

W, R, Q = synth.DRAFTER_WINDOW, synth.DRAFTER_RING, synth.DRAFT


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


def drafter_ctx(vfy, max_seqs=1):
    s = synth.LAGUNA
    return vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, window=W, ring_len=R, max_seqs=max_seqs,
                          max_queries_per_seq=Q, device=0)


def rings(rng, B):
    s = synth.LAGUNA
    k = synth.normal_bf16(rng, (B, s.num_kv_heads, R, s.head_dim))
    v = synth.normal_bf16(rng, (B, s.num_kv_heads, R, s.head_dim))
    return k, v


@pytest.mark.parametrize("splits", [0, 3, 16, 40])
def test_drafter_ring_window_4k(H, vfy, splits):
    rng = np.random.default_rng(40 + splits)
    s = synth.LAGUNA
    L = 262144
    k, v = rings(rng, 1)
    phi = synth.wrapping_ring_offset(rng, L, W + Q - 1, R)
    qb = synth.normal_bf16(rng, (Q, s.num_q_heads, s.head_dim))
    ctx = drafter_ctx(vfy)
    vfy.vfy_set_splits(ctx, 0, splits)
    got, lse = H.attend_swa(ctx, qb, [0, Q], k, v, [phi], [L])
    ref, rlse = O.attend_ring_seq(qb, k[0], v[0], phi, L, W)
    assert_attn_close(got, ref, f"drafter ring splits={splits}")
    assert_lse_close(lse, rlse, f"drafter ring splits={splits}")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK


@pytest.mark.parametrize("L", [16, 100, 4095, 4111, 4112, 6000])
def test_drafter_ring_short_contexts(H, vfy, L):
    """Contexts shorter than, equal to and just past the window plus the block."""
    rng = np.random.default_rng(L)
    s = synth.LAGUNA
    k, v = rings(rng, 1)
    phi = int(rng.integers(0, R))
    q = min(Q, L)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = drafter_ctx(vfy)
    got, lse = H.attend_swa(ctx, qb, [0, q], k, v, [phi], [L])
    ref, rlse = O.attend_ring_seq(qb, k[0], v[0], phi, L, W)
    assert_attn_close(got, ref, f"drafter ring L={L}")
    assert_lse_close(lse, rlse, f"drafter ring L={L}")


def test_drafter_ring_ragged_batch(H, vfy):
    rng = np.random.default_rng(50)
    s = synth.LAGUNA
    lens = [262144, 5000, 4200, 100000]
    qs = [16, 12, 5, 9]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    k, v = rings(rng, len(lens))
    phis = [synth.wrapping_ring_offset(rng, L, W + q - 1, R) for L, q in zip(lens, qs)]
    qb = synth.normal_bf16(rng, (int(cu_q[-1]), s.num_q_heads, s.head_dim))
    ctx = drafter_ctx(vfy, max_seqs=4)
    got, lse = H.attend_swa(ctx, qb, cu_q, k, v, phis, lens)
    ref, rlse = O.attend_ring(qb, cu_q, k, v, phis, lens, W)
    assert_attn_close(got, ref, "drafter ring ragged")
    assert_lse_close(lse, rlse, "drafter ring ragged")
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
