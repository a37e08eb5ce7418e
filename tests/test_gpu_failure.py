"""Failure detection without a GPU fault: every wait of the attention pipeline is bounded, and a
wait that runs out is reported through the context's error word while the context stays usable.

The test (vfy_test_wait_timeout) has every CTA of the next attention call wait 2 us on a barrier
that nothing completes: a flag nothing sets. That wait runs out, the CTA's other waits give up,
copies and MMAs in flight drain under the default limit. vfy_get_status must then say
VFY_EDEVICE_TIMEOUT, and the next call, with the test off, must return VFY_OK and match the
oracle. Each attention variant is covered: a full layer through the combine kernel (narrow and
wide tiles) and a window layer that merges its splits in a thread-block cluster."""
import numpy as np
import pytest

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

C = 64


@pytest.fixture(scope="module")
def env():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import harness, vfy
    return harness, vfy


def _full_case(rng, L, k):
    s = synth.LAGUNA
    n = (L + C - 1) // C
    resident = np.sort(np.concatenate([rng.choice(n - 1, k - 1, replace=False), [n - 1]])).astype(np.int32)
    slots = rng.permutation(k).astype(np.int32)
    kp = synth.normal_bf16(rng, (k, s.num_kv_heads, C, s.head_dim))
    vp = synth.normal_bf16(rng, (k, s.num_kv_heads, C, s.head_dim))
    qb = synth.normal_bf16(rng, (17, s.num_q_heads, s.head_dim))
    return qb, kp, vp, resident, slots


@pytest.mark.parametrize("splits", [0, 2])      # automatic (narrow tiles), 2 splits (wide tiles)
def test_full_layer_wait_timeout_is_reported_and_recovered(env, splits):
    H, vfy = env
    rng = np.random.default_rng(40 + splits)
    s = synth.LAGUNA
    L, k = 32768, 128
    qb, kp, vp, ids, slots = _full_case(rng, L, k)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_queries_per_seq=17, device=0)
    try:
        vfy.vfy_set_splits(ctx, splits, 0)
        assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
        vfy.vfy_test_wait_timeout(ctx, 2000)
        H.attend_full(ctx, qb, [0, 17], kp, vp, ids, slots, [0, k], [L])
        assert vfy.vfy_get_status(ctx) == vfy.VFY_EDEVICE_TIMEOUT
        assert vfy.vfy_get_status(ctx) == vfy.VFY_OK          # read and cleared
        vfy.vfy_test_wait_timeout(ctx, 0)
        got, lse = H.attend_full(ctx, qb, [0, 17], kp, vp, ids, slots, [0, k], [L])
        assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
        ref, rlse = O.attend_full_seq(qb, kp, vp, ids, slots, L)
        assert_attn_close(got, ref, "full layer after a timeout")
        assert_lse_close(lse, rlse, "full layer after a timeout")
    finally:
        ctx.close()


def test_window_layer_wait_timeout_is_reported_and_recovered(env):
    H, vfy = env
    rng = np.random.default_rng(47)
    s = synth.LAGUNA
    L = 32768
    phi = synth.wrapping_ring_offset(rng, L, synth.WINDOW + 16, synth.RING)
    kr = synth.normal_bf16(rng, (1, s.num_kv_heads, synth.RING, s.head_dim))
    vr = synth.normal_bf16(rng, (1, s.num_kv_heads, synth.RING, s.head_dim))
    qb = synth.normal_bf16(rng, (17, s.num_q_heads, s.head_dim))
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_queries_per_seq=17, device=0)
    try:
        vfy.vfy_test_wait_timeout(ctx, 2000)
        H.attend_swa(ctx, qb, [0, 17], kr, vr, [phi], [L])
        assert vfy.vfy_get_status(ctx) == vfy.VFY_EDEVICE_TIMEOUT
        vfy.vfy_test_wait_timeout(ctx, 0)
        got, lse = H.attend_swa(ctx, qb, [0, 17], kr, vr, [phi], [L])
        assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
        ref, rlse = O.attend_ring_seq(qb, kr[0], vr[0], phi, L, synth.WINDOW)
        assert_attn_close(got, ref, "window layer after a timeout")
        assert_lse_close(lse, rlse, "window layer after a timeout")
    finally:
        ctx.close()
