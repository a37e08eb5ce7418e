"""Block K/V append through the C ABI, bit-exact against the oracle: the block's rows land in the
chunk store (pinned host memory, written through over the host link, or device memory), in the
pool slot of resident chunks, and in the window layers' rings. Then append + attention in one
captured graph reads the block's own rows."""
import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

C = 64


@pytest.fixture(scope="module")
def vfy():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import vfy
    return vfy


def bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tensor(a, device="cuda", pin=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.to(device)


def i32(a):
    return torch.tensor(np.asarray(a, dtype=np.int32), dtype=torch.int32, device="cuda")


def full_case(rng, s, lens, qs):
    n_per = [(L + C - 1) // C for L in lens]
    cu_chunks = np.concatenate([[0], np.cumsum(n_per)]).astype(np.int32)
    n = int(cu_chunks[-1])
    slots = 3 * n // 4
    slot_of_chunk = np.full(n, -1, np.int32)
    chosen = rng.choice(n, slots - 2, replace=False)
    slot_of_chunk[chosen] = rng.permutation(slots)[: slots - 2]
    for b, L in enumerate(lens):                        # the block's last chunk is resident
        last = cu_chunks[b] + (L - 1) // C
        if slot_of_chunk[last] < 0:
            free = sorted(set(range(slots)) - set(slot_of_chunk[slot_of_chunk >= 0].tolist()))
            slot_of_chunk[last] = free[0]
    shape = (n, s.num_kv_heads, C, s.head_dim)
    store_k, store_v = synth.normal_bf16(rng, shape), synth.normal_bf16(rng, shape)
    pool_k = synth.normal_bf16(rng, (slots,) + shape[1:])
    pool_v = synth.normal_bf16(rng, (slots,) + shape[1:])
    T = int(sum(qs))
    k_new = synth.normal_bf16(rng, (T, s.num_kv_heads, s.head_dim))
    v_new = synth.normal_bf16(rng, (T, s.num_kv_heads, s.head_dim))
    return cu_chunks, slot_of_chunk, store_k, store_v, pool_k, pool_v, k_new, v_new


@pytest.mark.parametrize("pinned", [True, False])
def test_append_full_bit_exact(vfy, pinned):
    rng = np.random.default_rng(90 + pinned)
    s = synth.LAGUNA
    lens, qs = [130, 1000, 64, 5000], [3, 17, 1, 9]      # blocks crossing chunk boundaries, ragged
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    cu_chunks, soc, sk, sv, pk, pv, kn, vn = full_case(rng, s, lens, qs)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=4, max_queries_per_seq=17, device=0)
    hk, hv = tensor(sk, pin=pinned) if pinned else tensor(sk), tensor(sv, pin=pinned) if pinned else tensor(sv)
    dk, dv = tensor(pk), tensor(pv)
    vfy.vfy_append_full(ctx, tensor(kn), tensor(vn), i32(cu_q), i32(lens), i32(cu_chunks), i32(soc), hk, hv,
                        sk.shape[0], dk, dv, pk.shape[0], len(lens))
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    ek, ev, epk, epv = O.append_full(kn, vn, cu_q, lens, cu_chunks, soc, sk, sv, pk, pv)
    assert np.array_equal(bits(hk), ek) and np.array_equal(bits(hv), ev)
    assert np.array_equal(bits(dk), epk) and np.array_equal(bits(dv), epv)


def test_append_swa_bit_exact(vfy):
    rng = np.random.default_rng(95)
    s = synth.LAGUNA
    lens, qs = [9000, 40, 3000], [17, 5, 12]
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    phis = [synth.wrapping_ring_offset(rng, L, q, synth.RING) if L > q else 3 for L, q in zip(lens, qs)]
    phis[2] = -7                                          # taken mod R
    ring_shape = (len(lens), s.num_kv_heads, synth.RING, s.head_dim)
    kr, vr = synth.normal_bf16(rng, ring_shape), synth.normal_bf16(rng, ring_shape)
    T = int(cu_q[-1])
    kn = synth.normal_bf16(rng, (T, s.num_kv_heads, s.head_dim))
    vn = synth.normal_bf16(rng, (T, s.num_kv_heads, s.head_dim))
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=3, max_queries_per_seq=17, device=0)
    dk, dv = tensor(kr), tensor(vr)
    vfy.vfy_append_swa(ctx, tensor(kn), tensor(vn), i32(cu_q), i32(lens), i32(phis), dk, dv, len(lens))
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    ek, ev = O.append_ring(kn, vn, cu_q, lens, phis, kr, vr)
    assert np.array_equal(bits(dk), ek) and np.array_equal(bits(dv), ev)


def test_append_full_bad_chunk_is_reported(vfy):
    rng = np.random.default_rng(96)
    s = synth.LAGUNA
    cu_chunks, soc, sk, sv, pk, pv, kn, vn = full_case(rng, s, [500], [17])
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=1, max_queries_per_seq=17, device=0)
    hk, hv, dk, dv = tensor(sk), tensor(sv), tensor(pk), tensor(pv)
    # the store is declared one chunk shorter than the block's last chunk needs
    vfy.vfy_append_full(ctx, tensor(kn), tensor(vn), i32([0, 17]), i32([500]), i32(cu_chunks), i32(soc), hk, hv,
                        sk.shape[0] - 1, dk, dv, pk.shape[0], 1)
    assert vfy.vfy_get_status(ctx) == vfy.VFY_EDEVICE_INPUT


def test_append_full_rejects_pageable_store(vfy):
    rng = np.random.default_rng(97)
    s = synth.LAGUNA
    cu_chunks, soc, sk, sv, pk, pv, kn, vn = full_case(rng, s, [300], [5])
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=1, max_queries_per_seq=17, device=0)
    pageable = torch.from_numpy(sk.view(np.int16)).view(torch.bfloat16)
    with pytest.raises(vfy.VfyError):
        vfy.vfy_append_full(ctx, tensor(kn), tensor(vn), i32([0, 5]), i32([300]), i32(cu_chunks), i32(soc),
                            pageable, pageable, sk.shape[0], tensor(pk), tensor(pv), pk.shape[0], 1)


def test_append_then_attend_in_one_graph(vfy):
    """The block's K/V rows are written by the append and read by the attention of the same
    captured graph, for one full layer and one window layer."""
    rng = np.random.default_rng(98)
    s = synth.LAGUNA
    L, q = 2000, 17
    cu_chunks, soc, sk, sv, pk, pv, kn, vn = full_case(rng, s, [L], [q])
    # the pool holds every chunk in this case, so the attention sees the whole context
    n = sk.shape[0]
    soc = rng.permutation(n).astype(np.int32)
    pk = np.zeros((n,) + sk.shape[1:], np.uint16)
    pv = np.zeros_like(pk)
    pk[soc], pv[soc] = sk, sv
    ring_shape = (1, s.num_kv_heads, synth.RING, s.head_dim)
    kr, vr = synth.normal_bf16(rng, ring_shape), synth.normal_bf16(rng, ring_shape)
    phi = synth.wrapping_ring_offset(rng, L, synth.WINDOW + q - 1, synth.RING)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=1, max_queries_per_seq=q, device=0)
    hk, hv = tensor(sk, pin=True), tensor(sv, pin=True)
    dk, dv, rk, rv = tensor(pk), tensor(pv), tensor(kr), tensor(vr)
    knt, vnt, qt = tensor(kn), tensor(vn), tensor(qb)
    cu_q, lens, cuc, socd = i32([0, q]), i32([L]), i32(cu_chunks), i32(soc)
    ids, slots_t, cu_res = i32(np.arange(n)), i32(soc), i32([0, n])
    phid = i32([phi])
    of, lf = torch.empty_like(qt), torch.empty((q, s.num_q_heads), dtype=torch.float32, device="cuda")
    ow, lw = torch.empty_like(qt), torch.empty((q, s.num_q_heads), dtype=torch.float32, device="cuda")

    def step():
        vfy.vfy_append_full(ctx, knt, vnt, cu_q, lens, cuc, socd, hk, hv, n, dk, dv, n, 1)
        vfy.vfy_attend_full(ctx, qt, cu_q, dk, dv, n, ids, slots_t, cu_res, n, lens, of, lf, 1)
        vfy.vfy_append_swa(ctx, knt, vnt, cu_q, lens, phid, rk, rv, 1)
        vfy.vfy_attend_swa(ctx, qt, cu_q, rk, rv, phid, lens, ow, lw, 1)

    step()                                               # eager once (kernel attributes)
    torch.cuda.synchronize()
    dk.copy_(tensor(pk)); dv.copy_(tensor(pv)); rk.copy_(tensor(kr)); rv.copy_(tensor(vr))
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            step()
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    _, _, epk, epv = O.append_full(kn, vn, [0, q], [L], cu_chunks, soc, sk, sv, pk, pv)
    ekr, evr = O.append_ring(kn, vn, [0, q], [L], [phi], kr, vr)
    ref, rlse = O.attend_full_seq(qb, epk, epv, np.arange(n), soc, L)
    assert_attn_close(bits(of), ref, "append + full")
    assert_lse_close(lf.cpu().numpy(), rlse, "append + full")
    ref, rlse = O.attend_ring_seq(qb, ekr[0], evr[0], phi, L, synth.WINDOW)
    assert_attn_close(bits(ow), ref, "append + window")
    assert_lse_close(lw.cpu().numpy(), rlse, "append + window")
