"""The 40-layer verify pass at full size, in the launch configuration bench.py times (one CUDA
graph: residency top-128 of 4096 chunks, 16 page-ins per full layer from pinned host memory,
30 window layers and 10 full layers at 256K context, greedy acceptance over 17 x 131072 logits),
checked against the oracle after a replay:
  * residency ids, slots, slot map and page-in list: bit-exact;
  * every resident pool slot of a full layer holds its host chunk byte for byte;
  * one full layer and one window layer: every output row, within the attention tolerance;
  * acceptance: bit-exact.
Also the all-resident 256K full layer (4096 chunks, 512 MiB of KV) on sampled rows."""
import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu


def bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def pass256k():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import passes
    torch.cuda.set_device(0)
    vp = passes.VerifyPass(synth.workload_256k(), device=0, seed=3)
    vp.capture()
    for _ in range(3):                     # steady state: 16 new chunks per step
        vp.set_step_scores(vp.step)
        vp.step += 1
        vp.replay()
    torch.cuda.synchronize()
    yield vp
    vp.close()


def test_pass_residency_and_page_in(pass256k):
    vp = pass256k
    prev = vp.slot_of_chunk.cpu().numpy().copy()
    scores = vp.score_table[vp.step % vp.score_table.shape[0]].cpu().numpy()
    vp.set_step_scores(vp.step)
    vp.step += 1
    vp.replay()
    torch.cuda.synchronize()
    ref = O.select_resident(scores, [0, vp.n_chunks], vp.k, prev)
    assert np.array_equal(vp.res_ids.cpu().numpy(), ref["resident_ids"])
    assert np.array_equal(vp.res_slots.cpu().numpy(), ref["resident_slots"])
    assert np.array_equal(vp.slot_of_chunk.cpu().numpy(), ref["slot_of_chunk"])
    cnt = int(vp.pagein_count.item())
    assert cnt == 16
    assert vp.pagein_list.cpu().numpy()[:cnt].tolist() == [list(x) for x in ref["pagein"][0]]
    # every resident slot of a full layer holds its chunk, bit for bit
    l = vp.full_layers[-1]
    pk, pv = bits(vp.pool_k[l]), bits(vp.pool_v[l])
    hk, hv = bits(vp.host_k[l]), bits(vp.host_v[l])
    ids, slots = ref["resident_ids"], ref["resident_slots"]
    assert pk[slots].tobytes() == hk[ids].tobytes()
    assert pv[slots].tobytes() == hv[ids].tobytes()


def test_pass_layers_and_accept(pass256k):
    vp = pass256k
    torch.cuda.synchronize()
    ids = vp.res_ids.cpu().numpy()
    slots = vp.res_slots.cpu().numpy()
    # a full layer
    l = vp.full_layers[1]
    ref, rlse = O.attend_full_seq(bits(vp.qs[l]), bits(vp.pool_k[l]), bits(vp.pool_v[l]), ids, slots, vp.L)
    assert_attn_close(bits(vp.outs[l]), ref, f"full layer {l}")
    assert_lse_close(vp.lses[l].cpu().numpy(), rlse, f"full layer {l}")
    # a window layer
    l = vp.swa_layers[5]
    ref, rlse = O.attend_ring_seq(bits(vp.qs[l]), bits(vp.ring_k[l])[0], bits(vp.ring_v[l])[0],
                                  int(vp.ring_offset.item()), vp.L, synth.WINDOW)
    assert_attn_close(bits(vp.outs[l]), ref, f"window layer {l}")
    assert_lse_close(vp.lses[l].cpu().numpy(), rlse, f"window layer {l}")
    # acceptance
    n, b, c = O.accept(vp.logits.cpu().numpy(), vp.drafts.cpu().numpy(), [0, vp.q])
    assert int(vp.accepted.item()) == int(n[0]) and int(vp.bonus.item()) == int(b[0])
    assert vp.committed.cpu().numpy().tolist() == c.tolist()


def test_all_resident_256k_layer_sampled():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import passes
    wl = synth.Workload("all-resident", synth.LAGUNA, [262144], [16], n_full=1, n_swa=3, resident_chunks=0)
    ar = passes.VerifyPass(wl, device=0, seed=5, all_resident=True)
    try:
        l = ar.full_layers[0]
        ar.attend_full_layer(l)
        torch.cuda.synchronize()
        rows = [(0, 0), (3, 5), (8, 10), (16, 15), (16, 0), (11, 7)]
        ref, rlse = O.attend_full_seq(bits(ar.qs[l]), bits(ar.pool_k[l]), bits(ar.pool_v[l]),
                                      np.arange(ar.k), np.arange(ar.k), ar.L, rows=rows)
        got = bits(ar.outs[l])
        glse = ar.lses[l].cpu().numpy()
        for i, g in rows:
            assert_attn_close(got[i, g], ref[i, g], f"row {i},{g}")
            assert abs(glse[i, g] - rlse[i, g]) <= 2e-3 + 1e-3 * abs(rlse[i, g])
    finally:
        ar.close()


def test_pass_with_block_kv_append(pass256k):
    """The pass variant that appends the block's K/V rows in every layer before attending (full
    layers write through to the pinned chunk store): after one replay, the block rows of a full
    layer's pool and chunk store and of a window layer's ring are the oracle's, bit for bit, and
    both layers' outputs match the oracle on the updated data."""
    vp = pass256k
    g = vp.capture(append=True)
    lf, ls = vp.full_layers[2], vp.swa_layers[7]
    # the state the replay starts from (the capture's eager run already appended once; appending
    # the same rows again is idempotent)
    prev = vp.slot_of_chunk.cpu().numpy().copy()
    scores = vp.score_table[vp.step % vp.score_table.shape[0]].cpu().numpy()
    vp.set_step_scores(vp.step)
    vp.step += 1
    g.replay()
    torch.cuda.synchronize()
    ref_sel = O.select_resident(scores, [0, vp.n_chunks], vp.k, prev)
    soc = ref_sel["slot_of_chunk"]
    kn, vn = bits(vp.kv_new[lf, 0]), bits(vp.kv_new[lf, 1])
    cu_q, lens = [0, vp.q], [vp.L]
    hk, hv, pk, pv = bits(vp.host_k[lf]), bits(vp.host_v[lf]), bits(vp.pool_k[lf]), bits(vp.pool_v[lf])
    ek, ev, epk, epv = O.append_full(kn, vn, cu_q, lens, [0, vp.n_chunks], soc, hk, hv, pk, pv)
    assert np.array_equal(hk, ek) and np.array_equal(hv, ev)       # the rows are already in place
    assert np.array_equal(pk, epk) and np.array_equal(pv, epv)
    ids, slots = ref_sel["resident_ids"], ref_sel["resident_slots"]
    ref, rlse = O.attend_full_seq(bits(vp.qs[lf]), pk, pv, ids, slots, vp.L)
    assert_attn_close(bits(vp.outs[lf]), ref, f"full layer {lf} with append")
    assert_lse_close(vp.lses[lf].cpu().numpy(), rlse, f"full layer {lf} with append")
    kr, vr = bits(vp.ring_k[ls]), bits(vp.ring_v[ls])
    ekr, evr = O.append_ring(bits(vp.kv_new[ls, 0]), bits(vp.kv_new[ls, 1]), cu_q, lens,
                             [int(vp.ring_offset.item())], kr, vr)
    assert np.array_equal(kr, ekr) and np.array_equal(vr, evr)
    ref, rlse = O.attend_ring_seq(bits(vp.qs[ls]), kr[0], vr[0], int(vp.ring_offset.item()), vp.L, synth.WINDOW)
    assert_attn_close(bits(vp.outs[ls]), ref, f"window layer {ls} with append")
    assert_lse_close(vp.lses[ls].cpu().numpy(), rlse, f"window layer {ls} with append")
    assert vp.kernels_per_pass_append == vp.launches_per_step() + vp.n_layers


def test_pass_end_to_end_from_host(pass256k):
    """The end-to-end step (VerifyPass.enqueue_end_to_end, captured as one graph): the step's
    inputs are copied from pinned host memory, the later layers' queries and the logits on a copy
    stream while the first layers run, and the results come back to pinned host memory. With new
    queries, logits and drafts placed only in the host image, one replay must leave the device
    inputs equal to that image, produce the oracle's window-layer outputs for a layer whose
    queries came with the first copy and for one whose queries came on the copy stream, and
    return the oracle's acceptance on the new logits."""
    vp = pass256k
    hq, d = vp.shape.num_q_heads, vp.shape.head_dim
    in_host = vp.inputs.cpu().pin_memory()
    out_host = torch.full((vp.results.numel(),), -7, dtype=torch.int32).pin_memory()
    g = vp.capture_end_to_end(in_host, out_host)
    rng = np.random.default_rng(11)
    gen = torch.Generator().manual_seed(12)
    q_new = torch.randn((vp.n_layers, vp.q, hq, d), generator=gen).to(torch.bfloat16)
    qo = vp.input_offsets["q"]
    in_host[qo:qo + q_new.numel() * 2].copy_(q_new.reshape(-1).view(torch.uint8))
    targets = rng.integers(0, vp.vocab, vp.q)
    logits = synth.planted_logits(rng, targets, vp.vocab)
    drafts = synth.drafts_matching(rng, targets, 0.5, vp.vocab).astype(np.int32)
    lo, do = vp.input_offsets["logits"], vp.input_offsets["drafts"]
    in_host[lo:lo + logits.nbytes].copy_(torch.from_numpy(logits.reshape(-1).view(np.uint8)))
    in_host[do:do + drafts.nbytes].copy_(torch.from_numpy(drafts.view(np.uint8)))
    so = vp.input_offsets["scores"]
    sc = vp.score_table[vp.step % vp.score_table.shape[0]].cpu()
    in_host[so:so + sc.numel() * 4].copy_(sc.view(torch.uint8))
    vp.step += 1
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(vp.inputs.cpu(), in_host)
    n, b, c = O.accept(logits, drafts, [0, vp.q])
    got = out_host.numpy()
    assert int(got[0]) == int(n[0]) and int(got[1]) == int(b[0])
    assert got[2:].tolist() == c.tolist()
    qbits = q_new.view(torch.int16).numpy().view(np.uint16)
    for l in (vp.swa_layers[0], vp.swa_layers[5]):     # layer 0: first copy; layer 6: copy stream
        ref, rlse = O.attend_ring_seq(qbits[l], bits(vp.ring_k[l])[0], bits(vp.ring_v[l])[0],
                                      int(vp.ring_offset.item()), vp.L, synth.WINDOW)
        assert_attn_close(bits(vp.outs[l]), ref, f"window layer {l} end to end")
        assert_lse_close(vp.lses[l].cpu().numpy(), rlse, f"window layer {l} end to end")
