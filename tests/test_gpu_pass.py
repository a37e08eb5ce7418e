"""The 40-layer verify pass at full size, in the launch configuration bench.py times (one CUDA
graph: residency top-128 of 4096 chunks, 16 page-ins per full layer from pinned host memory,
30 window layers and 10 full layers at 256K context, greedy acceptance over 17 x 131072 logits),
checked against the oracle after replays:
  * residency ids, slots, slot map and page-in list: bit-exact against the oracle's selection
    replayed over every step the device has run (from an empty pool);
  * every resident pool slot of every full layer holds its host chunk byte for byte;
  * every layer (10 full, 30 window), every output row and its LSE, within the attention
    tolerance; the full layers attend the oracle's own resident list, read from the host store;
  * acceptance: bit-exact.
The same checks follow the pass variant that appends the block's K/V rows in every layer and
the end-to-end step whose inputs come from pinned host memory. Also the all-resident 256K full
layer (4096 chunks, 512 MiB of KV) on sampled rows.

The oracle runs in a process pool ("spawn", so that no child inherits the CUDA context)."""
import concurrent.futures as cf
import multiprocessing as mp
import os

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
def oracle_pool():
    ex = cf.ProcessPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)),
                                mp_context=mp.get_context("spawn"))
    yield ex
    ex.shutdown()


@pytest.fixture(scope="module")
def pass256k():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import passes
    torch.cuda.set_device(0)
    vp = passes.VerifyPass(synth.workload_256k(), device=0, seed=3)
    # every residency score vector the device's selection has consumed, in order
    vp.history = [vp.score_table[vp.step % vp.score_table.shape[0]].cpu().numpy()]
    vp.capture()                           # one eager pass (step 0), then the capture
    for _ in range(3):                     # steady state: 16 new chunks per step
        replay_step(vp, vp.graph)
    torch.cuda.synchronize()
    yield vp
    vp.close()


def replay_step(vp, graph):
    """Load the next step's scores, record them in the history, replay `graph`."""
    vp.history.append(vp.score_table[vp.step % vp.score_table.shape[0]].cpu().numpy())
    vp.set_step_scores(vp.step)
    vp.step += 1
    graph.replay()


def oracle_residency(vp):
    """The oracle's residency after every step in vp.history, starting from an empty pool."""
    soc = np.full(vp.n_chunks, -1, dtype=np.int64)
    ref = None
    for sc in vp.history:
        ref = O.select_resident(sc, [0, vp.n_chunks], vp.k, soc)
        soc = ref["slot_of_chunk"]
    return ref


def check_residency(vp, ref):
    assert np.array_equal(vp.res_ids.cpu().numpy(), ref["resident_ids"])
    assert np.array_equal(vp.res_slots.cpu().numpy(), ref["resident_slots"])
    assert np.array_equal(vp.slot_of_chunk.cpu().numpy(), ref["slot_of_chunk"])


def check_pools(vp, ref):
    """Every full layer: each resident slot holds its host chunk, K and V, bit for bit."""
    ids, slots = ref["resident_ids"], ref["resident_slots"]
    for l in vp.full_layers:
        pk, pv = bits(vp.pool_k[l]), bits(vp.pool_v[l])
        hk, hv = bits(vp.host_k[l]), bits(vp.host_v[l])
        assert pk[slots].tobytes() == hk[ids].tobytes(), f"K pool of full layer {l}"
        assert pv[slots].tobytes() == hv[ids].tobytes(), f"V pool of full layer {l}"


def check_all_layers(vp, ex, ref, q_bits=None, what=""):
    """Every layer's output rows and LSE against the oracle. Full layers: the oracle gathers the
    oracle-selected chunks from the host store (laid out as a pool of len(ids) slots), so the
    device's residency lists and pool take no part in the expected values."""
    ids = ref["resident_ids"]
    phi = int(vp.ring_offset.item())
    futs = {}
    for l in range(vp.n_layers):
        qb = q_bits[l] if q_bits is not None else bits(vp.qs[l])
        if l in vp.full_layers:
            hk, hv = bits(vp.host_k[l]), bits(vp.host_v[l])
            futs[l] = ex.submit(O.attend_full_seq, qb, hk[ids], hv[ids], ids, np.arange(len(ids)), vp.L)
        else:
            futs[l] = ex.submit(O.attend_ring_seq, qb, bits(vp.ring_k[l])[0], bits(vp.ring_v[l])[0], phi, vp.L,
                                synth.WINDOW)
    outs = bits(vp.out_all)
    lses = vp.lse_all.cpu().numpy()
    for l in range(vp.n_layers):
        kind = "full" if l in vp.full_layers else "window"
        o_ref, lse_ref = futs[l].result()
        assert_attn_close(outs[l], o_ref, f"{what}{kind} layer {l}")
        assert_lse_close(lses[l], lse_ref, f"{what}{kind} layer {l}")


def test_pass_residency_and_page_in(pass256k):
    vp = pass256k
    replay_step(vp, vp.graph)
    torch.cuda.synchronize()
    ref = oracle_residency(vp)
    check_residency(vp, ref)
    cnt = int(vp.pagein_count.item())
    assert cnt == 16
    assert vp.pagein_list.cpu().numpy()[:cnt].tolist() == [list(x) for x in ref["pagein"][0]]
    check_pools(vp, ref)


def test_pass_every_layer_and_accept(pass256k, oracle_pool):
    """After a replay: all 40 layers (every row of O and LSE), every full layer's pool and the
    acceptance against the oracle."""
    vp = pass256k
    torch.cuda.synchronize()
    ref = oracle_residency(vp)
    check_residency(vp, ref)
    check_pools(vp, ref)
    check_all_layers(vp, oracle_pool, ref)
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


def test_pass_with_block_kv_append(pass256k, oracle_pool):
    """The pass variant that appends the block's K/V rows in every layer before attending (full
    layers write through to the pinned chunk store): after one replay, the block rows of every
    full layer's pool and chunk store and of every window layer's ring are the oracle's, bit for
    bit, and every layer's output matches the oracle on the updated data."""
    vp = pass256k
    # capture() runs the append pass once eagerly (with the current step's scores) before
    # capturing it; appending the same rows again is idempotent
    vp.history.append(vp.score_table[vp.step % vp.score_table.shape[0]].cpu().numpy())
    g = vp.capture(append=True)
    before = {l: (bits(vp.ring_k[l]).copy(), bits(vp.ring_v[l]).copy()) for l in vp.swa_layers}
    before.update({l: (bits(vp.host_k[l]).copy(), bits(vp.host_v[l]).copy(), bits(vp.pool_k[l]).copy(),
                       bits(vp.pool_v[l]).copy()) for l in vp.full_layers})
    replay_step(vp, g)
    torch.cuda.synchronize()
    ref = oracle_residency(vp)
    check_residency(vp, ref)
    soc = ref["slot_of_chunk"]
    cu_q, lens, phi = [0, vp.q], [vp.L], [int(vp.ring_offset.item())]
    for l in vp.full_layers:
        hk, hv, pk, pv = before[l]
        ek, ev, epk, epv = O.append_full(bits(vp.kv_new[l, 0]), bits(vp.kv_new[l, 1]), cu_q, lens,
                                         [0, vp.n_chunks], soc, hk, hv, pk, pv)
        assert np.array_equal(bits(vp.host_k[l]), ek) and np.array_equal(bits(vp.host_v[l]), ev), f"store {l}"
        # the pool: the block rows of resident chunks as the oracle writes them, every resident
        # slot equal to its (updated) host chunk
        got_pk, got_pv = bits(vp.pool_k[l]), bits(vp.pool_v[l])
        ids, slots = ref["resident_ids"], ref["resident_slots"]
        assert got_pk[slots].tobytes() == ek[ids].tobytes(), f"K pool of full layer {l}"
        assert got_pv[slots].tobytes() == ev[ids].tobytes(), f"V pool of full layer {l}"
    for l in vp.swa_layers:
        kr, vr = before[l]
        ekr, evr = O.append_ring(bits(vp.kv_new[l, 0]), bits(vp.kv_new[l, 1]), cu_q, lens, phi, kr, vr)
        assert np.array_equal(bits(vp.ring_k[l]), ekr) and np.array_equal(bits(vp.ring_v[l]), evr), f"ring {l}"
    check_all_layers(vp, oracle_pool, ref, what="with append: ")
    assert vp.kernels_per_pass_append == vp.launches_per_step() + vp.n_layers


def test_pass_end_to_end_from_host(pass256k, oracle_pool):
    """The end-to-end step (VerifyPass.enqueue_end_to_end, captured as one graph): the step's
    inputs are copied from pinned host memory, the later layers' queries and the logits on
    other streams while the first layers run, and the results come back to pinned host memory.
    With new queries, logits and drafts placed only in the host image, one replay must leave the
    device inputs equal to that image, produce the oracle's output in every layer (queries that
    came with the first copy and on the copy stream alike), leave the oracle's residency and
    pools, and return the oracle's acceptance on the new logits."""
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
    vp.history.append(sc.numpy().copy())
    vp.step += 1
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(vp.inputs.cpu(), in_host)
    n, b, c = O.accept(logits, drafts, [0, vp.q])
    got = out_host.numpy()
    assert int(got[0]) == int(n[0]) and int(got[1]) == int(b[0])
    assert got[2:].tolist() == c.tolist()
    ref = oracle_residency(vp)
    check_residency(vp, ref)
    check_pools(vp, ref)
    qbits = q_new.view(torch.int16).numpy().view(np.uint16)
    check_all_layers(vp, oracle_pool, ref, q_bits=qbits, what="end to end: ")
