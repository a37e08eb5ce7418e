"""The ragged-batch workload at full size: 8 sequences with contexts drawn on [4000, 200000] and
draft depths drawn from {2, 4, 8, 11, 16} (`synth.workload_ragged(0)`; 'Width vs. Depth:
Speculating on the Margin', ragged speculation), 16 q-heads / 4 KV heads x 128. Each step runs for
the whole batch in one call, as a pass over this workload would:
  * one global layer with every chunk of every sequence resident in shuffled slots (about 1.6 GB
    of K+V; its splits hold far more than 8 chunks, so it streams two-chunk tiles): checked on
    sampled rows of every sequence;
  * one window layer (512-token window of 2048-slot rings, per-sequence write-head offsets that
    wrap): checked on every row;
  * greedy acceptance over (D_b + 1) x 131072 fp32 logits per sequence: bit-exact.
"""
import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

from gpu_util import assert_attn_close, assert_lse_close

pytestmark = pytest.mark.gpu

C = 64


def bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(scope="module")
def batch():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import vfy
    torch.cuda.set_device(0)
    w = synth.workload_ragged(0)
    s = w.shape
    qs = w.queries
    cu_q = np.concatenate([[0], np.cumsum(qs)]).astype(np.int32)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=w.num_seqs,
                         max_queries_per_seq=max(qs), device=0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4)
    q = torch.randn((int(cu_q[-1]), s.num_q_heads, s.head_dim), generator=gen, device="cuda",
                    dtype=torch.bfloat16)
    yield w, ctx, q, cu_q, gen, vfy
    ctx.close()


def test_ragged_global_layer_all_resident(batch):
    w, ctx, q, cu_q, gen, vfy = batch
    s = w.shape
    rng = np.random.default_rng(7)
    n_per = [(L + C - 1) // C for L in w.seq_lens]
    total = sum(n_per)
    kp = torch.randn((total, s.num_kv_heads, C, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    vp = torch.randn_like(kp)
    perm = rng.permutation(total).astype(np.int32)
    ids, slots, cu_res = [], [], [0]
    off = 0
    for n in n_per:
        ids.append(np.arange(n, dtype=np.int32))
        slots.append(perm[off:off + n])
        off += n
        cu_res.append(off)
    dev = lambda a: torch.tensor(np.concatenate(a) if isinstance(a, list) else a, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    vfy.vfy_attend_full(ctx, q, dev(cu_q), kp, vp, total, dev(ids), dev(slots), dev(np.array(cu_res)),
                        max(n_per), dev(np.array(w.seq_lens)), out, lse, w.num_seqs)
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    got, glse = bits(out), lse.cpu().numpy()
    for b in range(w.num_seqs):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        nq = e - a
        rows = [(0, 0), (nq - 1, s.num_q_heads - 1), (nq // 2, 7)]
        sl = torch.tensor(slots[b], dtype=torch.long, device="cuda")
        kb, vb = bits(kp.index_select(0, sl)), bits(vp.index_select(0, sl))
        ref, rlse = O.attend_full_seq(bits(q[a:e]), kb, vb, ids[b], np.arange(n_per[b]), w.seq_lens[b], rows=rows)
        for i, g in rows:
            assert_attn_close(got[a + i, g], ref[i, g], f"seq {b} row {i},{g}")
            assert abs(glse[a + i, g] - rlse[i, g]) <= 2e-3 + 1e-3 * abs(rlse[i, g]), f"seq {b} lse {i},{g}"


def test_ragged_window_layer(batch):
    w, ctx, q, cu_q, gen, vfy = batch
    s = w.shape
    rng = np.random.default_rng(8)
    R = synth.RING
    kr = torch.randn((w.num_seqs, s.num_kv_heads, R, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    vr = torch.randn_like(kr)
    phis = [synth.wrapping_ring_offset(rng, L, synth.WINDOW + qn - 1, R) for L, qn in zip(w.seq_lens, w.queries)]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    vfy.vfy_attend_swa(ctx, q, i32(cu_q), kr, vr, i32(phis), i32(w.seq_lens), out, lse, w.num_seqs)
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    ref, rlse = O.attend_ring(bits(q), cu_q, bits(kr), bits(vr), phis, w.seq_lens, synth.WINDOW)
    assert_attn_close(bits(out), ref, "ragged window")
    assert_lse_close(lse.cpu().numpy(), rlse, "ragged window")


def test_ragged_acceptance_full_vocab(batch):
    w, ctx, q, cu_q, gen, vfy = batch
    rng = np.random.default_rng(9)
    rows = w.queries
    cu_rows = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    logits, drafts = [], []
    for d in w.depths:
        targets = rng.integers(0, w.vocab, d + 1)
        logits.append(synth.planted_logits(rng, targets, w.vocab))
        drafts.append(synth.drafts_matching(rng, targets, 0.56, w.vocab))
    logits = np.concatenate(logits)
    drafts = np.concatenate(drafts).astype(np.int32)
    lg = torch.from_numpy(logits).cuda()
    acc = torch.zeros(w.num_seqs, dtype=torch.int32, device="cuda")
    bonus = torch.zeros_like(acc)
    committed = torch.zeros(int(cu_rows[-1]), dtype=torch.int32, device="cuda")
    vfy.vfy_accept(ctx, lg, w.vocab, torch.from_numpy(drafts).cuda(), torch.from_numpy(cu_rows).cuda(),
                   int(cu_rows[-1]), acc, bonus, committed, w.num_seqs)
    torch.cuda.synchronize()
    assert vfy.vfy_get_status(ctx) == vfy.VFY_OK
    n, b, c = O.accept(logits, drafts, cu_rows)
    assert acc.cpu().numpy().tolist() == [int(x) for x in n]
    assert bonus.cpu().numpy().tolist() == [int(x) for x in b]
    assert committed.cpu().numpy().tolist() == [int(x) for x in c]
