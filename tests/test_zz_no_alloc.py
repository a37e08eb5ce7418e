"""vfy_accept_static, the acceptance entry point for callers that cannot allocate device memory
(it needs no context; its scratch is a fixed array in the library), must give the same accepted
lengths, bonus tokens and committed tokens as vfy_accept, call after call. This file is named so
that pytest collects it last."""
import numpy as np
import pytest
import torch

from oracle import vfy_oracle as O
from speculative_decode_verify_attn_gb300 import synth

pytestmark = pytest.mark.gpu


def test_static_accept_matches_vfy_accept_on_two_calls_in_a_row():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import harness as H
    from speculative_decode_verify_attn_gb300 import vfy
    torch.cuda.set_device(0)
    ctx = vfy.vfy_create(16, 4, 128, max_seqs=8, max_queries_per_seq=17, device=0)
    rng = np.random.default_rng(11)
    V = synth.VOCAB
    depths = [16, 2, 11, 4, 8, 0, 16, 2]
    cu = np.concatenate([[0], np.cumsum([d + 1 for d in depths])]).astype(np.int32)
    rows = int(cu[-1])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        for call in range(2):
            targets = rng.integers(0, V, rows)
            logits = synth.planted_logits(rng, targets, V)
            drafts = np.concatenate([synth.drafts_matching(rng, targets[cu[b]:cu[b + 1]], 0.56, V)
                                     for b in range(len(depths))]).astype(np.int32)
            ref_n, ref_b, ref_c = H.accept(ctx, logits, drafts, cu)
            lg, dr, cr = H.dev_f32(logits), H.dev_i32(drafts), H.dev_i32(cu)
            n = torch.full((len(depths),), -7, dtype=torch.int32, device="cuda")
            b = torch.full_like(n, -7)
            c = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
            vfy.vfy_accept_static(lg, V, dr, cr, len(depths), rows, n, b, c, err)
            torch.cuda.synchronize()
            assert n.cpu().numpy().tolist() == ref_n.tolist()
            assert b.cpu().numpy().tolist() == ref_b.tolist()
            assert c.cpu().numpy().tolist() == ref_c.tolist()
            on, ob, oc = O.accept(logits, drafts, cu)
            assert ref_n.tolist() == on.tolist() and ref_c.tolist() == oc.tolist()
        assert int(err.item()) == 0
        with pytest.raises(vfy.VfyError) as e:          # beyond the fixed scratch
            vfy.vfy_accept_static(lg, V, dr, cr, len(depths), 1025, n, b, c, err)
        assert e.value.status == vfy.VFY_EINVAL
    finally:
        ctx.close()


def _static_env():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decode_verify_attn_gb300 import harness as H
    from speculative_decode_verify_attn_gb300 import vfy
    torch.cuda.set_device(0)
    return H, vfy


def _batch(rng, depths, vocab):
    cu = np.concatenate([[0], np.cumsum([d + 1 for d in depths])]).astype(np.int32)
    rows = int(cu[-1])
    targets = rng.integers(0, vocab, rows)
    logits = synth.planted_logits(rng, targets, vocab)
    drafts = np.concatenate([synth.drafts_matching(rng, targets[cu[b]:cu[b + 1]], 0.56, vocab)
                             for b in range(len(depths))]).astype(np.int32)
    return cu, logits, drafts


def test_static_accept_at_its_row_limit_and_on_a_second_stream():
    """All 1024 rows of the fixed scratch in use (60 sequences of depth 16 and one of depth 3),
    compared with vfy_accept; then a call on a second stream, ordered after the first by an
    event, which must see the scratch cleared by its own call."""
    H, vfy = _static_env()
    rng = np.random.default_rng(12)
    V = 4096
    depths = [16] * 60 + [3]
    ctx = vfy.vfy_create(16, 4, 128, max_seqs=len(depths), max_queries_per_seq=17, device=0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        cu, logits, drafts = _batch(rng, depths, V)
        rows = int(cu[-1])
        assert rows == 1024
        ref_n, ref_b, ref_c = H.accept(ctx, logits, drafts, cu)
        lg, dr, cr = H.dev_f32(logits), H.dev_i32(drafts), H.dev_i32(cu)
        out = [(torch.full((len(depths),), -7, dtype=torch.int32, device="cuda"),
                torch.full((len(depths),), -7, dtype=torch.int32, device="cuda"),
                torch.full((rows,), -7, dtype=torch.int32, device="cuda")) for _ in range(2)]
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        ev = torch.cuda.Event()
        torch.cuda.synchronize()
        vfy.vfy_accept_static(lg, V, dr, cr, len(depths), rows, *out[0], err, stream=s1)
        ev.record(s1)
        s2.wait_event(ev)                 # the documented ordering: calls must not overlap
        vfy.vfy_accept_static(lg, V, dr, cr, len(depths), rows, *out[1], err, stream=s2)
        torch.cuda.synchronize()
        for n, b, c in out:
            assert n.cpu().numpy().tolist() == ref_n.tolist()
            assert b.cpu().numpy().tolist() == ref_b.tolist()
            assert c.cpu().numpy().tolist() == ref_c.tolist()
        assert int(err.item()) == 0
    finally:
        ctx.close()


def test_static_accept_reports_a_bad_row_list_in_the_callers_word():
    """cu_rows[B] beyond max_rows: the sequences that fit are accepted as usual, the others are
    skipped, and error bit 1 lands in the caller's device word."""
    H, vfy = _static_env()
    rng = np.random.default_rng(13)
    V = 2048
    depths = [16, 16]
    cu, logits, drafts = _batch(rng, depths, V)
    max_rows = 20                                     # the second sequence ends at row 34
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    b = torch.full_like(n, -7)
    c = torch.full((int(cu[-1]),), -7, dtype=torch.int32, device="cuda")
    vfy.vfy_accept_static(H.dev_f32(logits), V, H.dev_i32(drafts), H.dev_i32(cu), 2, max_rows, n, b, c, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    on, ob, oc = O.accept(logits[:17], drafts[:16], [0, 17])
    assert int(n[0].item()) == int(on[0]) and int(b[0].item()) == int(ob[0])
    assert c[:17].cpu().numpy().tolist() == oc.tolist()
