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
