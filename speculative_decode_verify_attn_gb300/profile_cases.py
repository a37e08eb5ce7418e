"""Small, self-contained launches of one kernel family for Nsight Compute captures.

  python -m speculative_decode_verify_attn_gb300.profile_cases CASE [--reps N]

CASE:
  full8k     one full-attention layer of the 256K workload: 128 of 4096 chunks resident (16 MiB)
  prefill    a 1024-query block over the same 128 resident chunks (one split per row tile, which
             writes its own output)
  drafter    one layer of the drafter's context-KV ring (window 4096 in an 8192-slot ring)
  full256k   one full-attention layer with all 4096 chunks resident (512 MiB of KV)
  swa        one window layer (512-token window, 2048-slot ring, wrapping)
  accept     argmax + acceptance over 17 x 131072 fp32 logits
  select     residency top-128 of 4096 chunks
Each repetition writes a 256 MiB buffer first, so the kernel reads HBM, not L2. The device
holds under 1 GiB in every case; the largest is full256k, with 512 MiB of K/V beside the
256 MiB flush buffer.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from speculative_decode_verify_attn_gb300 import build, synth, vfy  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["full8k", "full256k", "swa", "accept", "select", "prefill", "drafter"])
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    build.build()
    torch.cuda.set_device(0)
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    rng = np.random.default_rng(0)
    s = synth.LAGUNA
    q, L = (1024 if a.case == "prefill" else 16 if a.case == "drafter" else 17), 262144
    W, R = (synth.DRAFTER_WINDOW, synth.DRAFTER_RING) if a.case == "drafter" else (synth.WINDOW, synth.RING)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, window=W, ring_len=R, max_queries_per_seq=q,
                         device=0)
    # as in the 40-layer pass: the per-step metadata is set before the kernels run
    vfy.vfy_set_stable_metadata(ctx, True)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    cu_q = torch.tensor([0, q], dtype=torch.int32, device=dev)
    seq_len = torch.tensor([L], dtype=torch.int32, device=dev)
    qt = torch.randn((q, s.num_q_heads, s.head_dim), generator=g, device=dev, dtype=torch.bfloat16)
    out = torch.empty_like(qt)
    lse = torch.empty((q, s.num_q_heads), dtype=torch.float32, device=dev)

    if a.case in ("full8k", "full256k", "prefill"):
        n = 4096 if a.case == "full256k" else 128
        kp = torch.randn((n, s.num_kv_heads, 64, s.head_dim), generator=g, device=dev, dtype=torch.bfloat16)
        vp = torch.randn_like(kp)
        if n == 4096:
            ids = np.arange(n)
        else:
            ids = np.sort(np.concatenate([rng.choice(4095, n - 1, replace=False), [4095]]))
        ids_t = torch.tensor(ids, dtype=torch.int32, device=dev)
        slots_t = torch.tensor(rng.permutation(n), dtype=torch.int32, device=dev)
        cu_res = torch.tensor([0, n], dtype=torch.int32, device=dev)

        def run():
            vfy.vfy_attend_full(ctx, qt, cu_q, kp, vp, n, ids_t, slots_t, cu_res, n, seq_len, out, lse, 1)
    elif a.case in ("swa", "drafter"):
        rk = torch.randn((1, s.num_kv_heads, R, s.head_dim), generator=g, device=dev, dtype=torch.bfloat16)
        rv = torch.randn_like(rk)
        phi = synth.wrapping_ring_offset(rng, L, W + q - 1, R)
        off = torch.tensor([phi], dtype=torch.int32, device=dev)

        def run():
            vfy.vfy_attend_swa(ctx, qt, cu_q, rk, rv, off, seq_len, out, lse, 1)
    elif a.case == "accept":
        targets = rng.integers(0, synth.VOCAB, q)
        logits = torch.from_numpy(synth.planted_logits(rng, targets, synth.VOCAB)).to(dev)
        drafts = torch.from_numpy(synth.drafts_matching(rng, targets, 0.56, synth.VOCAB)).to(dev)
        cu_rows = torch.tensor([0, q], dtype=torch.int32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        bon = torch.empty(1, dtype=torch.int32, device=dev)
        com = torch.empty(q, dtype=torch.int32, device=dev)

        def run():
            vfy.vfy_accept(ctx, logits, synth.VOCAB, drafts, cu_rows, q, acc, bon, com, 1)
    else:
        rot = synth.rotating_residency(rng, 4096, 128, 16, L, q)
        scores = torch.from_numpy(rot.scores(0)).to(dev)
        cu = torch.tensor([0, 4096], dtype=torch.int32, device=dev)
        som = torch.full((4096,), -1, dtype=torch.int32, device=dev)
        ids = torch.empty(128, dtype=torch.int32, device=dev)
        sl = torch.empty(128, dtype=torch.int32, device=dev)
        cur = torch.empty(2, dtype=torch.int32, device=dev)
        pl = torch.empty((128, 2), dtype=torch.int32, device=dev)
        pc = torch.empty(1, dtype=torch.int32, device=dev)

        def run():
            vfy.vfy_select_resident(ctx, scores, cu, 1, 4096, 128, som, ids, sl, cur, pl, pc)

    for _ in range(a.reps):
        flush.zero_()
        run()
    torch.cuda.synchronize()
    st = vfy.vfy_get_status(ctx)
    ctx.close()
    if st != vfy.VFY_OK:
        raise SystemExit(f"device status {vfy.strerror(st)}")
    print(f"{a.case}: {a.reps} reps ok")


if __name__ == "__main__":
    main()
