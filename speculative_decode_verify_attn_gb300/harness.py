"""Host-side plumbing around the binding: numpy <-> device tensors, output allocation, and one
call per step. It holds none of the verify step's arithmetic; every result comes from libvfy."""
from __future__ import annotations

import numpy as np
import torch

from . import vfy


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> a bf16 device tensor with the same bytes."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def host_bf16(bits: np.ndarray, pinned: bool = True) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def dev_f32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def cu_from_counts(counts) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(counts, dtype=np.int64))]).astype(np.int32)


def attend_full(ctx, q_bits, cu_q, k_pool_bits, v_pool_bits, resident_ids, resident_slots, cu_resident,
                seq_len, device="cuda", with_lse=True):
    q = dev_bf16(q_bits, device)
    kp, vp = dev_bf16(k_pool_bits, device), dev_bf16(v_pool_bits, device)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=device) if with_lse else None
    cu_res = np.asarray(cu_resident)
    max_res = int(np.max(np.diff(cu_res))) if len(cu_res) > 1 else 0
    vfy.vfy_attend_full(ctx, q, dev_i32(cu_q, device), kp, vp, kp.shape[0], dev_i32(resident_ids, device),
                        dev_i32(resident_slots, device), dev_i32(cu_res, device), max_res,
                        dev_i32(seq_len, device), out, lse, len(cu_q) - 1)
    torch.cuda.synchronize()
    return bits_of(out), (lse.cpu().numpy() if with_lse else None)


def attend_swa(ctx, q_bits, cu_q, k_ring_bits, v_ring_bits, ring_offset, seq_len, device="cuda", with_lse=True):
    q = dev_bf16(q_bits, device)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=device) if with_lse else None
    vfy.vfy_attend_swa(ctx, q, dev_i32(cu_q, device), dev_bf16(k_ring_bits, device), dev_bf16(v_ring_bits, device),
                       dev_i32(ring_offset, device), dev_i32(seq_len, device), out, lse, len(cu_q) - 1)
    torch.cuda.synchronize()
    return bits_of(out), (lse.cpu().numpy() if with_lse else None)


def accept(ctx, logits, drafts, cu_rows, device="cuda"):
    cu_rows = np.asarray(cu_rows, dtype=np.int32)
    B = len(cu_rows) - 1
    rows = int(cu_rows[-1])
    acc = torch.full((B,), -7, dtype=torch.int32, device=device)
    bonus = torch.full((B,), -7, dtype=torch.int32, device=device)
    committed = torch.full((rows,), -7, dtype=torch.int32, device=device)
    d = dev_i32(drafts if len(drafts) else np.zeros(1, np.int32), device)
    vfy.vfy_accept(ctx, dev_f32(logits, device), int(np.asarray(logits).shape[1]), d, dev_i32(cu_rows, device),
                   rows, acc, bonus, committed, B)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), bonus.cpu().numpy(), committed.cpu().numpy()


def select_resident(ctx, scores, cu_chunks, k, slot_of_chunk, device="cuda"):
    cu_chunks = np.asarray(cu_chunks, dtype=np.int32)
    B = len(cu_chunks) - 1
    n_max = int(np.max(np.diff(cu_chunks)))
    total = sum(min(k, int(n)) for n in np.diff(cu_chunks))
    ids = torch.full((max(total, 1),), -7, dtype=torch.int32, device=device)
    slots = torch.full((max(total, 1),), -7, dtype=torch.int32, device=device)
    cu_res = torch.full((B + 1,), -7, dtype=torch.int32, device=device)
    plist = torch.full((B * k, 2), -7, dtype=torch.int32, device=device)
    pcount = torch.full((B,), -7, dtype=torch.int32, device=device)
    som = dev_i32(slot_of_chunk, device)
    vfy.vfy_select_resident(ctx, dev_f32(scores, device), dev_i32(cu_chunks, device), B, n_max, k, som,
                            ids, slots, cu_res, plist, pcount)
    torch.cuda.synchronize()
    return {"resident_ids": ids.cpu().numpy()[:total], "resident_slots": slots.cpu().numpy()[:total],
            "cu_resident": cu_res.cpu().numpy(), "pagein_list": plist.cpu().numpy(),
            "pagein_count": pcount.cpu().numpy(), "slot_of_chunk": som.cpu().numpy()}
