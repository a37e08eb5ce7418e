"""Oracle for the speculative-decoding verify step: a plain, slow CPU restatement in fp64.

TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the CPU-baseline leg
of bench.py may import or run this module. The CUDA library shares no code with it, and the
product path never calls it.

What it restates, and where the pages say so (cited by page title and section):

[LX] "Laguna XS 2.1 33B on a RTX 3090: 296 tok/s peak, 152 tok/s at 256K context" (lucebox)
     - "The model, fast MoE with a drafter in the box": the target verifies 16 drafted tokens in
       one batched forward and commits only tokens it would itself emit (exact greedy).
     - "Three optimizations", item 1: full-attention layers read a pool of 64-token chunks; a
       resident subset stays on the GPU, chosen from per-chunk residency scores; cold chunks
       are copied from host memory bit-exact.
     - "Three optimizations", item 3: sliding-window layers attend a 512-token window kept in a
       position ring, slot = pos mod 2048.
[CM] "The Death of the Compute-Moat: How Laguna XS 2.1 Shatters the 256K Context Barrier",
     "DFlash Drafters and the End of Speculative Loss": propose 16, verify, commit; the
     conceptual loop's fallback branch (no draft accepted) still commits the target's token.
[WD] "Width vs. Depth: Speculating on the Margin": ragged speculation, a draft depth per
     sequence.

Readings taken where the pages are silent:
  * L (the sequence length) counts the verify block itself; query i of a q-token block sits at
    position L - q + i.
  * Residency is top-k over fp32 scores: higher score first, ties to the lower chunk index,
    -0 equal to +0, NaN below every number (including -inf); k >= n keeps every chunk.
  * Slot reconciliation: sequence b owns pool slots [b*k, b*k + k). A chosen chunk that already
    holds a slot in that range keeps it; the other chosen chunks, in ascending chunk order, take
    the free slots of the range in ascending order; those (chunk, slot) pairs are the page-in
    list. Chunks not chosen lose their slot (-1).
  * Attention: softmax(scale * q.k) over the attended keys, scale = 1/sqrt(head_dim); q-head g
    reads KV head g // G (G = Hq / Hkv). A full layer attends the resident chunks' positions
    p <= p_i (and p < L). A window layer attends positions [max(0, p_i - W + 1), p_i], read from
    ring slot (p + phi) mod R with a per-sequence offset phi (phi = 0 is the page's rule).
    A row with no attended key outputs 0 and LSE = -inf.
  * Acceptance: a_r = argmax of row r (ties to the lowest index; a NaN counts as the maximum,
    first NaN wins). Row r is compared with draft d_r; n = length of the longest matching
    prefix; committed = d_0..d_{n-1}, a_n; bonus = a_n; unused committed entries are -1.

Parity status: every function below is pinned by the CPU tests (tests/test_oracle_*.py) against
brute force, closed forms, library routines or hand-worked cases. None is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

CHUNK_TOKENS = 64  # [LX] "Three optimizations", item 1: 64-token chunks


# --------------------------------------------------------------------------------------------
# Data decoding
# --------------------------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Widen bf16 values, given as their uint16 bit patterns, to float64 exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------------------------
# Small definitions (kept separate so that a test can plant a mistake in exactly one of them)
# --------------------------------------------------------------------------------------------

def _query_position(seq_len: int, num_queries: int, i: int) -> int:
    """Position of block query i: the block is the last `num_queries` positions of the sequence."""
    return seq_len - num_queries + i


def _kv_head_of(q_head: int, group: int) -> int:
    """GQA: q-heads are grouped contiguously, `group` q-heads per KV head."""
    return q_head // group


def _window_start(p: int, window: int) -> int:
    """First position a window query at position p attends: `window` positions including itself."""
    return max(0, p - window + 1)


def _ring_slot(pos: int, phi: int, ring_len: int) -> int:
    """Ring slot of a position: [LX] item 3 gives slot = pos mod 2048; phi shifts the write head."""
    return (pos + phi) % ring_len


def _default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


# --------------------------------------------------------------------------------------------
# a1: residency top-k and slot reconciliation  ([LX] "Three optimizations", item 1)
# --------------------------------------------------------------------------------------------

def rank_chunks(scores) -> list[int]:
    """Chunk indices best-first: score descending, ties to the lower index, NaN after all numbers."""
    scores = np.asarray(scores, dtype=np.float32)

    def key(j):
        s = float(scores[j])
        if math.isnan(s):
            return (1, 0.0, j)
        return (0, -s, j)  # -0.0 == 0.0, so signed zeros tie and fall back to the index

    return sorted(range(len(scores)), key=key)


def select_resident_one(scores, k: int, prev_slot, slot_base: int):
    """Residency for one sequence.

    scores     fp32 [n]   per-chunk residency scores
    k          int        pool slots of this sequence (the resident budget)
    prev_slot  int [n]    slot each chunk held before this step, -1 if not resident
    slot_base  int        first pool slot owned by this sequence

    Returns (ids, slots, pagein, new_slot):
      ids      ascending chunk indices of the chosen min(k, n) chunks
      slots    their pool slots
      pagein   [(chunk, slot)] for chosen chunks that were not resident, ascending chunk order
      new_slot int [n], the slot map after this step
    """
    scores = np.asarray(scores, dtype=np.float32)
    prev_slot = np.asarray(prev_slot, dtype=np.int64)
    n = len(scores)
    chosen = sorted(rank_chunks(scores)[: min(k, n)])
    kept = {}
    for c in chosen:
        s = int(prev_slot[c])
        if slot_base <= s < slot_base + k:
            if s in kept.values():
                raise ValueError(f"slot {s} is held by two chunks")
            kept[c] = s
    used = set(kept.values())
    free = [s for s in range(slot_base, slot_base + k) if s not in used]
    new = [c for c in chosen if c not in kept]
    assign = dict(zip(new, free))
    slots = [kept[c] if c in kept else assign[c] for c in chosen]
    pagein = [(c, assign[c]) for c in new]
    new_slot = np.full(n, -1, dtype=np.int64)
    for c, s in zip(chosen, slots):
        new_slot[c] = s
    return chosen, slots, pagein, new_slot


def select_resident(scores, cu_chunks, k: int, slot_of_chunk):
    """Residency for a batch of sequences; sequence b owns slots [b*k, b*k + k).

    Returns dict with flat arrays laid out like the library's outputs:
      resident_ids / resident_slots  concatenated per sequence, offsets cu_resident [B+1]
      pagein   list per sequence of (global chunk index, slot)
      slot_of_chunk  the updated map (global chunk index -> slot or -1)
    """
    cu_chunks = [int(x) for x in cu_chunks]
    slot_of_chunk = np.asarray(slot_of_chunk, dtype=np.int64)
    ids, slots, cu_res, pagein = [], [], [0], []
    new_map = np.full_like(slot_of_chunk, -1)
    for b in range(len(cu_chunks) - 1):
        c0, c1 = cu_chunks[b], cu_chunks[b + 1]
        i_b, s_b, p_b, m_b = select_resident_one(
            np.asarray(scores)[c0:c1], k, slot_of_chunk[c0:c1], b * k)
        ids += i_b
        slots += s_b
        cu_res.append(cu_res[-1] + len(i_b))
        pagein.append([(c0 + c, s) for c, s in p_b])
        new_map[c0:c1] = m_b
    return {"resident_ids": np.array(ids, dtype=np.int64),
            "resident_slots": np.array(slots, dtype=np.int64),
            "cu_resident": np.array(cu_res, dtype=np.int64),
            "pagein": pagein,
            "slot_of_chunk": new_map}


# --------------------------------------------------------------------------------------------
# a2: page-in, a bit-exact copy of host chunks into pool slots  ([LX] item 1)
# --------------------------------------------------------------------------------------------

def page_in(host_k, host_v, k_pool, v_pool, pagein_pairs):
    """Copy chunk `c` of the host store ([chunk][Hkv][64][d]) into pool slot `s` for every (c, s)."""
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    for c, s in pagein_pairs:
        k_pool[s] = host_k[c]
        v_pool[s] = host_v[c]
    return k_pool, v_pool


# --------------------------------------------------------------------------------------------
# Confidence-gated draft depths  ([WD] "Width vs. Depth: Speculating on the Margin": draft depth
# allocated unevenly by drafter confidence beats fixed depths; it needs ragged speculation)
# --------------------------------------------------------------------------------------------

def expected_committed(confidence: float, depth: int) -> float:
    """Expected tokens one verify step commits for a sequence whose drafted positions are each
    accepted with probability c, independently: the accepted prefix plus the bonus token,
    1 + c + c^2 + ... + c^depth."""
    return sum(confidence ** k for k in range(depth + 1))


def gate_depths(confidence, row_budget: int, max_depth: int) -> list[int]:
    """Draft depths D_b that maximise the expected committed tokens sum_b expected_committed(c_b,
    D_b) under a budget of verify rows sum_b (D_b + 1) <= row_budget and 0 <= D_b <= max_depth.
    Adding one drafted position to sequence b gains c_b^(D_b + 1), which shrinks as D_b grows,
    so handing out the rows one at a time to the largest gain (ties to the lower index) reaches
    the maximum. Every sequence keeps its one row for the committed token."""
    depth = [0] * len(confidence)
    rows = len(confidence)
    while rows < row_budget:
        best, gain = -1, -1.0
        for b, c in enumerate(confidence):
            if depth[b] < max_depth:
                g = float(c) ** (depth[b] + 1)
                if g > gain:
                    best, gain = b, g
        if best < 0:
            break
        depth[best] += 1
        rows += 1
    return depth


# --------------------------------------------------------------------------------------------
# Block K/V append  ([LX] "Three optimizations", item 1: the pool pages cold 64-token chunks to
# host RAM bit-exact; item 3: window layers keep slot = pos mod 2048)
# --------------------------------------------------------------------------------------------

def append_full(k_new, v_new, cu_q, seq_len, cu_chunks, slot_of_chunk, host_k, host_v, k_pool, v_pool):
    """Write the verify block's K/V rows of one full layer where later steps read them.

    Block token i of sequence b sits at position p = L_b - q_b + i. Its row goes to row p mod 64
    of chunk cu_chunks[b] + p // 64 of the chunk store ([chunk][Hkv][64][d]), and, when that
    chunk holds a pool slot (0 <= slot_of_chunk[chunk] < slots), to the same row of the slot.
    Writing through to the store keeps every chunk's host copy bit-exact with the pool, so a
    chunk that leaves the pool needs no separate page-out.
    k_new, v_new: bf16 bits [T][Hkv][d]. Returns new (host_k, host_v, k_pool, v_pool).
    """
    host_k, host_v = np.array(host_k, copy=True), np.array(host_v, copy=True)
    k_pool, v_pool = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    for b in range(len(cu_q) - 1):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        for i in range(e - a):
            p = _query_position(int(seq_len[b]), e - a, i)
            c = int(cu_chunks[b]) + p // CHUNK_TOKENS
            r = p % CHUNK_TOKENS
            host_k[c, :, r, :] = k_new[a + i]
            host_v[c, :, r, :] = v_new[a + i]
            slot = int(slot_of_chunk[c])
            if 0 <= slot < k_pool.shape[0]:
                k_pool[slot, :, r, :] = k_new[a + i]
                v_pool[slot, :, r, :] = v_new[a + i]
    return host_k, host_v, k_pool, v_pool


def append_ring(k_new, v_new, cu_q, seq_len, ring_offset, k_ring, v_ring):
    """Write block token i of sequence b (position p = L_b - q_b + i) into ring slot
    (p + phi_b) mod R of every KV head of its window layer's ring ([B][Hkv][R][d]).
    Returns new (k_ring, v_ring)."""
    k_ring, v_ring = np.array(k_ring, copy=True), np.array(v_ring, copy=True)
    ring_len = k_ring.shape[2]
    for b in range(len(cu_q) - 1):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        for i in range(e - a):
            p = _query_position(int(seq_len[b]), e - a, i)
            slot = _ring_slot(p, int(ring_offset[b]), ring_len)
            k_ring[b, :, slot, :] = k_new[a + i]
            v_ring[b, :, slot, :] = v_new[a + i]
    return k_ring, v_ring


# --------------------------------------------------------------------------------------------
# a3 + a4 + a5: masked softmax attention over an explicitly gathered key list
# --------------------------------------------------------------------------------------------

def softmax_attend(q, keys, values, scale: float):
    """y = sum_j softmax(scale * <q, k_j>)_j v_j in fp64, max-subtracted.

    Returns (y, lse, row_sum). With no key: y = 0, lse = -inf, row_sum = 0.
    """
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1]), -math.inf, 0.0
    s = scale * (keys @ q)
    m = s.max()
    w = np.exp(s - m)
    z = w.sum()
    p = w / z
    return p @ values, m + math.log(z), p.sum()


def attend_full_seq(q, k_pool, v_pool, resident_ids, resident_slots, seq_len: int,
                    scale: float | None = None, return_rowsum: bool = False, rows=None):
    """One sequence of a full-attention layer over the resident chunks of its KVFlash pool.

    q        bf16 bits [q][Hq][d]          the verify block's queries
    k_pool   bf16 bits [slots][Hkv][64][d] pool (v_pool alike)
    resident_ids, resident_slots           resident chunk indices and the slots holding them
    seq_len  L, including the q block tokens
    rows     optional list of (query i, q-head g) to compute (the others are left NaN), for
             samples of large cases
    Returns O [q][Hq][d] f64, LSE [q][Hq] f64 (and the softmax row sums if asked).
    """
    qf = bf16_to_f64(q)
    nq, hq_count, d = qf.shape
    hkv = k_pool.shape[1]
    group = hq_count // hkv
    scale = _default_scale(d) if scale is None else scale
    # Gather: the explicit (position, K, V) list of every resident token.
    pos, ks, vs = [], [], []
    for cid, slot in zip(resident_ids, resident_slots):
        p = int(cid) * CHUNK_TOKENS + np.arange(CHUNK_TOKENS)
        keep = p < seq_len
        pos.append(p[keep])
        ks.append(bf16_to_f64(k_pool[int(slot)])[:, keep, :])  # [Hkv][t][d]
        vs.append(bf16_to_f64(v_pool[int(slot)])[:, keep, :])
    pos = np.concatenate(pos) if pos else np.zeros(0, dtype=np.int64)
    kk = np.concatenate(ks, axis=1) if ks else np.zeros((hkv, 0, d))
    vv = np.concatenate(vs, axis=1) if vs else np.zeros((hkv, 0, d))
    fill = np.nan if rows is not None else 0.0
    out = np.full((nq, hq_count, d), fill)
    lse = np.full((nq, hq_count), fill)
    rsum = np.full((nq, hq_count), fill)
    todo = rows if rows is not None else [(i, g) for i in range(nq) for g in range(hq_count)]
    for i, g in todo:
        p_i = _query_position(seq_len, nq, i)
        sel = pos <= p_i
        h = _kv_head_of(g, group)
        out[i, g], lse[i, g], rsum[i, g] = softmax_attend(qf[i, g], kk[h][sel], vv[h][sel], scale)
    return (out, lse, rsum) if return_rowsum else (out, lse)


def attend_ring_seq(q, k_ring, v_ring, phi: int, seq_len: int, window: int,
                    scale: float | None = None, return_rowsum: bool = False):
    """One sequence of a sliding-window layer read from its position ring.

    q       bf16 bits [q][Hq][d]
    k_ring  bf16 bits [Hkv][R][d]   (v_ring alike); position p sits in slot (p + phi) mod R
    Query i attends positions [max(0, p_i - window + 1), p_i].
    """
    qf = bf16_to_f64(q)
    nq, hq_count, d = qf.shape
    hkv, ring_len, _ = k_ring.shape
    group = hq_count // hkv
    scale = _default_scale(d) if scale is None else scale
    out = np.zeros((nq, hq_count, d))
    lse = np.zeros((nq, hq_count))
    rsum = np.zeros((nq, hq_count))
    for i in range(nq):
        p_i = _query_position(seq_len, nq, i)
        positions = range(_window_start(p_i, window), p_i + 1)
        slots = np.array([_ring_slot(p, phi, ring_len) for p in positions], dtype=np.int64)
        for g in range(hq_count):
            h = _kv_head_of(g, group)
            keys = bf16_to_f64(k_ring[h][slots]) if len(slots) else np.zeros((0, d))
            vals = bf16_to_f64(v_ring[h][slots]) if len(slots) else np.zeros((0, d))
            out[i, g], lse[i, g], rsum[i, g] = softmax_attend(qf[i, g], keys, vals, scale)
    return (out, lse, rsum) if return_rowsum else (out, lse)


def attend_full(q, cu_q, k_pool, v_pool, resident_ids, resident_slots, cu_resident, seq_len,
                scale: float | None = None):
    """Batch form of attend_full_seq: q [T][Hq][d] with sequence b owning rows cu_q[b]:cu_q[b+1]."""
    out = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:2], dtype=np.float64)
    for b in range(len(cu_q) - 1):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        r0, r1 = int(cu_resident[b]), int(cu_resident[b + 1])
        out[a:e], lse[a:e] = attend_full_seq(q[a:e], k_pool, v_pool, resident_ids[r0:r1],
                                             resident_slots[r0:r1], int(seq_len[b]), scale)
    return out, lse


def attend_ring(q, cu_q, k_ring, v_ring, ring_offset, seq_len, window: int,
                scale: float | None = None):
    """Batch form of attend_ring_seq: k_ring [B][Hkv][R][d]."""
    out = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:2], dtype=np.float64)
    for b in range(len(cu_q) - 1):
        a, e = int(cu_q[b]), int(cu_q[b + 1])
        out[a:e], lse[a:e] = attend_ring_seq(q[a:e], k_ring[b], v_ring[b], int(ring_offset[b]),
                                             int(seq_len[b]), window, scale)
    return out, lse


# --------------------------------------------------------------------------------------------
# a6: greedy acceptance  ([LX] "The model ..."; [CM] "DFlash Drafters ...")
# --------------------------------------------------------------------------------------------

def argmax_row(row) -> int:
    """Index of the greatest fp32 value; ties to the lowest index; a NaN is the greatest (first wins)."""
    row = np.asarray(row, dtype=np.float32)
    nan = np.flatnonzero(np.isnan(row))
    if nan.size:
        return int(nan[0])
    return int(np.flatnonzero(row == row.max())[0])


def accept_seq(logits, drafts):
    """One sequence: logits [D+1][V] fp32, drafts [D] -> (n, bonus, committed [D+1])."""
    a = [argmax_row(r) for r in logits]
    depth = len(drafts)
    n = 0
    while n < depth and a[n] == int(drafts[n]):
        n += 1
    committed = [int(x) for x in drafts[:n]] + [a[n]] + [-1] * (depth - n)
    return n, a[n], committed


def accept(logits, drafts, cu_rows):
    """Batch: sequence b owns logit rows cu_rows[b]:cu_rows[b+1] (D_b + 1 rows) and drafts
    (cu_rows[b] - b) : (cu_rows[b+1] - b - 1)."""
    ns, bonus, committed = [], [], []
    for b in range(len(cu_rows) - 1):
        r0, r1 = int(cu_rows[b]), int(cu_rows[b + 1])
        n, a, c = accept_seq(logits[r0:r1], drafts[r0 - b: r1 - b - 1])
        ns.append(n)
        bonus.append(a)
        committed += c
    return (np.array(ns, dtype=np.int64), np.array(bonus, dtype=np.int64),
            np.array(committed, dtype=np.int64))
