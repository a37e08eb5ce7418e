"""Pins of the oracle's block K/V append (oracle/vfy_oracle.py append_full / append_ring) against
hand-worked coordinates: which chunk row, pool slot and ring slot each block token lands in."""
import numpy as np

from oracle import vfy_oracle as O


def test_append_full_hand_case():
    """L = 130, q = 3: positions 127, 128, 129 -> chunk 1 row 63, chunk 2 rows 0 and 1. Chunk 1 is
    resident in slot 5, chunk 2 in slot 2, chunk 0 nowhere. Two KV heads, d = 4."""
    hkv, d = 2, 4
    k_new = np.array([[[11] * d, [12] * d], [[21] * d, [22] * d], [[31] * d, [32] * d]], np.uint16)
    v_new = k_new + 100
    host_k = np.zeros((3, hkv, 64, d), np.uint16)
    host_v = np.zeros_like(host_k)
    pool_k = np.zeros((6, hkv, 64, d), np.uint16)
    pool_v = np.zeros_like(pool_k)
    hk, hv, pk, pv = O.append_full(k_new, v_new, [0, 3], [130], [0, 3], [-1, 5, 2], host_k, host_v, pool_k, pool_v)
    want = np.zeros_like(host_k)
    want[1, 0, 63], want[1, 1, 63] = 11, 12
    want[2, 0, 0], want[2, 1, 0] = 21, 22
    want[2, 0, 1], want[2, 1, 1] = 31, 32
    assert (hk == want).all() and (hv == np.where(want > 0, want + 100, 0)).all()
    wantp = np.zeros_like(pool_k)
    wantp[5, :, 63] = want[1, :, 63]
    wantp[2, :, 0] = want[2, :, 0]
    wantp[2, :, 1] = want[2, :, 1]
    assert (pk == wantp).all() and (pv == np.where(wantp > 0, wantp + 100, 0)).all()


def test_append_full_second_sequence_offsets():
    """Sequence 1's chunks start at cu_chunks[1] = 4 of the store; its block (L = 70, q = 2:
    positions 68, 69) lands in its chunk 1 = store chunk 5, rows 4 and 5; chunk 5 is not
    resident, so no pool row changes."""
    k_new = np.array([[[1, 1]], [[7, 7]], [[8, 8]]], np.uint16)        # seq 0: 1 token, seq 1: 2 tokens
    store = np.zeros((6, 1, 64, 2), np.uint16)
    pool = np.zeros((2, 1, 64, 2), np.uint16)
    slot_of_chunk = [0, -1, -1, -1, -1, -1]
    hk, _, pk, _ = O.append_full(k_new, k_new, [0, 1, 3], [64, 70], [0, 4, 6], slot_of_chunk, store, store, pool, pool)
    assert hk[0, 0, 63].tolist() == [1, 1] and pk[0, 0, 63].tolist() == [1, 1]   # seq 0: p = 63
    assert hk[5, 0, 4].tolist() == [7, 7] and hk[5, 0, 5].tolist() == [8, 8]
    assert int(hk.sum()) == 2 * (1 + 7 + 8) and int(pk.sum()) == 2


def test_append_ring_wraps():
    """R = 8, phi = 7, L = 10, q = 3: positions 7, 8, 9 -> slots 6, 7, 0."""
    k_new = np.array([[[5]], [[6]], [[7]]], np.uint16)
    ring = np.zeros((1, 1, 8, 1), np.uint16)
    kr, vr = O.append_ring(k_new, k_new + 1, [0, 3], [10], [7], ring, ring)
    assert kr[0, 0, :, 0].tolist() == [7, 0, 0, 0, 0, 0, 5, 6]
    assert vr[0, 0, :, 0].tolist() == [8, 0, 0, 0, 0, 0, 6, 7]


def test_append_ring_negative_offset_and_batch():
    """phi is taken mod R (Python's %, non-negative): phi = -1 with R = 4 is phi = 3."""
    k_new = np.array([[[1]], [[2]]], np.uint16)
    ring = np.zeros((2, 1, 4, 1), np.uint16)
    kr, _ = O.append_ring(k_new, k_new, [0, 1, 2], [5, 2], [-1, 0], ring, ring)
    assert kr[0, 0, :, 0].tolist() == [0, 0, 0, 1]        # seq 0: p = 4 -> (4 + 3) % 4 = 3
    assert kr[1, 0, :, 0].tolist() == [0, 2, 0, 0]        # seq 1: p = 1 -> slot 1
