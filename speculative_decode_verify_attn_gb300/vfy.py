"""Thin Python binding of libvfy.so (ctypes). The functions carry the C ABI's names and only
marshal arguments: torch tensors become device (or pinned host) pointers, the current torch CUDA
stream becomes the stream handle. Every step of the verify path runs in the library's kernels.
There is no fallback: if the library is not built, or its device is absent, calls raise."""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

VFY_OK, VFY_EINVAL, VFY_ECUDA, VFY_ENOMEM, VFY_EUNSUPPORTED, VFY_EDEVICE_INPUT, VFY_EDEVICE_TIMEOUT = range(7)

EXPORTS = ("vfy_create", "vfy_destroy", "vfy_get_status", "vfy_strerror", "vfy_set_splits",
           "vfy_select_resident", "vfy_page_in", "vfy_attend_full", "vfy_attend_swa", "vfy_accept",
           "vfy_accept_static", "vfy_launch_count", "vfy_append_full", "vfy_append_swa",
           "vfy_gate_depths", "vfy_test_wait_timeout", "vfy_set_stable_metadata", "vfy_set_pagein_ctas")


class VfyError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("chunk_tokens", ctypes.c_int), ("window", ctypes.c_int), ("ring_len", ctypes.c_int),
                ("max_seqs", ctypes.c_int), ("max_queries_per_seq", ctypes.c_int),
                ("max_splits", ctypes.c_int), ("softmax_scale", ctypes.c_float)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libvfy.so (built in-tree by build.build())."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(or python -m speculative_decode_verify_attn_gb300.build)")
        L = ctypes.CDLL(path)
        L.vfy_create.argtypes = [ctypes.POINTER(Config), _I, ctypes.POINTER(_P)]
        L.vfy_destroy.argtypes = [_P]
        L.vfy_destroy.restype = None
        L.vfy_get_status.argtypes = [_P, _P]
        L.vfy_strerror.argtypes = [_I]
        L.vfy_strerror.restype = ctypes.c_char_p
        L.vfy_set_splits.argtypes = [_P, _I, _I]
        L.vfy_test_wait_timeout.argtypes = [_P, ctypes.c_uint64]
        L.vfy_set_stable_metadata.argtypes = [_P, _I]
        L.vfy_set_pagein_ctas.argtypes = [_P, _I]
        L.vfy_select_resident.argtypes = [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
        L.vfy_page_in.argtypes = [_P, _P, _P, ctypes.c_int64, _P, _P, _I, _P, _P, _I, _I, _P]
        L.vfy_attend_full.argtypes = [_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _I, _P]
        L.vfy_attend_swa.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]
        L.vfy_accept.argtypes = [_P, _P, _I, _P, _P, _I, _P, _P, _P, _I, _P]
        L.vfy_accept_static.argtypes = [_P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P]
        L.vfy_append_full.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P, _I, _I, _P]
        L.vfy_append_swa.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P]
        L.vfy_gate_depths.argtypes = [_P, _I, _I, _I, _P]
        L.vfy_launch_count.argtypes = [_P]
        L.vfy_launch_count.restype = ctypes.c_ulonglong
        for name in EXPORTS:
            if name not in ("vfy_destroy", "vfy_strerror", "vfy_launch_count"):
                getattr(L, name).restype = _I
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().vfy_strerror(status).decode()


def _check(status: int, what: str):
    if status != VFY_OK:
        raise VfyError(status, what)


# ---------------------------------------------------------------------------------------------
# Pointer marshalling
# ---------------------------------------------------------------------------------------------

def _dev(t: torch.Tensor | None, dtypes, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host(t: torch.Tensor, dtypes, name: str):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


BF16 = (torch.bfloat16, torch.int16)
I32 = (torch.int32,)
F32 = (torch.float32,)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------------------------------------
# The C ABI, one function each
# ---------------------------------------------------------------------------------------------

class Context:
    """Owns a vfy_ctx (created by vfy_create, freed by vfy_destroy / close())."""

    def __init__(self, handle: ctypes.c_void_p, cfg: Config, device: int):
        self.handle = handle
        self.cfg = cfg
        self.device = device

    def close(self):
        if self.handle:
            lib().vfy_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def vfy_create(num_q_heads: int, num_kv_heads: int, head_dim: int, *, window: int = 512,
               ring_len: int = 2048, max_seqs: int = 1, max_queries_per_seq: int = 17,
               max_splits: int = 64, softmax_scale: float = 0.0, device: int | None = None,
               chunk_tokens: int = 64) -> Context:
    dev = torch.cuda.current_device() if device is None else int(device)
    cfg = Config(num_q_heads, num_kv_heads, head_dim, chunk_tokens, window, ring_len, max_seqs,
                 max_queries_per_seq, max_splits, softmax_scale)
    h = ctypes.c_void_p()
    _check(lib().vfy_create(ctypes.byref(cfg), dev, ctypes.byref(h)), "vfy_create")
    return Context(h, cfg, dev)


def vfy_destroy(ctx: Context):
    ctx.close()


def vfy_get_status(ctx: Context, stream=None) -> int:
    return lib().vfy_get_status(ctx.handle, _stream(stream))


def vfy_launch_count(ctx: Context) -> int:
    return int(lib().vfy_launch_count(ctx.handle))


def vfy_gate_depths(confidence, row_budget: int, max_depth: int) -> list[int]:
    """Host function (no device): confidence-gated draft depths. `confidence` is a sequence of
    per-sequence acceptance probabilities in [0, 1]."""
    import numpy as _np
    c = _np.ascontiguousarray(_np.asarray(confidence, dtype=_np.float32))
    d = _np.zeros(len(c), dtype=_np.int32)
    _check(lib().vfy_gate_depths(c.ctypes.data_as(_P), len(c), int(row_budget), int(max_depth),
                                 d.ctypes.data_as(_P)), "vfy_gate_depths")
    return d.tolist()


def vfy_set_splits(ctx: Context, full_splits: int = 0, swa_splits: int = 0):
    _check(lib().vfy_set_splits(ctx.handle, full_splits, swa_splits), "vfy_set_splits")


def vfy_test_wait_timeout(ctx: Context, limit_ns: int = 0):
    """Test of the timeout path: every attention CTA enqueued afterwards first runs one wait of
    limit_ns that cannot complete (0 turns the test off). See include/vfy.h."""
    _check(lib().vfy_test_wait_timeout(ctx.handle, int(limit_ns)), "vfy_test_wait_timeout")


def vfy_set_pagein_ctas(ctx: Context, ctas_per_chunk: int = 0):
    """CTAs per chunk of the page-ins enqueued afterwards (1-4; 0 = 2). See include/vfy.h."""
    _check(lib().vfy_set_pagein_ctas(ctx.handle, int(ctas_per_chunk)), "vfy_set_pagein_ctas")


def vfy_set_stable_metadata(ctx: Context, stable: bool = True):
    """Declare that this context's per-step attention metadata is final before its kernels start
    (see include/vfy.h); the kernels then read it before waiting for the previous kernel."""
    _check(lib().vfy_set_stable_metadata(ctx.handle, 1 if stable else 0), "vfy_set_stable_metadata")


def vfy_select_resident(ctx: Context, scores, cu_chunks, num_seqs: int, max_chunks_per_seq: int, k: int,
                        slot_of_chunk, resident_ids, resident_slots, cu_resident, pagein_list,
                        pagein_count, stream=None):
    _check(lib().vfy_select_resident(
        ctx.handle, _dev(scores, F32, "scores"), _dev(cu_chunks, I32, "cu_chunks"), num_seqs,
        max_chunks_per_seq, k, _dev(slot_of_chunk, I32, "slot_of_chunk"),
        _dev(resident_ids, I32, "resident_ids"), _dev(resident_slots, I32, "resident_slots"),
        _dev(cu_resident, I32, "cu_resident"), _dev(pagein_list, I32, "pagein_list"),
        _dev(pagein_count, I32, "pagein_count"), _stream(stream)), "vfy_select_resident")


def vfy_page_in(ctx: Context, host_k, host_v, num_host_chunks: int, k_pool, v_pool, num_slots: int,
                pagein_list, pagein_count, num_seqs: int, k: int, stream=None):
    hk = _dev(host_k, BF16, "host_k") if host_k.is_cuda else _host(host_k, BF16, "host_k")
    hv = _dev(host_v, BF16, "host_v") if host_v.is_cuda else _host(host_v, BF16, "host_v")
    _check(lib().vfy_page_in(
        ctx.handle, hk, hv, num_host_chunks, _dev(k_pool, BF16, "k_pool"), _dev(v_pool, BF16, "v_pool"),
        num_slots, _dev(pagein_list, I32, "pagein_list"), _dev(pagein_count, I32, "pagein_count"),
        num_seqs, k, _stream(stream)), "vfy_page_in")


def vfy_append_full(ctx: Context, k_new, v_new, cu_q, seq_len, cu_chunks, slot_of_chunk, host_k, host_v,
                    num_host_chunks: int, k_pool, v_pool, num_slots: int, num_seqs: int, stream=None):
    hk = _dev(host_k, BF16, "host_k") if host_k.is_cuda else _host(host_k, BF16, "host_k")
    hv = _dev(host_v, BF16, "host_v") if host_v.is_cuda else _host(host_v, BF16, "host_v")
    _check(lib().vfy_append_full(
        ctx.handle, _dev(k_new, BF16, "k_new"), _dev(v_new, BF16, "v_new"), _dev(cu_q, I32, "cu_q"),
        _dev(seq_len, I32, "seq_len"), _dev(cu_chunks, I32, "cu_chunks"), _dev(slot_of_chunk, I32, "slot_of_chunk"),
        hk, hv, num_host_chunks, _dev(k_pool, BF16, "k_pool"), _dev(v_pool, BF16, "v_pool"), num_slots, num_seqs,
        _stream(stream)), "vfy_append_full")


def vfy_append_swa(ctx: Context, k_new, v_new, cu_q, seq_len, ring_offset, k_ring, v_ring, num_seqs: int,
                   stream=None):
    _check(lib().vfy_append_swa(
        ctx.handle, _dev(k_new, BF16, "k_new"), _dev(v_new, BF16, "v_new"), _dev(cu_q, I32, "cu_q"),
        _dev(seq_len, I32, "seq_len"), _dev(ring_offset, I32, "ring_offset"), _dev(k_ring, BF16, "k_ring"),
        _dev(v_ring, BF16, "v_ring"), num_seqs, _stream(stream)), "vfy_append_swa")


def vfy_attend_full(ctx: Context, q, cu_q, k_pool, v_pool, num_slots: int, resident_ids, resident_slots,
                    cu_resident, max_resident_per_seq: int, seq_len, out, lse, num_seqs: int, stream=None):
    _check(lib().vfy_attend_full(
        ctx.handle, _dev(q, BF16, "q"), _dev(cu_q, I32, "cu_q"), _dev(k_pool, BF16, "k_pool"),
        _dev(v_pool, BF16, "v_pool"), num_slots, _dev(resident_ids, I32, "resident_ids"),
        _dev(resident_slots, I32, "resident_slots"), _dev(cu_resident, I32, "cu_resident"),
        max_resident_per_seq, _dev(seq_len, I32, "seq_len"), _dev(out, BF16, "out"),
        _dev(lse, F32, "lse"), num_seqs, _stream(stream)), "vfy_attend_full")


def vfy_attend_swa(ctx: Context, q, cu_q, k_ring, v_ring, ring_offset, seq_len, out, lse, num_seqs: int,
                   stream=None):
    _check(lib().vfy_attend_swa(
        ctx.handle, _dev(q, BF16, "q"), _dev(cu_q, I32, "cu_q"), _dev(k_ring, BF16, "k_ring"),
        _dev(v_ring, BF16, "v_ring"), _dev(ring_offset, I32, "ring_offset"), _dev(seq_len, I32, "seq_len"),
        _dev(out, BF16, "out"), _dev(lse, F32, "lse"), num_seqs, _stream(stream)), "vfy_attend_swa")


def vfy_accept(ctx: Context, logits, vocab: int, drafts, cu_rows, max_rows: int, accepted_len, bonus,
               committed, num_seqs: int, stream=None):
    _check(lib().vfy_accept(
        ctx.handle, _dev(logits, F32, "logits"), vocab, _dev(drafts, I32, "drafts"), _dev(cu_rows, I32, "cu_rows"),
        max_rows, _dev(accepted_len, I32, "accepted_len"), _dev(bonus, I32, "bonus"),
        _dev(committed, I32, "committed"), num_seqs, _stream(stream)), "vfy_accept")


def vfy_accept_static(logits, vocab: int, drafts, cu_rows, num_seqs: int, max_rows: int, accepted_len, bonus,
                      committed, device_error=None, stream=None):
    """vfy_accept without a context and without allocating (for callers that cannot allocate
    device memory); max_rows <= 1024. See include/vfy.h."""
    _check(lib().vfy_accept_static(
        _dev(logits, F32, "logits"), vocab, _dev(drafts, I32, "drafts"), _dev(cu_rows, I32, "cu_rows"),
        num_seqs, max_rows, _dev(accepted_len, I32, "accepted_len"), _dev(bonus, I32, "bonus"),
        _dev(committed, I32, "committed"), _dev(device_error, I32, "device_error"), _stream(stream)),
        "vfy_accept_static")
