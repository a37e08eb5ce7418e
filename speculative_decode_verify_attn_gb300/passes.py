"""A whole verify pass over a synthetic model, captured once as a CUDA graph and replayed.

The pass is the data-parallel hot path of one speculative-decoding step at long context
('Laguna XS 2.1 33B on a RTX 3090' (lucebox): 40 layers in a 3-in-4 window pattern, 'Three
optimizations' items 1 and 3; CUDA-graph replay of the decode loop):

  vfy_select_resident      (side stream)    residency for this step (one chunk table for all
                                            full layers; each full layer has its own pool)
  vfy_page_in x n_full      (side stream)   the step's newly resident chunks, host -> pools
  for layer l in 0..n_layers-1:             window layers where l % 4 != 3, full where l % 4 == 3
      vfy_attend_swa / vfy_attend_full      (a full layer waits for its own page-in)
  vfy_accept                                argmax + greedy acceptance over the block's logits

Every per-step value (scores, lengths, lists, offsets, drafts) sits in device memory at a fixed
address, so one graph serves every step. Inputs are synthetic (synth.py) with the shapes of the
pages' workloads; model weights do not enter: the block's Q rows and KV are random bf16.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import synth, vfy

CHUNK = 64
# CTAs per chunk of the page-ins. The first full layer waits for the first page-in; the others
# run beside the layers, whose attention kernels their host reads in flight slow down. On GB300,
# 3 or 4 CTAs for all cost the pass 2 and 12 us; 1 for the page-ins after the first was 0.1
# us/layer faster than 2 on one box and 0.02 slower on another (the host link differs by box),
# so both keep 2.
PAGEIN_CTAS_FIRST = 2
PAGEIN_CTAS_REST = 2


def _packed(layout, dev):
    """One uint8 device buffer with 256-byte-aligned byte views {name: view} for [(name, nbytes)],
    and the byte offset of every view."""
    offs, off = {}, 0
    for name, nbytes in layout:
        offs[name] = (off, nbytes)
        off += (nbytes + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=dev)
    return buf, {name: buf.narrow(0, o, n) for name, (o, n) in offs.items()}, {k: o for k, (o, _) in offs.items()}


def is_full_layer(layer: int) -> bool:
    """3-in-4 pattern: layers 3, 7, 11, ... are full attention, the others window layers."""
    return layer % 4 == 3


def join_points(n_full: int) -> dict[int, int]:
    """Where the layer chain waits for the paging stream: {full layer j: last page-in it waits for}.

    Page-ins complete in order on one stream, so waiting for page-in m covers every page-in up to
    m. Full layer j joins up to page-in min(2j, n_full - 1) unless an earlier join already covered
    page-in j: joins at j = 0, 1, 3, 7, ... with groups of 1, 2, 4, 8, ... page-ins. Each group is
    due well after it completes (a full layer comes every four layers, while a page-in takes about
    as long as one layer), and every full layer j still waits for its own page-in j.
    """
    joins, covered = {}, -1
    for j in range(n_full):
        if j > covered:
            covered = min(2 * j, n_full - 1)
            joins[j] = covered
    return joins


@dataclass
class PassSizes:
    n_layers: int
    n_full: int
    n_swa: int
    bytes_full: int       # algorithmic bytes of one full layer (KV read + Q read + O write)
    bytes_swa: int
    bytes_accept: int
    bytes_pass: int


class VerifyPass:
    """Single-sequence 256K pass (one replica per GPU)."""

    def __init__(self, workload: synth.Workload, device: int = 0, seed: int = 0, all_resident: bool = False,
                 match_prob: float = 0.56, stable_metadata: bool = True):
        assert workload.num_seqs == 1
        self.w = workload
        self.dev = torch.device("cuda", device)
        s = workload.shape
        self.shape = s
        self.L = workload.seq_lens[0]
        self.q = workload.queries[0]
        self.n_chunks = (self.L + CHUNK - 1) // CHUNK
        self.all_resident = all_resident
        self.k = self.n_chunks if all_resident else workload.resident_chunks
        self.n_layers = workload.n_full + workload.n_swa
        self.vocab = workload.vocab
        rng = np.random.default_rng(seed)
        gen = torch.Generator(device=self.dev)
        gen.manual_seed(seed)
        dev = self.dev
        hkv, d, hq = s.num_kv_heads, s.head_dim, s.num_q_heads
        torch.cuda.set_device(dev)

        self.ctx = vfy.vfy_create(hq, hkv, d, window=synth.WINDOW, ring_len=synth.RING, max_seqs=1,
                                  max_queries_per_seq=self.q, max_splits=64, device=device)
        # The pass's metadata (lengths, offsets, block offsets) is set before any step, and its
        # residency lists come from the paging stream, which the layer chain joins through events:
        # every kernel that writes them has completed before a layer that reads them starts.
        vfy.vfy_set_stable_metadata(self.ctx, stable_metadata)
        # --- per-step residency inputs ---
        self.rot = synth.rotating_residency(rng, self.n_chunks, self.k, workload.pagein_per_step or 16,
                                            self.L, self.q) if not all_resident else None
        self.cu_chunks = torch.tensor([0, self.n_chunks], dtype=torch.int32, device=dev)
        # One device buffer holds every per-step input (block queries, residency scores, logits,
        # drafts) and one holds every per-step result (accepted length, bonus, committed tokens),
        # so a caller moves a step's data with one copy each way.
        # The order is the order a step needs them in: the residency scores (first kernel), the
        # layers' queries, then the logits and drafts (last kernel).
        qbytes = self.n_layers * self.q * hq * d * 2
        layout = [("scores", self.n_chunks * 4), ("q", qbytes), ("logits", self.q * workload.vocab * 4),
                  ("drafts", max(self.q - 1, 1) * 4)]
        self.inputs, views, self.input_offsets = _packed(layout, dev)
        self.q_layer_bytes = self.q * hq * d * 2
        self.scores = views["scores"].view(torch.float32)
        self.scores.zero_()
        self.slot_of_chunk = torch.full((self.n_chunks,), -1, dtype=torch.int32, device=dev)
        self.res_ids = torch.zeros(self.k, dtype=torch.int32, device=dev)
        self.res_slots = torch.zeros(self.k, dtype=torch.int32, device=dev)
        self.cu_res = torch.tensor([0, self.k], dtype=torch.int32, device=dev)
        self.pagein_list = torch.zeros((self.k, 2), dtype=torch.int32, device=dev)
        self.pagein_count = torch.zeros(1, dtype=torch.int32, device=dev)
        if all_resident:
            self.res_ids.copy_(torch.arange(self.k, dtype=torch.int32, device=dev))
            self.res_slots.copy_(torch.arange(self.k, dtype=torch.int32, device=dev))
        self.score_table = (torch.from_numpy(np.stack([self.rot.scores(t) for t in range(len(self.rot.groups))]))
                            .to(dev)) if self.rot is not None else None
        # --- KV: per full layer a pool (+ a pinned host store when paging), per window layer a ring
        self.full_layers = [l for l in range(self.n_layers) if is_full_layer(l)]
        self.swa_layers = [l for l in range(self.n_layers) if not is_full_layer(l)]
        pool_shape = (self.k, hkv, CHUNK, d)
        self.pool_k, self.pool_v, self.host_k, self.host_v = {}, {}, {}, {}
        for l in self.full_layers:
            if all_resident:
                self.pool_k[l] = torch.randn(pool_shape, generator=gen, device=dev, dtype=torch.bfloat16)
                self.pool_v[l] = torch.randn(pool_shape, generator=gen, device=dev, dtype=torch.bfloat16)
            else:
                self.pool_k[l] = torch.zeros(pool_shape, device=dev, dtype=torch.bfloat16)
                self.pool_v[l] = torch.zeros(pool_shape, device=dev, dtype=torch.bfloat16)
                store = (self.n_chunks, hkv, CHUNK, d)
                self.host_k[l] = torch.empty(store, dtype=torch.bfloat16, pin_memory=True)
                self.host_v[l] = torch.empty(store, dtype=torch.bfloat16, pin_memory=True)
                self.host_k[l].copy_(torch.randn(store, generator=gen, device=dev, dtype=torch.bfloat16))
                self.host_v[l].copy_(torch.randn(store, generator=gen, device=dev, dtype=torch.bfloat16))
        self.ring_k, self.ring_v = {}, {}
        ring_shape = (1, hkv, synth.RING, d)
        for l in self.swa_layers:
            self.ring_k[l] = torch.randn(ring_shape, generator=gen, device=dev, dtype=torch.bfloat16)
            self.ring_v[l] = torch.randn(ring_shape, generator=gen, device=dev, dtype=torch.bfloat16)
        phi = synth.wrapping_ring_offset(rng, self.L, synth.WINDOW + self.q - 1, synth.RING)
        self.ring_offset = torch.tensor([phi], dtype=torch.int32, device=dev)
        # --- block: queries per layer, outputs, lengths ---
        self.cu_q = torch.tensor([0, self.q], dtype=torch.int32, device=dev)
        self.seq_len = torch.tensor([self.L], dtype=torch.int32, device=dev)
        # one buffer for all layers' block queries (one host->device copy per step end to end)
        self.q_all = views["q"].view(torch.bfloat16).view(self.n_layers, self.q, hq, d)
        self.q_all.copy_(torch.randn((self.n_layers, self.q, hq, d), generator=gen, device=dev, dtype=torch.bfloat16))
        self.qs = [self.q_all[l] for l in range(self.n_layers)]
        self.out_all = torch.empty((self.n_layers, self.q, hq, d), device=dev, dtype=torch.bfloat16)
        self.outs = [self.out_all[l] for l in range(self.n_layers)]
        self.lse_all = torch.empty((self.n_layers, self.q, hq), device=dev, dtype=torch.float32)
        self.lses = [self.lse_all[l] for l in range(self.n_layers)]
        # the block's own K/V rows of every layer (for passes that append them before attending)
        self.kv_new = torch.randn((self.n_layers, 2, self.q, hkv, d), generator=gen, device=dev, dtype=torch.bfloat16)
        # --- acceptance ---
        targets = rng.integers(0, self.vocab, self.q)
        self.targets = targets
        self.logits = views["logits"].view(torch.float32).view(self.q, self.vocab)
        self.logits.copy_(torch.from_numpy(synth.planted_logits(rng, targets, self.vocab)))
        drafts = torch.from_numpy(synth.drafts_matching(rng, targets, match_prob, self.vocab))
        self.drafts = views["drafts"].view(torch.int32)[: drafts.numel()]
        self.drafts.copy_(drafts)
        self.cu_rows = torch.tensor([0, self.q], dtype=torch.int32, device=dev)
        self.results = torch.zeros(2 + self.q, dtype=torch.int32, device=dev)
        self.accepted = self.results[0:1]
        self.bonus = self.results[1:2]
        self.committed = self.results[2:]
        # Paging gets the higher priority: its CTAs go ahead of queued layer CTAs as SMs free up.
        self.side = torch.cuda.Stream(device=dev, priority=-1)
        self.copy = torch.cuda.Stream(device=dev)       # host->device input copies (end to end)
        self.graph = None
        self.kernels_per_pass = None
        self.kernels_per_pass_append = None
        self.step = 0

    # ------------------------------------------------------------------------------------------
    def sizes(self) -> PassSizes:
        s = self.shape
        per_tok = s.num_kv_heads * s.head_dim * 2 * 2                    # K + V bf16
        qo = 2 * self.q * s.num_q_heads * s.head_dim * 2                 # Q read + O write
        bytes_full = self.k * CHUNK * per_tok + qo
        span = min(self.L, synth.WINDOW + self.q - 1)
        bytes_swa = span * per_tok + qo
        bytes_accept = self.q * self.vocab * 4
        n_full, n_swa = len(self.full_layers), len(self.swa_layers)
        return PassSizes(self.n_layers, n_full, n_swa, bytes_full, bytes_swa, bytes_accept,
                         n_full * bytes_full + n_swa * bytes_swa + bytes_accept)

    def launches_per_step(self) -> int:
        """Kernels one replay of the pass graph launches, as the library counted them while the
        pass was captured (an attention call is one kernel or two, depending on its splits)."""
        if self.kernels_per_pass is None:
            raise RuntimeError("capture() the pass first")
        return self.kernels_per_pass

    def set_step_scores(self, t: int):
        """Load step t's residency scores into the fixed score buffer (outside the graph)."""
        if self.score_table is not None:
            self.scores.copy_(self.score_table[t % self.score_table.shape[0]], non_blocking=True)

    def attend_full_layer(self, l: int, stream=None):
        vfy.vfy_attend_full(self.ctx, self.qs[l], self.cu_q, self.pool_k[l], self.pool_v[l], self.k,
                            self.res_ids, self.res_slots, self.cu_res, self.k, self.seq_len, self.outs[l],
                            self.lses[l], 1, stream)

    def attend_swa_layer(self, l: int, stream=None):
        vfy.vfy_attend_swa(self.ctx, self.qs[l], self.cu_q, self.ring_k[l], self.ring_v[l], self.ring_offset,
                           self.seq_len, self.outs[l], self.lses[l], 1, stream)

    def enqueue_paging(self):
        """Residency selection and the page-ins of every full layer, on the current stream only."""
        main = torch.cuda.current_stream(self.dev)
        vfy.vfy_select_resident(self.ctx, self.scores, self.cu_chunks, 1, self.n_chunks, self.k,
                                self.slot_of_chunk, self.res_ids, self.res_slots, self.cu_res,
                                self.pagein_list, self.pagein_count, main)
        for i, l in enumerate(self.full_layers):
            vfy.vfy_set_pagein_ctas(self.ctx, PAGEIN_CTAS_FIRST if i == 0 else PAGEIN_CTAS_REST)
            vfy.vfy_page_in(self.ctx, self.host_k[l], self.host_v[l], self.n_chunks, self.pool_k[l],
                            self.pool_v[l], self.k, self.pagein_list, self.pagein_count, 1, self.k, main)
        vfy.vfy_set_pagein_ctas(self.ctx, 0)

    def enqueue_layers(self):
        """The attention layers alone, in pass order, on the current stream."""
        main = torch.cuda.current_stream(self.dev)
        for l in range(self.n_layers):
            if is_full_layer(l):
                self.attend_full_layer(l, main)
            else:
                self.attend_swa_layer(l, main)

    def enqueue_accept(self):
        vfy.vfy_accept(self.ctx, self.logits, self.vocab, self.drafts, self.cu_rows, self.q, self.accepted,
                       self.bonus, self.committed, 1, torch.cuda.current_stream(self.dev))

    def append_layer(self, l: int, stream=None):
        """The block's K/V rows of layer l into its pool slot and chunk store (written through
        to pinned host memory) or into its ring."""
        kn, vn = self.kv_new[l, 0], self.kv_new[l, 1]
        if is_full_layer(l):
            vfy.vfy_append_full(self.ctx, kn, vn, self.cu_q, self.seq_len, self.cu_chunks, self.slot_of_chunk,
                                self.host_k[l] if self.host_k else self.pool_k[l],
                                self.host_v[l] if self.host_v else self.pool_v[l],
                                self.n_chunks if self.host_k else self.k, self.pool_k[l], self.pool_v[l], self.k, 1,
                                stream)
        else:
            vfy.vfy_append_swa(self.ctx, kn, vn, self.cu_q, self.seq_len, self.ring_offset, self.ring_k[l],
                               self.ring_v[l], 1, stream)

    def enqueue(self, append: bool = False, waits: dict | None = None, paging_tail=None):
        """Enqueue one pass on the current stream (used for capture and for eager runs). With
        append, every layer first writes the block's own K/V rows (block KV append inside the
        graph); without, they are a precondition of the pass. `waits` maps a layer index, or
        "accept", to an event the chain waits for before that kernel (inputs still arriving).
        `paging_tail`, if given, is called on the paging stream after the last page-in and
        returns an event the acceptance waits for."""
        waits = dict(waits or {})
        main = torch.cuda.current_stream(self.dev)
        events = {}
        joins = {}
        if not self.all_resident:
            # Residency and page-in run on a side stream beside the window layers. A full layer
            # must not start before its own page-in, but every cross-stream wait in the layer
            # chain costs the overlap of one kernel launch, so the chain joins the side stream
            # only at the full layers join_points() names, each time for a group of page-ins.
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                vfy.vfy_select_resident(self.ctx, self.scores, self.cu_chunks, 1, self.n_chunks, self.k,
                                        self.slot_of_chunk, self.res_ids, self.res_slots, self.cu_res,
                                        self.pagein_list, self.pagein_count, self.side)
                for i, l in enumerate(self.full_layers):
                    vfy.vfy_set_pagein_ctas(self.ctx, PAGEIN_CTAS_FIRST if i == 0 else PAGEIN_CTAS_REST)
                    vfy.vfy_page_in(self.ctx, self.host_k[l], self.host_v[l], self.n_chunks, self.pool_k[l],
                                    self.pool_v[l], self.k, self.pagein_list, self.pagein_count, 1, self.k,
                                    self.side)
                    ev = torch.cuda.Event()
                    ev.record(self.side)
                    events[l] = ev
                vfy.vfy_set_pagein_ctas(self.ctx, 0)
                if paging_tail is not None:
                    waits["accept"] = paging_tail()
            joins = join_points(len(self.full_layers))
        fi = 0
        for l in range(self.n_layers):
            if l in waits:
                main.wait_event(waits[l])
            if is_full_layer(l):
                if fi in joins:
                    main.wait_event(events[self.full_layers[joins[fi]]])
                if append:
                    self.append_layer(l, main)
                self.attend_full_layer(l, main)
                fi += 1
            else:
                if append:
                    self.append_layer(l, main)
                self.attend_swa_layer(l, main)
        if "accept" in waits:
            main.wait_event(waits["accept"])
        vfy.vfy_accept(self.ctx, self.logits, self.vocab, self.drafts, self.cu_rows, self.q, self.accepted,
                       self.bonus, self.committed, 1, main)
        if not self.all_resident:
            main.wait_stream(self.side)

    def enqueue_end_to_end(self, in_host: torch.Tensor, out_host: torch.Tensor, front_layers: int = 4):
        """One step from pinned host memory: copy the step's inputs (the image of self.inputs in
        in_host) to the device, run the pass, and copy its results back to out_host. The scores
        and the first `front_layers` layers' queries go first on the current stream; the other
        queries follow on a copy stream while the first layers run. The logits and drafts, which
        only the acceptance reads, go on the paging stream after the last page-in, so that they
        do not share the host link with the page-ins. The chain waits for each part only where it
        needs it."""
        main = torch.cuda.current_stream(self.dev)
        split_q = self.input_offsets["q"] + front_layers * self.q_layer_bytes
        split_l = self.input_offsets["logits"]
        n = self.inputs.numel()
        self.inputs[:split_q].copy_(in_host[:split_q], non_blocking=True)
        self.copy.wait_stream(main)
        with torch.cuda.stream(self.copy):
            self.inputs[split_q:split_l].copy_(in_host[split_q:split_l], non_blocking=True)
            ev_q = torch.cuda.Event()
            ev_q.record(self.copy)

        def logits_after_paging():
            self.inputs[split_l:n].copy_(in_host[split_l:n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream(self.dev))
            return ev

        self.enqueue(waits={front_layers: ev_q}, paging_tail=logits_after_paging)
        out_host.copy_(self.results, non_blocking=True)

    def capture_end_to_end(self, in_host: torch.Tensor, out_host: torch.Tensor):
        """Capture enqueue_end_to_end as a graph (returned); the pass graph itself is unchanged."""
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                self.enqueue_end_to_end(in_host, out_host)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        return graph

    def capture(self, append: bool = False):
        """Capture the pass as self.graph (with append, the variant that appends the block's
        K/V rows in every layer; its kernel count goes to kernels_per_pass_append)."""
        # one eager pass first (also sets kernel attributes outside capture)
        self.set_step_scores(self.step)
        self.enqueue(append)
        torch.cuda.synchronize(self.dev)
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        n0 = vfy.vfy_launch_count(self.ctx)
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                self.enqueue(append)
        if append:
            self.kernels_per_pass_append = vfy.vfy_launch_count(self.ctx) - n0
            torch.cuda.current_stream(self.dev).wait_stream(s)
            torch.cuda.synchronize(self.dev)
            return graph
        self.graph = graph
        self.kernels_per_pass = vfy.vfy_launch_count(self.ctx) - n0
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        self.step = 1

    def replay(self):
        self.graph.replay()

    def close(self):
        self.graph = None
        self.ctx.close()
