#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify pass on GB300.

Workload: one verify step at 256K context with a 16-token draft, the 40-layer pass of the
Laguna XS 2.1 shape (16 q-heads / 4 KV heads x 128; 30 window layers over a 2048-slot ring,
10 full layers over an 8K-token resident pool of 4096 64-token chunks, 16 chunks paged in from
pinned host memory per step; greedy acceptance over 17 x 131072 fp32 logits at a 56% draft match
rate), captured once as a CUDA graph and replayed. Inputs are synthetic and seeded.

One JSON line on stdout (rank 0):
  metric/unit   verify-attention microseconds per layer (lower is better), whole pass / 40 layers,
                KV GB/s and the fraction of measured HBM bandwidth reported beside it
  value         device time of the graph replay; between steps the L2 is flushed by writing a
                256 MiB buffer and then reading it back, so each step starts with an L2 that
                holds none of its inputs and no dirty lines
  e2e           the same, with the step's inputs copied host->device from pinned memory and the
                accepted tokens copied back inside the timed region
  kernels       per kernel of the pass (window attention, full attention + combine, acceptance):
                launches per pass, device time per launch in a chain of its own launches (CUDA
                events around one graph replay of that chain, L2 flushed before it), algorithmic
                bytes per launch, GB/s, fraction of HBM, share of the pass
  roofline      the kernels entry with the largest share of the pass
  cpu_baseline  the fp64 CPU oracle on a bounded sample, one host core
Multi-GPU (torchrun): replicas only, one pass per GPU, no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-attn µs/layer and KV GB/s (% of HBM peak) at 256K ctx, 16-token draft"
UNIT = "us/layer"
FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts the L2 (129 MB) between timed steps: write a buffer twice its size, then (clean)
    read it back with a reduction. The write alone would leave the L2 full of dirty lines whose
    write-back then falls inside the next timed region (about 129 MB of HBM writes, 19 us at
    full bandwidth); the read evicts them before the timing starts."""

    def __init__(self, nbytes: int, clean: bool = True, buf=None):
        import torch
        self.buf = buf if buf is not None else torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        self.out = torch.empty((), dtype=torch.float32, device="cuda")
        self.clean = clean

    def __call__(self):
        import torch
        self.buf.zero_()
        if self.clean:
            torch.sum(self.buf, 0, out=self.out)

    def dirty(self) -> "L2Flush":
        """The same buffer, write-only (the L2 left full of dirty lines)."""
        return L2Flush(0, clean=False, buf=self.buf)
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the all-resident and per-kernel points")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host copies) measurement")
    ap.add_argument("--oracle-sample", type=float, default=0.0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-steps", default="", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------------
# Distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------------

def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_setup(backend):
    import torch.distributed as dist
    rank, local, world = dist_info()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return rank, local, world


def dist_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_us_per_layer(ms_per_step_max: float, layers: int, n_gpus: int) -> float:
    """Whole-job time per layer: all ranks' layers in the slowest rank's time."""
    return ms_per_step_max * 1000.0 / (layers * n_gpus)


# ---------------------------------------------------------------------------------------------
# Clocks
# ---------------------------------------------------------------------------------------------

def start_clock_sampler(device_index: int, path: str):
    import torch
    ident = str(device_index)
    try:
        uuid = torch.cuda.get_device_properties(device_index).uuid
        ident = "GPU-" + str(uuid)
    except Exception:
        pass
    try:
        f = open(path, "w")
        return subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                 "-lms", "100", "-i", ident], stdout=f, stderr=subprocess.DEVNULL), f
    except Exception:
        return None, None


def stop_clock_sampler(proc, f, path):
    if proc is None:
        return None
    proc.terminate()
    try:
        proc.wait(timeout=5)
    except Exception:
        proc.kill()
    f.close()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for name, val in zip(names, parts[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# Peaks
# ---------------------------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor TFLOP/s: the measured burst figure, else the fallback (1.9 PFLOP/s)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


# ---------------------------------------------------------------------------------------------
# CPU oracle sample (one host core)
# ---------------------------------------------------------------------------------------------

def _oracle_rep_fn():
    """Build the oracle sample's inputs once and return a function that runs one repetition of
    it: one full layer (8K resident of 4096 chunks), one window layer, the residency selection,
    16 page-ins and the acceptance. It returns the seconds each part took."""
    import numpy as np

    from oracle import vfy_oracle as O
    from speculative_decode_verify_attn_gb300 import synth

    rng = np.random.default_rng(0)
    s = synth.LAGUNA
    L, q, n, k = 262144, 17, 4096, 128
    rot = synth.rotating_residency(rng, n, k, 16, L, q)
    scores = rot.scores(1)
    prev = np.full(n, -1)
    res0 = O.select_resident(rot.scores(0), [0, n], k, prev)
    pool_k = synth.normal_bf16(rng, (k, s.num_kv_heads, 64, s.head_dim))
    pool_v = synth.normal_bf16(rng, (k, s.num_kv_heads, 64, s.head_dim))
    host_k = synth.normal_bf16(rng, (32, s.num_kv_heads, 64, s.head_dim))
    host_v = synth.normal_bf16(rng, (32, s.num_kv_heads, 64, s.head_dim))
    ring_k = synth.normal_bf16(rng, (s.num_kv_heads, synth.RING, s.head_dim))
    ring_v = synth.normal_bf16(rng, (s.num_kv_heads, synth.RING, s.head_dim))
    phi = synth.wrapping_ring_offset(rng, L, 512 + q - 1, synth.RING)
    qb = synth.normal_bf16(rng, (q, s.num_q_heads, s.head_dim))
    targets = rng.integers(0, synth.VOCAB, q)
    logits = synth.planted_logits(rng, targets, synth.VOCAB)
    drafts = synth.drafts_matching(rng, targets, 0.56, synth.VOCAB)

    def rep() -> dict:
        a = time.perf_counter()
        res = O.select_resident(scores, [0, n], k, res0["slot_of_chunk"])
        b = time.perf_counter()
        pairs = [(c % 32, s_) for c, s_ in res["pagein"][0]]
        O.page_in(host_k, host_v, pool_k, pool_v, pairs)
        c = time.perf_counter()
        O.attend_full_seq(qb, pool_k, pool_v, res["resident_ids"], res["resident_slots"], L)
        d = time.perf_counter()
        O.attend_ring_seq(qb, ring_k, ring_v, phi, L, 512)
        e = time.perf_counter()
        O.accept(logits, drafts, [0, q])
        f = time.perf_counter()
        return dict(zip(("select", "page_in", "full", "swa", "accept"), (b - a, c - b, d - c, e - d, f - e)))

    return rep


def _pass_seconds(m: dict) -> float:
    """Scale one repetition's parts to the 40-layer pass: 10 full + 30 window layers."""
    return m["select"] + 10 * m["page_in"] + 10 * m["full"] + 30 * m["swa"] + m["accept"]


def oracle_sample_seconds(budget_s: float) -> dict:
    """Repeat the oracle sample for about budget_s (at least once); mean us per layer."""
    rep = _oracle_rep_fn()
    t = {"select": [], "page_in": [], "full": [], "swa": [], "accept": []}
    t_end = time.perf_counter() + budget_s
    reps = 0
    while reps < 1 or time.perf_counter() < t_end:
        for key, dt in rep().items():
            t[key].append(dt)
        reps += 1
    m = {key: statistics.mean(v) for key, v in t.items()}
    pass_s = _pass_seconds(m)
    return {"us_per_layer": pass_s * 1e6 / 40, "reps": reps, "parts_s": m, "pass_s": pass_s}


def run_oracle_child(budget_s: float, steps_spec: str = "", threads: int = 1) -> dict:
    """Run the oracle sample (or the reference arm's whole-pass loop, with steps_spec
    "W,K,budget") in a child process whose BLAS / OpenMP pools have `threads` threads."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__)]
    cmd += ["--oracle-steps", steps_spec] if steps_spec else ["--oracle-sample", str(budget_s)]
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
    if out.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_baseline_obj(res: dict, cores: int = 1) -> dict:
    threads = "one thread" if cores == 1 else f"{cores} BLAS threads"
    return {"value": round(res["us_per_layer"], 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"fp64 numpy oracle, {threads}: 1 full layer (128 of 4096 chunks resident, 17 queries x "
                       f"16 heads), 1 window layer, residency top-128 of 4096, 16 page-ins, accept over 17 x 131072; "
                       f"{res['reps']} repetitions, scaled to 10 full + 30 window layers per pass / 40")}


# ---------------------------------------------------------------------------------------------
# Reference arm: the oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------------------------

REFERENCE_WARMUP = (3, 5)       # the reference arm's warm-up steps: at least 3, at most 5
REFERENCE_BUDGET_S = 120.0      # timed oracle work at most (a whole pass takes seconds on one core)


def _oracle_pass_fn():
    """Build the inputs of the whole 40-layer pass once and return a function that runs one step
    of it through the oracle: residency top-128 of 4096 chunks (16 new chunks per step), the 16
    page-ins of each of the 10 full layers, the 10 full layers over their 8K-token pools, the 30
    window layers over their rings (window 512, ring 2048, wrapping) and the acceptance over
    17 x 131072 logits. The host store of each full layer holds 32 distinct chunks, which stand
    for the 4096 of the context (a page-in copies chunk id mod 32: the same bytes moved)."""
    import numpy as np

    from oracle import vfy_oracle as O
    from speculative_decode_verify_attn_gb300 import synth

    rng = np.random.default_rng(0)
    s = synth.LAGUNA
    L, q, n, k = 262144, 17, 4096, 128
    layers = list(range(40))
    full = [l for l in layers if l % 4 == 3]
    swa = [l for l in layers if l % 4 != 3]
    rot = synth.rotating_residency(rng, n, k, 16, L, q)
    hkv, d = s.num_kv_heads, s.head_dim
    pools = {l: [synth.normal_bf16(rng, (k, hkv, 64, d)), synth.normal_bf16(rng, (k, hkv, 64, d))] for l in full}
    stores = {l: (synth.normal_bf16(rng, (32, hkv, 64, d)), synth.normal_bf16(rng, (32, hkv, 64, d))) for l in full}
    rings = {l: (synth.normal_bf16(rng, (hkv, synth.RING, d)), synth.normal_bf16(rng, (hkv, synth.RING, d)))
             for l in swa}
    phi = synth.wrapping_ring_offset(rng, L, synth.WINDOW + q - 1, synth.RING)
    qs = {l: synth.normal_bf16(rng, (q, s.num_q_heads, d)) for l in layers}
    targets = rng.integers(0, synth.VOCAB, q)
    logits = synth.planted_logits(rng, targets, synth.VOCAB)
    drafts = synth.drafts_matching(rng, targets, 0.56, synth.VOCAB)
    state = {"soc": np.full(n, -1), "t": 0}

    def step() -> float:
        t0 = time.perf_counter()
        res = O.select_resident(rot.scores(state["t"]), [0, n], k, state["soc"])
        state["soc"], state["t"] = res["slot_of_chunk"], state["t"] + 1
        pairs = [(c % 32, s_) for c, s_ in res["pagein"][0]]
        for l in full:
            pools[l] = list(O.page_in(stores[l][0], stores[l][1], pools[l][0], pools[l][1], pairs))
        for l in layers:
            if l in pools:
                O.attend_full_seq(qs[l], pools[l][0], pools[l][1], res["resident_ids"], res["resident_slots"], L)
            else:
                O.attend_ring_seq(qs[l], rings[l][0], rings[l][1], phi, L, synth.WINDOW)
        O.accept(logits, drafts, [0, q])
        return time.perf_counter() - t0

    return step


def oracle_pass_steps(warm: int, steps: int, budget_s: float) -> dict:
    """The reference arm's loop, in one process: `warm` untimed whole-pass steps, then up to
    `steps` timed ones, stopping early once budget_s of timed work has run (at least one step).
    Returns every timed step's seconds."""
    step = _oracle_pass_fn()
    for _ in range(warm):
        step()
    secs = []
    t0 = time.perf_counter()
    while len(secs) < steps and (not secs or time.perf_counter() - t0 < budget_s):
        secs.append(step())
    return {"warmup": warm, "steps": len(secs), "step_s": secs, "timed_s": time.perf_counter() - t0}


def run_reference(args):
    rank, local, world = dist_info()
    if rank != 0:
        return 0
    warm = min(max(args.warmup, REFERENCE_WARMUP[0]), REFERENCE_WARMUP[1])
    steps = max(1, args.steps)
    t0 = time.perf_counter()
    res = run_oracle_child(0.0, f"{warm},{steps},{REFERENCE_BUDGET_S}")
    wall = time.perf_counter() - t0
    secs = res["step_s"]
    ms_per_step = 1000.0 * statistics.mean(secs)
    value = ms_per_step * 1000.0 / 40
    sample = ("fp64 numpy oracle, one thread; each step is the whole 40-layer pass: residency top-128 of 4096, "
              "16 page-ins into each of 10 pools, 10 full layers (128 of 4096 chunks resident, 17 queries x 16 heads), "
              "30 window layers, accept over 17 x 131072")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": res["steps"], "warmup": res["warmup"],
            "ms_per_step": round(ms_per_step, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "verify pass, 256K context, 16-token draft, 10 full (8K pool) + 30 window layers "
                                   "(fp64 oracle on the host cores, whole pass per step)",
                       "steps_requested": args.steps, "timed_budget_s": REFERENCE_BUDGET_S,
                       "timed_s": round(res["timed_s"], 2), "wall_s": round(wall, 2)},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------------

def event_time_graph(graph, flush, steps, pre=None):
    """Mean / median device time (ms) of graph replays, L2 flushed (`flush()`) before each."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if pre is not None:
            pre(i)
        flush()
        starts[i].record()
        graph.replay()
        ends[i].record()
    torch.cuda.synchronize()
    ts = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return statistics.mean(ts), statistics.median(ts), ts


PROFILES = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles")
CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "speculative_decode_verify_attn_gb300", "csrc")
NOMINAL_HBM_GBS = 7900.0        # GB300 HBM3e, nominal (context beside the measured peak)


def profiled_traffic(profile: str, source: str):
    """DRAM bytes per launch of a kernel from its committed ncu summary (profiles/<profile>, the
    lines "traffic_bytes: N" and "source_sha256_16: H"), or None when csrc/<source> differs from
    the source the counters were taken on."""
    import hashlib
    try:
        text = open(os.path.join(PROFILES, profile)).read()
        fields = dict(line.split(": ", 1) for line in text.splitlines()
                      if line.startswith(("traffic_bytes: ", "source_sha256_16: ")))
        src = hashlib.sha256(open(os.path.join(CSRC, source), "rb").read()).hexdigest()[:16]
        if fields.get("source_sha256_16", "").strip() != src:
            return None
        return int(fields["traffic_bytes"])
    except (OSError, KeyError, ValueError):
        return None


def chain_points(vp, flush, steps, peak, peak_kind):
    """Per-kernel device time in a chain of the kernel's own launches, as the pass runs them
    (programmatic dependent launch between neighbours, one CUDA graph): the pass's 30 window
    layers alone, its 10 full layers alone (attention + combine each), and 8 acceptances over 8
    distinct 17 x 131072 logit buffers (71 MB, so each reads HBM after the flush). CUDA events
    around each replay on the replaying stream, L2 flushed before it; time per launch = replay
    time / launches. Each entry: algorithmic bytes per launch, GB/s, fraction of the HBM peak,
    and its share of the pass (launches per pass x time per launch over the sum)."""
    import torch

    from speculative_decode_verify_attn_gb300 import vfy
    sz = vp.sizes()

    def swa_chain():
        for l in vp.swa_layers:
            vp.attend_swa_layer(l)

    def full_chain():
        for l in vp.full_layers:
            vp.attend_full_layer(l)

    n_acc = 8
    logit_bufs = [vp.logits.clone() for _ in range(n_acc)]

    def accept_chain():
        for lg in logit_bufs:
            vfy.vfy_accept(vp.ctx, lg, vp.vocab, vp.drafts, vp.cu_rows, vp.q, vp.accepted, vp.bonus, vp.committed, 1)

    n0 = vfy.vfy_launch_count(vp.ctx)
    g_full = capture(full_chain)
    full_kernels = (vfy.vfy_launch_count(vp.ctx) - n0) // 2 // len(vp.full_layers)   # eager run + capture
    out = {}
    for name, fn, launches, per_pass, nbytes, kernel, profile in (
            ("window_attention", swa_chain, len(vp.swa_layers), len(vp.swa_layers), sz.bytes_swa,
             "attend_kernel<128,true,true,false> (window 512 in a 2048-slot ring, splits merged in a cluster)",
             "attend_swa_window512.md"),
            ("full_attention", None, len(vp.full_layers), len(vp.full_layers), sz.bytes_full,
             f"attend_kernel<128,false,...> + its split merge (8K resident of 256K; {full_kernels} kernel(s) a layer)",
             "attend_full_8k_resident.md"),
            ("accept", accept_chain, n_acc, 1, sz.bytes_accept,
             "accept_kernel<true> (argmax + greedy acceptance, 17 x 131072 fp32)", "accept_17x131072.md")):
        g = g_full if fn is None else capture(fn)
        mean_ms, med_ms, _ = event_time_graph(g, flush, steps)
        del g
        us = mean_ms * 1000.0 / launches
        gbs = nbytes / (us * 1e-6) / 1e9
        src = "accept.cu" if name == "accept" else "attend.cu"
        out[name] = {"kernel": kernel, "launches_per_pass": per_pass, "us_per_launch": round(us, 3),
                     "chain_launches": launches, "algorithmic_bytes": nbytes, "achieved": round(gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                     "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4), "peak_kind": peak_kind,
                     "traffic": profiled_traffic(profile, src)}
    del g_full, logit_bufs
    total = sum(e["us_per_launch"] * e["launches_per_pass"] for e in out.values())
    for e in out.values():
        e["pass_share"] = round(e["us_per_launch"] * e["launches_per_pass"] / total, 4)
    return out


def prefill_shaped_point(vp, flush, local, rank, steps, tf_peak):
    """A 1024-query block (a prefill-sized batch through the pool) over one full layer of the
    pass: the same 128 resident chunks at 256K context, the block at the end of the context.
    Tensor-bound: useful flops = 4 per attended (row, key) pair and head dimension (S = Q K^T
    and P V, 2 flops per multiply-add), counted exactly from the resident list."""
    import numpy as np
    import torch

    from speculative_decode_verify_attn_gb300 import passes, synth, vfy
    s = synth.LAGUNA
    QB = 1024
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rank + 21)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=1, max_queries_per_seq=QB,
                         max_splits=16, device=local)
    q = torch.randn((QB, s.num_q_heads, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((QB, s.num_q_heads), dtype=torch.float32, device="cuda")
    cu_q = torch.tensor([0, QB], dtype=torch.int32, device="cuda")
    l = vp.full_layers[0]

    def layer():
        vfy.vfy_attend_full(ctx, q, cu_q, vp.pool_k[l], vp.pool_v[l], vp.k, vp.res_ids, vp.res_slots, vp.cu_res,
                            vp.k, vp.seq_len, out, lse, 1)

    g = capture(layer)
    mean_ms, _, _ = event_time_graph(g, flush, steps)
    del g
    ctx.close()
    ids = vp.res_ids.cpu().numpy().astype(np.int64)
    L = vp.L
    pos = (ids[:, None] * passes.CHUNK + np.arange(passes.CHUNK)[None, :]).ravel()
    pos = np.sort(pos[pos < L])
    p_i = L - QB + np.arange(QB)
    pairs = int(np.searchsorted(pos, p_i, side="right").sum())     # attended (query, key) pairs
    flops = pairs * s.num_q_heads * s.head_dim * 4
    tf = flops / (mean_ms * 1e-3) / 1e12
    return {"queries": QB, "resident_chunks": int(vp.k), "us": round(mean_ms * 1000, 2), "useful_gflop": round(flops / 1e9, 2),
            "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / tf_peak, 4) if tf_peak else None}


def depth_policy_point(flush, local, rank, steps):
    """Confidence-gated draft depths against a fixed depth on the ragged batch (8 sequences,
    contexts on [4000, 200000], 16 q / 4 KV heads x 128). Per-sequence acceptance probabilities
    are drawn from Beta(2.8, 2.2) (mean 0.56, the pages' acceptance rate). The fixed policy drafts
    8 tokens per sequence (72 verify rows); the gated one spends the same 72 rows by
    vfy_gate_depths. Expected committed tokens per step: 1 + c + ... + c^D per sequence. The
    verify step is timed on the kernels: one all-resident global layer and one window layer for
    each depth vector, scaled to 12 global + 36 window layers."""
    import numpy as np
    import torch

    from speculative_decode_verify_attn_gb300 import synth, vfy
    w = synth.workload_ragged(0)
    s = w.shape
    B = w.num_seqs
    rng = np.random.default_rng(rank + 31)
    conf = rng.beta(2.8, 2.2, B).astype(np.float32)
    fixed = [8] * B
    budget = sum(d + 1 for d in fixed)
    gated = vfy.vfy_gate_depths(conf, budget, synth.DRAFT)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rank + 31)
    n_per = [(L + 63) // 64 for L in w.seq_lens]
    total = sum(n_per)
    kp = torch.randn((total, s.num_kv_heads, 64, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    vp_ = torch.randn_like(kp)
    kr = torch.randn((B, s.num_kv_heads, synth.RING, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    vr = torch.randn_like(kr)
    i32 = lambda a: torch.tensor(np.asarray(a, dtype=np.int32), dtype=torch.int32, device="cuda")
    ids = i32(np.concatenate([np.arange(n) for n in n_per]))
    slots = i32(rng.permutation(total))
    cu_res = i32(np.concatenate([[0], np.cumsum(n_per)]))
    seq_len = i32(w.seq_lens)
    phis = i32([synth.wrapping_ring_offset(rng, L, synth.WINDOW + 16, synth.RING) for L in w.seq_lens])
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, max_seqs=B, max_queries_per_seq=synth.DRAFT + 1,
                         device=local)
    out = {"sequences": B, "confidence_mean": round(float(conf.mean()), 3), "row_budget": budget}
    for name, depths in (("fixed", fixed), ("gated", gated)):
        qs = [d + 1 for d in depths]
        cu_q = i32(np.concatenate([[0], np.cumsum(qs)]))
        q = torch.randn((sum(qs), s.num_q_heads, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((sum(qs), s.num_q_heads), dtype=torch.float32, device="cuda")
        g_full = capture(lambda: vfy.vfy_attend_full(ctx, q, cu_q, kp, vp_, total, ids, slots, cu_res, max(n_per),
                                                     seq_len, o, lse, B))
        t_full, _, _ = event_time_graph(g_full, flush, steps)
        g_win = capture(lambda: vfy.vfy_attend_swa(ctx, q, cu_q, kr, vr, phis, seq_len, o, lse, B))
        t_win, _, _ = event_time_graph(g_win, flush, steps)
        del g_full, g_win
        step_us = 1000 * (12 * t_full + 36 * t_win)
        tokens = float(sum(sum(float(c) ** k for k in range(d + 1)) for c, d in zip(conf, depths)))
        out[name] = {"depths": depths, "tokens_per_step": round(tokens, 3), "step_us": round(step_us, 1),
                     "tokens_per_s": round(tokens / (step_us * 1e-6), 1)}
    out["gated_over_fixed"] = round(out["gated"]["tokens_per_s"] / out["fixed"]["tokens_per_s"], 4)
    ctx.close()
    return out


def drafter_ring_point(flush, local, rank, steps, peak):
    """The drafter's context-KV ring: the 5 layers of the drafter head attend a 4096-position
    window in an 8192-slot ring (16 proposals, 256K context, a wrapping write head), one graph.
    Bytes per layer are the attended span's K and V: (4096 + 15) x 4 heads x 128 x 2 B x 2."""
    import numpy as np
    import torch

    from speculative_decode_verify_attn_gb300 import synth, vfy
    s = synth.LAGUNA
    W, R, Q, NL = synth.DRAFTER_WINDOW, synth.DRAFTER_RING, synth.DRAFT, synth.DRAFTER_LAYERS
    L = 262144
    rng = np.random.default_rng(rank + 11)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rank + 11)
    ctx = vfy.vfy_create(s.num_q_heads, s.num_kv_heads, s.head_dim, window=W, ring_len=R, max_seqs=1,
                         max_queries_per_seq=Q, device=local)
    shape = (1, s.num_kv_heads, R, s.head_dim)
    kr = [torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16) for _ in range(NL)]
    vr = [torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16) for _ in range(NL)]
    q = torch.randn((NL, Q, s.num_q_heads, s.head_dim), generator=gen, device="cuda", dtype=torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((NL, Q, s.num_q_heads), dtype=torch.float32, device="cuda")
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    cu_q, seq_len = i32([0, Q]), i32([L])
    phi = i32([synth.wrapping_ring_offset(rng, L, W + Q - 1, R)])

    def layers():
        for l in range(NL):
            vfy.vfy_attend_swa(ctx, q[l], cu_q, kr[l], vr[l], phi, seq_len, out[l], lse[l], 1)

    g = capture(layers)
    mean_ms, _, _ = event_time_graph(g, flush, steps)
    del g
    ctx.close()
    per_layer_bytes = (W + Q - 1) * s.num_kv_heads * s.head_dim * 2 * 2 + 2 * Q * s.num_q_heads * s.head_dim * 2
    us = mean_ms * 1000
    return {"layers": NL, "window": W, "ring": R, "us": round(us, 3), "us_per_layer": round(us / NL, 3),
            "gbs": round(NL * per_layer_bytes / (mean_ms * 1e-3) / 1e9, 1),
            "frac": round(NL * per_layer_bytes / (mean_ms * 1e-3) / 1e9 / peak, 4)}


def capture(fn):
    import torch
    fn()                      # eager once (sets kernel attributes outside capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def measure_e2e(vp, flush, args, local, sz, world):
    """The pass through the C ABI from host buffers: each step copies its inputs (residency
    scores, block queries of all layers, logits, drafts) from pinned host memory, runs the pass and
    copies its results (accepted length, bonus, committed tokens) back to pinned host memory, all
    in one captured graph per step. The queries of later layers and the logits arrive on a copy
    stream while the first layers run (VerifyPass.enqueue_end_to_end)."""
    import torch
    in_host = vp.inputs.cpu().pin_memory()
    score_view = vp.scores.view(torch.uint8)
    s_off = score_view.data_ptr() - vp.inputs.data_ptr()
    score_host = [vp.score_table[t].cpu().view(torch.uint8) for t in range(vp.score_table.shape[0])]
    out_host = torch.empty(vp.results.numel(), dtype=torch.int32).pin_memory()
    h2d = in_host.numel()
    d2h = out_host.numel() * 4
    g = vp.capture_end_to_end(in_host, out_host)
    e_steps = max(20, min(args.steps, 500))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    for i in range(-3, e_steps):
        # this step's residency scores, written into the pinned input image on the host
        in_host.narrow(0, s_off, score_view.numel()).copy_(score_host[vp.step % len(score_host)])
        vp.step += 1
        flush()
        if i < 0:                      # warm-up replays
            g.replay()
            torch.cuda.synchronize()
            continue
        starts[i].record()
        g.replay()
        ends[i].record()
        ends[i].synchronize()
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
    e2e_ms = dist_max(e2e_ms, torch.device("cuda", local))
    del g
    return {"value": round(aggregate_us_per_layer(e2e_ms, sz.n_layers, world), 4), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "accepted_last_step": int(out_host[0])}


def run_ours(args):
    import torch

    import __graft_entry__
    from speculative_decode_verify_attn_gb300 import passes, synth

    rank, local, world = dist_setup("nccl" if args.gpus > 1 else "gloo")
    torch.cuda.set_device(local)
    __graft_entry__.build()
    peak, peak_kind = hbm_peak()

    wl = synth.workload_256k()
    vp = passes.VerifyPass(wl, device=local, seed=rank)
    sz = vp.sizes()
    vp.capture()
    flush = L2Flush(FLUSH_BYTES)

    # warm-up: steady-state residency (16 new chunks per step)
    for i in range(max(args.warmup, 3)):
        vp.set_step_scores(vp.step)
        vp.step += 1
        flush()
        vp.replay()
    torch.cuda.synchronize()

    def next_scores(i):
        vp.set_step_scores(vp.step)
        vp.step += 1

    clk_path = os.path.join(tempfile.gettempdir(), f"vfy_clocks_{os.getpid()}.csv")
    proc, fh = start_clock_sampler(local, clk_path)
    time.sleep(0.3)
    dist_barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    mean_ms, med_ms, ts = event_time_graph(vp.graph, flush, args.steps, pre=next_scores)
    torch.cuda.synchronize()
    dist_barrier()
    wall = time.perf_counter() - wall0
    clocks = stop_clock_sampler(proc, fh, clk_path)
    ms_max = dist_max(mean_ms, torch.device("cuda", local))
    accepted = int(vp.accepted.item())

    launches = vp.launches_per_step() * args.steps
    value = aggregate_us_per_layer(ms_max, sz.n_layers, world)
    kv_gbs = sz.bytes_pass / (mean_ms * 1e-3) / 1e9

    extras = {}
    roofline = None
    if not args.no_extras:
        # per-kernel points: one full layer, one window layer, acceptance, select + page-in
        lf, ls = vp.full_layers[0], vp.swa_layers[0]
        g_full = capture(lambda: vp.attend_full_layer(lf))
        g_swa = capture(lambda: vp.attend_swa_layer(ls))
        k_steps = max(50, min(args.steps, 500))
        f_mean, f_med, _ = event_time_graph(g_full, flush, k_steps)
        s_mean, s_med, _ = event_time_graph(g_swa, flush, k_steps)
        # per kernel, in a chain of its own launches; the roofline is the one with the largest
        # share of the pass
        kernels = chain_points(vp, flush, k_steps, peak, peak_kind)
        extras["kernels"] = kernels
        top = max(kernels, key=lambda name: kernels[name]["pass_share"])
        e = kernels[top]
        roofline = {"bound": "hbm", "kernel": f"{top}: {e['kernel']}", "achieved": e["achieved"], "peak": peak,
                    "unit": "GB/s", "frac": e["frac"], "traffic": e["traffic"],
                    "algorithmic_bytes": e["algorithmic_bytes"], "us_per_launch": e["us_per_launch"],
                    "pass_share": e["pass_share"], "peak_kind": peak_kind}
        g_layers = capture(vp.enqueue_layers)
        l_mean, _, _ = event_time_graph(g_layers, flush, k_steps)
        g_acc = capture(vp.enqueue_accept)
        c_mean, _, _ = event_time_graph(g_acc, flush, k_steps)
        g_pg = capture(vp.enqueue_paging)
        p_mean, _, _ = event_time_graph(g_pg, flush, min(k_steps, 100), pre=next_scores)
        # the pass with the block's K/V rows appended in every layer (full layers write through to
        # the pinned chunk store): block KV append inside the graph
        g_app = vp.capture(append=True)
        ap_mean, _, _ = event_time_graph(g_app, flush, k_steps, pre=next_scores)
        extras["pass_with_append"] = {"us_per_layer": round(ap_mean * 1000 / sz.n_layers, 3),
                                      "kernels": vp.kernels_per_pass_append}
        del g_app
        pg_bytes = len(vp.full_layers) * wl.pagein_per_step * vp.shape.num_kv_heads * 64 * vp.shape.head_dim * 4
        extras["layers_only_us_per_layer"] = round(l_mean * 1000 / sz.n_layers, 3)
        extras["layers_only_kv_gbs"] = round((sz.bytes_pass - sz.bytes_accept) / (l_mean * 1e-3) / 1e9, 1)
        extras["accept_us"] = round(c_mean * 1000, 3)
        extras["accept_gbs"] = round(sz.bytes_accept / (c_mean * 1e-3) / 1e9, 1)
        extras["select_plus_pagein_us"] = round(p_mean * 1000, 3)
        extras["pagein_host_gbs"] = round(pg_bytes / (p_mean * 1e-3) / 1e9, 1)
        del g_layers, g_acc, g_pg
        # one layer alone in a graph of its own (includes the graph's launch)
        extras["full_layer_us"] = round(f_mean * 1000, 3)
        extras["swa_layer_us"] = round(s_mean * 1000, 3)
        extras["swa_layer_gbs"] = round(sz.bytes_swa / (s_mean * 1e-3) / 1e9, 1)
        del g_full, g_swa
        # the all-resident 256K full layer (4096 chunks = 512 MiB of KV): the clean bandwidth point
        wl1 = synth.Workload("all-resident", synth.LAGUNA, [262144], [16], n_full=1, n_swa=3, resident_chunks=0)
        ar = passes.VerifyPass(wl1, device=local, seed=rank + 1, all_resident=True)
        g_ar = capture(lambda: ar.attend_full_layer(ar.full_layers[0]))
        a_mean, a_med, _ = event_time_graph(g_ar, flush, max(20, min(args.steps, 200)))
        a_bytes = ar.sizes().bytes_full
        extras["all_resident_256k_layer"] = {"us": round(a_mean * 1000, 2), "bytes": a_bytes,
                                             "gbs": round(a_bytes / (a_mean * 1e-3) / 1e9, 1),
                                             "frac": round(a_bytes / (a_mean * 1e-3) / 1e9 / peak, 4),
                                             "frac_of_nominal": round(a_bytes / (a_mean * 1e-3) / 1e9 /
                                                                      NOMINAL_HBM_GBS, 4)}
        # the same two graphs with the write-only flush: the L2 starts each step full of dirty lines
        dflush = flush.dirty()
        d_ar, _, _ = event_time_graph(g_ar, dflush, max(20, min(args.steps, 200)))
        d_pass, _, _ = event_time_graph(vp.graph, dflush, min(args.steps, 500), pre=next_scores)
        extras["write_only_l2_flush"] = {"pass_us_per_layer": round(d_pass * 1000 / sz.n_layers, 3),
                                         "all_resident_256k_layer_us": round(d_ar * 1000, 2)}
        del g_ar
        ar.close()
        extras["drafter_ring"] = drafter_ring_point(flush, local, rank, max(20, min(args.steps, 500)), peak)
        extras["prefill_shaped_verify"] = prefill_shaped_point(vp, flush, local, rank, max(20, min(args.steps, 200)),
                                                               bf16_peak())
        extras["depth_policy"] = depth_policy_point(flush, local, rank, max(20, min(args.steps, 100)))

    # end to end: inputs host->device from pinned memory, accepted tokens back, inside the timing
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(vp, flush, args, local, sz, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline_obj(run_oracle_child(12.0))
        except Exception as e:  # reported, not fatal
            cpu = {"error": str(e)[:200]}

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": wl.name, "seq_len": wl.seq_lens[0], "draft": wl.depths[0],
                           "layers": sz.n_layers, "full_layers": sz.n_full, "window_layers": sz.n_swa,
                           "resident_chunks": wl.resident_chunks, "pagein_per_step": wl.pagein_per_step,
                           "heads": "16q/4kv x 128", "l2": "flushed between steps (256 MiB write, then read back)",
                           "parallelism": f"replicas x{world}", "timing": "CUDA events around each graph replay"},
                "kv_gbs": round(kv_gbs, 1), "kv_frac_of_hbm": round(kv_gbs / peak, 4),
                "kv_frac_of_nominal_hbm": round(kv_gbs / NOMINAL_HBM_GBS, 4),
                "median_ms_per_step": round(med_ms, 5),
                "p90_ms_per_step": round(sorted(ts)[min(len(ts) - 1, (9 * len(ts)) // 10)], 5),
                "wall_s": round(wall, 3),
                "pass_bytes": sz.bytes_pass, "accepted_last_step": accepted,
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
                "e2e": e2e,
                "gpu_launches": launches}
        line.update(extras)
        print(json.dumps(line), flush=True)
    vp.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_steps:
        w, k, budget = args.oracle_steps.split(",")
        print(json.dumps(oracle_pass_steps(int(w), int(k), float(budget))))
        return 0
    if args.oracle_sample or "--oracle-sample" in (argv or sys.argv):
        print(json.dumps(oracle_sample_seconds(args.oracle_sample)))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
