"""Seeded synthetic inputs for the verify step, shared by the tests, the smoke check and bench.py.

This module only draws and lays out inputs; it computes none of the verify step's results
(no softmax, no top-k, no argmax). Where an input must relate to a result (drafts that match
the target's greedy tokens, residency scores with a known winner set), the relation is planted
by construction and the planted values are returned beside the inputs.

Distributions follow the workloads of the pages' long-context runs (Laguna XS 2.1 at 256K with
an 8K KVFlash pool, 64-token chunks, a 512-token window in a 2048-slot ring, 16 drafted tokens
per step; Laguna S 2.1 for the 48-layer ragged batch). Host RNG: NumPy PCG64 default_rng(seed).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CHUNK = 64


# --------------------------------------------------------------------------------------------
# bf16 as raw bits
# --------------------------------------------------------------------------------------------

def bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even; NaN stays a quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return rounded


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


# --------------------------------------------------------------------------------------------
# Residency scores
# --------------------------------------------------------------------------------------------

def gumbel_scores(rng: np.random.Generator, n: int) -> np.ndarray:
    """Gumbel(0, 1) = -ln(-ln U), U uniform on (0, 1), as fp32."""
    u = rng.random(n)
    u = np.clip(u, 1e-12, 1.0 - 1e-12)
    return (-np.log(-np.log(u))).astype(np.float32)


def block_chunks(seq_len: int, num_queries: int) -> range:
    """Chunks that hold the verify block's own positions [L - q, L - 1]."""
    return range((seq_len - num_queries) // CHUNK, (seq_len - 1) // CHUNK + 1)


def force_block_resident(scores: np.ndarray, seq_len: int, num_queries: int) -> np.ndarray:
    """Caller convention: the chunks holding the block get score +inf so they always stay."""
    scores = scores.copy()
    for c in block_chunks(seq_len, num_queries):
        scores[c] = np.inf
    return scores


@dataclass
class RotatingResidency:
    """Per-step residency scores where exactly `rotate` new chunks enter at every step.

    A hot set of (k - rotate - block chunks) chunks always wins, the block chunks are +inf, and
    step t adds group t mod len(groups) of `rotate` chunks. Consecutive groups are disjoint, so
    every step evicts the previous group and pages in the next one.
    """
    n: int
    k: int
    rotate: int
    hot: np.ndarray
    groups: np.ndarray          # [num_groups][rotate]
    base: np.ndarray            # fp32 [n] Gumbel noise
    block: np.ndarray           # block chunk indices

    def scores(self, step: int) -> np.ndarray:
        s = self.base.copy()
        s[self.hot] += np.float32(100.0)
        s[self.groups[step % len(self.groups)]] += np.float32(50.0)
        s[self.block] = np.inf
        return s

    def winners(self, step: int) -> np.ndarray:
        """The planted resident set of `step`, ascending."""
        return np.sort(np.concatenate([self.hot, self.groups[step % len(self.groups)],
                                       self.block]))


def rotating_residency(rng, n: int, k: int, rotate: int, seq_len: int, num_queries: int,
                       num_groups: int = 32) -> RotatingResidency:
    block = np.array(list(block_chunks(seq_len, num_queries)), dtype=np.int64)
    others = np.setdiff1d(np.arange(n), block)
    perm = rng.permutation(others)
    n_hot = k - rotate - len(block)
    hot = np.sort(perm[:n_hot])
    rest = perm[n_hot:]
    num_groups = min(num_groups, len(rest) // rotate)
    groups = rest[: num_groups * rotate].reshape(num_groups, rotate)
    return RotatingResidency(n, k, rotate, hot, groups, gumbel_scores(rng, n), block)


# --------------------------------------------------------------------------------------------
# Window ring
# --------------------------------------------------------------------------------------------

def wrapping_ring_offset(rng, seq_len: int, span: int, ring_len: int) -> int:
    """phi such that the last `span` positions, at slots (pos + phi) mod R, cross slot R-1 -> 0."""
    lo = seq_len - span
    while True:
        phi = int(rng.integers(0, ring_len))
        first = (lo + phi) % ring_len
        if first + span > ring_len and first != 0:
            return phi


# --------------------------------------------------------------------------------------------
# Logits and drafts
# --------------------------------------------------------------------------------------------

def normal_logits(rng, rows: int, vocab: int) -> np.ndarray:
    return rng.standard_normal((rows, vocab), dtype=np.float32)


def planted_logits(rng, targets, vocab: int) -> np.ndarray:
    """N(0,1) logits clipped to [-5, 5] with the value 6 at `targets[r]`: row r's greedy token
    is targets[r] by construction."""
    rows = len(targets)
    x = np.clip(rng.standard_normal((rows, vocab), dtype=np.float32), -5.0, 5.0)
    x[np.arange(rows), np.asarray(targets)] = 6.0
    return x


def other_token(rng, token: int, vocab: int) -> int:
    t = int(rng.integers(0, vocab - 1))
    return t + 1 if t >= token else t


def drafts_matching(rng, targets, match_prob: float, vocab: int) -> np.ndarray:
    """Drafts for a block whose target tokens are `targets` (D+1 of them): d_r = targets[r] with
    probability match_prob, independently, else a uniform token different from targets[r]."""
    depth = len(targets) - 1
    out = np.empty(depth, dtype=np.int32)
    for r in range(depth):
        out[r] = targets[r] if rng.random() < match_prob else other_token(rng, int(targets[r]), vocab)
    return out


def drafts_prefix(rng, targets, n_match: int, vocab: int) -> np.ndarray:
    """d_r = targets[r] for r < n_match, d_{n_match} != targets[n_match], the rest uniform."""
    depth = len(targets) - 1
    out = rng.integers(0, vocab, depth).astype(np.int32)
    out[:n_match] = np.asarray(targets[:n_match])
    if n_match < depth:
        out[n_match] = other_token(rng, int(targets[n_match]), vocab)
    return out


# --------------------------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


TINY = Shape(4, 1, 64)
LAGUNA = Shape(16, 4, 128)        # hidden 2048 = 16 q-heads x 128; 4 KV heads

WINDOW = 512                      # sliding-window width (positions, including self)
RING = 2048                       # ring slots
DRAFT = 16                        # drafted tokens per step
POOL_CHUNKS = 128                 # 8K-token resident pool = 128 chunks of 64
VOCAB = 131072
# The drafter's context-KV ring ('Laguna XS 2.1 33B on a RTX 3090', 'Three optimizations' item 2:
# a feature window of up to 4K tokens, a position-indexed ring; 'The model ...': a 5-layer head
# proposing 16 tokens). The pages give no drafter head counts: the target's 16 q / 4 KV x 128
# are reused. The ring holds twice the window.
DRAFTER_WINDOW = 4096
DRAFTER_RING = 8192
DRAFTER_LAYERS = 5


@dataclass
class Workload:
    """A named workload: shapes and sizes only."""
    name: str
    shape: Shape
    seq_lens: list
    depths: list                  # drafted tokens per sequence (queries = depth + 1)
    n_full: int = 0               # full-attention layers per pass
    n_swa: int = 0                # window layers per pass
    resident_chunks: int = POOL_CHUNKS   # 0 = every chunk resident
    pagein_per_step: int = 0
    vocab: int = VOCAB
    notes: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens)

    @property
    def queries(self) -> list:
        return [d + 1 for d in self.depths]


def workload_256k() -> Workload:
    """40-layer verify pass at 256K context: 10 full layers over a 128-chunk resident pool out of
    4096 chunks (16 paged in per step), 30 ring layers, accept over 17 x 131072 logits."""
    return Workload("verify pass, 256K context, 16-token draft, 10 full (8K pool) + 30 window layers",
                    LAGUNA, [262144], [DRAFT], n_full=10, n_swa=30, resident_chunks=POOL_CHUNKS,
                    pagein_per_step=16)


def workload_ragged(seed: int = 0) -> Workload:
    """8 sequences, contexts uniform on [4000, 200000], depths from {2, 4, 8, 11, 16}; 48 layers
    (36 window + 12 full, every chunk resident)."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(4000, 200001, 8)]
    depths = [int(x) for x in rng.choice([2, 4, 8, 11, 16], 8)]
    return Workload("ragged batch of 8, contexts 4K-200K, depths {2,4,8,11,16}, 12 full + 36 window",
                    LAGUNA, lens, depths, n_full=12, n_swa=36, resident_chunks=0)
