// Verify attention on sm_103a: split-KV flash-decode with TMA-staged bf16 K/V tiles, tcgen05
// tensor-core tiles for S = Q K^T and O += P V (fp32 accumulators in tensor memory), an fp32
// online softmax, and the splits merged either in a thread-block cluster (distributed shared
// memory) or by a combine kernel.
//
// Sources ("Laguna XS 2.1 33B on a RTX 3090" (lucebox)):
//  - "The model, fast MoE with a drafter in the box": the 16 drafted tokens and the last committed
//    token are verified in one batched target forward. Here the q = D + 1 block queries of one
//    KV head's G q-heads form q * G <= 128 rows, the M = 128 side of one tcgen05 MMA.
//  - "Three optimizations", item 1: full layers read a pool of 64-token chunks, of which a resident
//    subset is on the GPU. Each resident chunk is one 64-token tile, fetched by TMA from its slot.
//  - item 3: window layers attend a 512-token window kept in a 2048-slot position ring. The ring
//    tiles are 64-slot aligned, so a tile never crosses the ring's end.
//
// One CTA handles one (sequence b, KV head h, split s): a contiguous run of tiles. Warp roles:
//   warps 0-7  load Q, then the masked online softmax and the epilogue. Warps w and w + 4 share
//              TMEM lane quarter w % 4 (one row per lane); warpgroup h takes the second or first
//              half of every tile's keys and keeps its own running maximum, row sum and O
//              accumulator (O_h += P_h V_h), so the two halves never wait on each other; they are
//              merged once, in the epilogue. A tile is two 64-token chunks (one per warpgroup) in
//              full layers whose splits hold at least 8 chunks, and one chunk (32 keys per
//              warpgroup) otherwise: short splits and merging launches are latency-bound. Warp 2
//              also relays each tile's V to the issuer through its arrival on the tile's P barrier.
//   warp 8     TMA producer of K tiles (a ring of smem stages, released when S has read them) and
//              of the tile geometry the softmax needs (a ring of its own)
//   warp 9     TMA producer of V tiles (a ring released when P.V has read them)
//   warp 10    TMEM owner and MMA issuer (one lane)
// Row r = i * G + g (query i, q-head g of the group) sits in TMEM lane r for r < 64, lane r + 32 for
// 64 <= r < 96 and lane r - 32 above: lane quarter 2 holds rows only in blocks of more than 96.
// Warps are spread over the SM's four sub-partitions by warp index mod 4, so the softmax warps of
// quarter 2 (warps 2 and 6) then have nothing to compute, and the MMA issuer, warp 10, has its
// sub-partition to itself: tcgen05.mma issue blocks while the tensor pipe is busy, so the
// tensor core idles whenever that thread waits for an issue slot.
#include <cuda_bf16.h>

#include <type_traits>

#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kVProducerWarp = 9;
constexpr int kMmaWarp = 10;
constexpr int kVRelayWarp = 2;    // softmax warp of TMEM lane quarter 2: tile rows 96-127
constexpr int kGeo = 16;          // tile-geometry ring: at least the K stages plus the S buffers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // two O accumulators (one per warpgroup) of d columns, 128 apart
constexpr uint32_t kColS = 256;   // S buffers of one column per key; warpgroup h writes its P (bf16,
                                  // two per column) over the first half of its own S columns
constexpr int kPrefetch = 6;      // tiles prefetched into L2 beyond the shared-memory stages
// A row keeps a stale reference maximum until a tile's maximum exceeds it by this much (log2
// units); then O and l are rescaled. The result is exact either way: O and l share the reference.
constexpr float kRescaleLog2 = 8.0f;
constexpr int kBarsBytes = 4096;  // shared memory reserved for the barrier block (Bars)

// MERGE: the splits of one (b, h) form a cluster and merge in the kernel. Every CTA then keeps a
// receive area where the other splits store their partial rows: for the block rows it owns (rows
// rank, rank + n, ...; slot k holds row rank + n k) one fp32 (m, l) pair and one bf16 O row
// (normalised by l) per split, at index k * n + split. k * n + split < kMaxRows + n, so
// kMaxRows + kMaxClusterSplits entries cover every cluster size. A merging CTA processes few
// tiles, so it takes fewer K/V stages. Sending the rows as bf16 halved what the merge moves
// (window layers 7.50 -> 7.30 us in their chain; the rounding, about 2^-9 of a partial, stays far
// inside the attention tolerance), and sending them straight from the softmax threads' registers,
// with no staging in shared memory and no barrier before the sends, 7.09 -> 6.68 us.
template <int HD, bool RING, bool MERGE, bool WIDE>
struct Cfg {
  static_assert(!WIDE || (!RING && !MERGE), "wide tiles are for full layers without the cluster merge");
  static constexpr int kCPT = WIDE ? 2 : 1;             // 64-token chunks per tile
  static constexpr int kKT = kCPT * kChunk;             // keys per tile
  static constexpr int kKH = kKT / 2;                   // keys per warpgroup half
  static constexpr int kSBufs = kCPT == 2 ? 2 : 3;      // S issued up to kSBufs - 1 tiles ahead
  static constexpr int kBoxes = HD / 64;               // 128-byte (64-column) boxes per row
  static constexpr int kBoxBytes = kKT * 128;          // one box: a tile's rows, 128 bytes each
  static constexpr int kChunkRowsBytes = kChunk * 128; // one chunk's rows within a box
  static constexpr int kQBoxBytes = kMaxRows * 128;
  static constexpr int kQBytes = kMaxRows * HD * 2;
  static constexpr int kTileBytes = kKT * HD * 2;
  static constexpr int kChunkBytes = kChunk * HD * 2;
  // K and V stage rings. A K stage frees as soon as S has read it, a V stage only after P.V, a
  // tile later; with wide tiles V gets the extra stage so that its loads start as far ahead.
  static constexpr int kKStages = WIDE ? (HD == 128 ? 2 : 4) : (HD == 128 ? (MERGE ? 3 : 6) : 8);
  static constexpr int kVStages = WIDE ? (HD == 128 ? 3 : 5) : (HD == 128 ? (MERGE ? 3 : 5) : 8);
  static_assert(kKStages <= 8 && kVStages <= 8 && kKStages + kSBufs <= kGeo, "rings");
  static_assert(kColS + kSBufs * kKT <= kTmemCols, "tensor memory");
  static constexpr int kRecvEntries = kMaxRows + kMaxClusterSplits;
  static constexpr int kRecvOffset = kQBytes + (kKStages + kVStages) * kTileBytes;
  static constexpr int kRecvMlOffset = kRecvOffset + (MERGE ? kRecvEntries * HD * 2 : 0);
  static constexpr int kBarOffset = kRecvMlOffset + (MERGE ? kRecvEntries * 8 : 0);
  static constexpr int kSmemBytes = kBarOffset + kBarsBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct Bars {
  uint64_t k_full[8];
  uint64_t v_full[8];
  uint64_t k_empty[8];
  uint64_t v_empty[8];
  uint64_t geo_full[kGeo];  // tile j's geometry is in entry j % kGeo
  uint64_t s_full[3];
  uint64_t p_full[3];     // [S buffer]: both warpgroups' P of the tile (every softmax thread arrives)
  uint64_t o_full[2][2];  // [warpgroup][tile parity]: one phase per P.V MMA of that parity (waited on
                          // before rescaling O_h)
  uint64_t o_done;     // one phase, after the last P.V MMA (the epilogue waits on it)
  uint64_t q_ready;
  uint64_t drain;
  uint64_t never;       // no thread ever arrives: the timeout test's wait
  uint64_t xchg_l[4];   // per lane quarter: the two halves' (m, l) at the end
  uint32_t tmem_base;
  int abort;
  int tile_base[kGeo][2];  // per tile (j % kGeo) and chunk: what the mask needs (written by the K
  int tile_valid[kGeo][2]; // producer before it arrives on geo_full, read by the softmax after)
  int tile_zero[kGeo];     // some key of the tile lies outside every query's range
  float xm[2][128];       // [warpgroup][TMEM lane]
  float xl[2][128];
  float2 sml[128];        // cluster merge: this split's (m, l) per block row
};
static_assert(sizeof(Bars) <= kBarsBytes, "barrier block overflows its reservation");

// The per-CTA work item.
struct Work {
  int b, h, s;
  int q0, nq;
  int rt, row0;    // row tile: block rows [row0, row0 + rows) of the sequence's q * G
  int rows;
  int L;
  int tb, nt;      // first tile (index within the (b, h) tile list) and number of tiles
  int r0;          // full: resident-list offset of sequence b
  int nres;        // full: resident chunks of sequence b
  int lo, span;    // ring: first attended position of the tile's rows and the union span length
  int s_lo;        // ring: slot of position lo
  bool bad;        // the sequence's q or L is out of range: it is skipped
};

template <bool RING, int CPT>
__device__ __forceinline__ Work make_work(const AttnParams& p) {
  Work w;
  // A verify block is one row tile: no integer division on the path to the first load.
  w.b = p.row_tiles == 1 ? static_cast<int>(blockIdx.z) : static_cast<int>(blockIdx.z) / p.row_tiles;
  w.rt = static_cast<int>(blockIdx.z) - w.b * p.row_tiles;
  w.row0 = w.rt * kMaxRows;
  w.h = blockIdx.y;
  w.s = blockIdx.x;
  // Every per-sequence value is loaded at once (one round trip to memory before the first tile
  // can be addressed); all of them are in bounds for every b < B.
  const int cq0 = p.cu_q[w.b], cq1 = p.cu_q[w.b + 1], len = p.seq_len[w.b];
  const int cr0 = RING ? 0 : p.cu_res[w.b];
  const int cr1 = RING ? 0 : p.cu_res[w.b + 1];
  const int roff = RING ? p.ring_off[w.b] : 0;
  w.q0 = cq0;
  w.nq = cq1 - cq0;
  w.L = len;
  w.tb = 0;
  w.nt = 0;
  w.r0 = 0;
  w.nres = 0;
  w.lo = 0;
  w.span = 0;
  w.s_lo = 0;
  w.bad = w.nq < 0 || w.nq > p.max_q || w.L < w.nq || w.q0 < 0;
  if (w.bad) {
    w.nq = 0;
    w.rows = 0;
    return w;
  }
  w.rows = min(kMaxRows, max(0, w.nq * p.group - w.row0));
  if (w.rows == 0) return w;                     // a row tile past this sequence's block
  int n_tiles;
  if (!RING) {
    w.r0 = cr0;
    w.nres = max(0, cr1 - cr0);
    n_tiles = (w.nres + CPT - 1) / CPT;
  } else {
    // Unsigned 32-bit arithmetic on the way to the first load: lo < 2^31 and phi < R <= 2^31, so
    // lo + phi fits.
    const int R = p.ring_len;
    const unsigned phi = static_cast<unsigned>(roff % R + R) % static_cast<unsigned>(R);
    // The tile's queries are i in [row0 / G, (row0 + rows - 1) / G], at positions L - nq + i.
    const bool whole = p.row_tiles == 1;               // then the tile is the whole block
    const int i_first = whole ? 0 : w.row0 / p.group;
    const int i_last = whole ? w.nq - 1 : (w.row0 + w.rows - 1) / p.group;
    w.lo = max(0, w.L - w.nq + i_first - p.window + 1);
    w.span = w.L - w.nq + i_last + 1 - w.lo;
    w.s_lo = static_cast<int>((static_cast<unsigned>(w.lo) + phi) % static_cast<unsigned>(R));
    n_tiles = w.span > 0 ? ((w.s_lo & (kChunk - 1)) + w.span + kChunk - 1) / kChunk : 0;
  }
  // (s + 1) * n_tiles < 64 * 2^26: unsigned 32-bit division
  const unsigned ns = static_cast<unsigned>(p.num_splits);
  w.tb = static_cast<int>((static_cast<unsigned>(w.s) * static_cast<unsigned>(n_tiles)) / ns);
  w.nt = static_cast<int>((static_cast<unsigned>(w.s + 1) * static_cast<unsigned>(n_tiles)) / ns) - w.tb;
  return w;
}

// Geometry of chunk c of tile j: the TMA row coordinate of its first token, and what the mask
// needs.
struct Tile {
  int y;          // row of the 2-D [rows][d] view of the pool / ring
  int base;       // full: position of token 0; ring: offset (from s_lo, mod R) of slot 0
  bool valid;     // full: slot and chunk id in range
  bool present;   // full: the sequence has this chunk (the last tile may hold one chunk only)
};

template <bool RING, int CPT>
__device__ __forceinline__ Tile tile_at(const AttnParams& p, const Work& w, int j, int c) {
  Tile t;
  t.present = true;
  if (!RING) {
    const int e = (w.tb + j) * CPT + c;
    t.present = e < w.nres;
    const int idx = w.r0 + (t.present ? e : 0);
    const int cid = t.present ? p.res_ids[idx] : -1;
    const int slot = t.present ? p.res_slots[idx] : -1;
    t.valid = t.present && cid >= 0 && cid < (1 << 25) && slot >= 0 && slot < p.num_slots;
    t.y = (t.valid ? (slot * p.hkv + w.h) : w.h) * kChunk;
    t.base = t.valid ? cid * kChunk : 0;
  } else {
    const int R = p.ring_len;
    const unsigned tiles_per_ring = static_cast<unsigned>(R / kChunk);
    const int ti = static_cast<int>(static_cast<unsigned>(w.s_lo / kChunk + w.tb + j) % tiles_per_ring);
    t.valid = true;
    t.y = ((w.b * p.hkv + w.h) * R) + ti * kChunk;
    const int d = ti * kChunk - w.s_lo;                // in (-R, R)
    t.base = d < 0 ? d + R : d;
  }
  return t;
}

// Is key k of the tile at a position some block query attends (inside the union span)?
template <bool RING>
__device__ __forceinline__ bool key_in_union(const AttnParams& p, const Work& w, const Tile& t, int k,
                                             int* pos_out) {
  if (!RING) {
    const int pos = t.base + k;
    *pos_out = pos;
    return t.valid && pos < w.L;
  } else {
    int off = t.base + k;
    if (off >= p.ring_len) off -= p.ring_len;
    *pos_out = w.lo + off;
    return off < w.span;
  }
}

// Does some key of the tile lie outside the union span (so that its V row must be zeroed)? Full:
// the tile's chunk is invalid or its last key is at or past L. Ring: offsets run base, base + 1, ...
// (mod R); a tile that wraps holds offsets near R, past the span (the ring holds at least the span
// plus one tile), so the tile is clean only when base + 63 < span.
template <bool RING>
__device__ __forceinline__ bool tile_has_outside_keys(const Work& w, const Tile& t) {
  if (!RING) return !t.valid || t.base + kChunk - 1 >= w.L;
  return t.base + kChunk - 1 >= w.span;
}

// The keys of a tile that one row attends form an interval [klo, khi] of tile indices:
//  full: positions base + k <= p_i (and the tile's chunk is valid);
//  ring: offsets (from s_lo) in [max(0, p_i - W + 1 - lo), p_i - lo]. In the one tile that holds
//  both ring ends (base + 63 >= R) the indices below R - base map to offsets near R, which lie
//  outside every window (the ring holds at least the span plus one tile), so shifting by R
//  keeps the valid keys an interval.
template <bool RING>
__device__ __forceinline__ void key_interval(const AttnParams& p, const Work& w, const Tile& t, int p_i, int* klo,
                                             int* khi) {
  if (!RING) {
    *klo = 0;
    *khi = t.valid ? min(kChunk - 1, p_i - t.base) : -1;
  } else {
    const int shift = t.base + kChunk - 1 < p.ring_len ? t.base : t.base - p.ring_len;
    const int a = max(0, p_i - p.window + 1 - w.lo);
    const int b = p_i - w.lo;
    *klo = a - shift;
    *khi = b - shift;
  }
}

template <int HD, bool RING, bool MERGE, bool WIDE, bool DIRECT = false>
__global__ void __launch_bounds__(kThreads, 1)
    attend_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
  static_assert(!DIRECT || !MERGE, "a single split writes its output without a merge");
  using C = Cfg<HD, RING, MERGE, WIDE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQBytes;
  uint8_t* sV = sK + C::kKStages * C::kTileBytes;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- prologue (overlaps the previous kernel under programmatic dependent launch) ----------
  if (threadIdx.x == kProducerWarp * 32) {
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < kGeo; ++i) mbar_init(&bars->geo_full[i], 1);
    for (int i = 0; i < C::kSBufs; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kSoftmaxThreads);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars->o_full[i >> 1][i & 1], 1);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->q_ready, kSoftmaxThreads);
    for (int i = 0; i < 4; ++i) mbar_init(&bars->xchg_l[i], 64);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->never, 1);
    bars->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  volatile int* abort = &bars->abort;

  // Let the next kernel in the stream launch now: its prologue overlaps this kernel, and its
  // griddepcontrol.wait still waits for this grid to complete.
  pdl_launch_dependents();
  // The work item comes from per-step metadata. When the caller has declared that metadata
  // stable (written only by work that completed before this kernel started), it is read before
  // waiting for the previous kernel, off the critical path.
  if (!p.stable_metadata) pdl_wait();
  const Work w = make_work<RING, C::kCPT>(p);
  if (p.stable_metadata) pdl_wait();
  if (w.bad && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, kErrDeviceInput);

  const uint32_t idesc_s = idesc_bf16_f32(128, C::kKT, 0, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, HD, 0, 1);
  const size_t pidx = ((static_cast<size_t>(w.b) * p.row_tiles + w.rt) * p.hkv + w.h) * p.num_splits + w.s;

  if (warp == kProducerWarp) {
    // ------------------------------ K producer (and tile geometry) -----------------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto prefetch_tile = [&](int f) {
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) {
          const Tile tf = tile_at<RING, C::kCPT>(p, w, f, c);
          if (!tf.present) continue;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            tma_prefetch_2d(&tmap_k, bx * 64, tf.y);
            tma_prefetch_2d(&tmap_v, bx * 64, tf.y);
          }
        }
      };
      int issued = 0;
      bool reported = false;
      for (int j = 0; j < w.nt; ++j) {
        const int st = j % C::kKStages;
        if (j >= C::kKStages && !mbar_wait(&bars->k_empty[st], ((j / C::kKStages) - 1) & 1, abort, p.err)) break;
        Tile t[C::kCPT];
        int n_present = 0;
        bool zero = false;
        const int g = j % kGeo;
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) {
          t[c] = tile_at<RING, C::kCPT>(p, w, j, c);
          if (t[c].present && !t[c].valid && !reported) {
            atomicOr(p.err, kErrDeviceInput);
            reported = true;
          }
          bars->tile_base[g][c] = t[c].base;
          bars->tile_valid[g][c] = t[c].valid ? 1 : 0;
          zero = zero || !t[c].present || tile_has_outside_keys<RING>(w, t[c]);
          n_present += t[c].present ? 1 : 0;
        }
        bars->tile_zero[g] = zero ? 1 : 0;
        mbar_arrive(&bars->geo_full[g]);
        // A chunk the sequence lacks is not loaded: its K and V rows keep stale data, which the
        // mask and the V zeroing make harmless.
        mbar_arrive_expect_tx(&bars->k_full[st], n_present * C::kChunkBytes);
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) {
          if (!t[c].present) continue;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_2d(sK + st * C::kTileBytes + bx * C::kBoxBytes + c * C::kChunkRowsBytes, &tmap_k,
                        &bars->k_full[st], bx * 64, t[c].y, pol);
        }
        // Ask L2 for the tiles that follow the shared-memory stages, so that more of the stream is
        // in flight from HBM than the stages alone can hold.
        if (j == C::kKStages - 1) {
          for (int f = C::kKStages; f < C::kKStages + kPrefetch && f < w.nt; ++f) prefetch_tile(f);
        } else if (j >= C::kKStages && j + kPrefetch < w.nt) {
          prefetch_tile(j + kPrefetch);
        }
        issued = j + 1;
      }
      // Every copy lands before the CTA can exit, whether or not the pipeline was aborted (a wait
      // that ran out elsewhere may have ended the consumers before they saw the last tiles). In a
      // normal run these phases have completed already.
      for (int j = max(0, issued - C::kKStages); j < issued; ++j)
        mbar_drain(&bars->k_full[j % C::kKStages], (j / C::kKStages) & 1, p.err);
    }
  } else if (warp == kVProducerWarp) {
    // ------------------------------ V producer --------------------------------------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int j = 0; j < w.nt; ++j) {
        const int st = j % C::kVStages;
        if (j >= C::kVStages && !mbar_wait(&bars->v_empty[st], ((j / C::kVStages) - 1) & 1, abort, p.err)) break;
        Tile t[C::kCPT];
        int n_present = 0;
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) {
          t[c] = tile_at<RING, C::kCPT>(p, w, j, c);
          n_present += t[c].present ? 1 : 0;
        }
        mbar_arrive_expect_tx(&bars->v_full[st], n_present * C::kChunkBytes);
#pragma unroll
        for (int c = 0; c < C::kCPT; ++c) {
          if (!t[c].present) continue;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_2d(sV + st * C::kTileBytes + bx * C::kBoxBytes + c * C::kChunkRowsBytes, &tmap_v,
                        &bars->v_full[st], bx * 64, t[c].y, pol);
        }
        issued = j + 1;
      }
      for (int j = max(0, issued - C::kVStages); j < issued; ++j)
        mbar_drain(&bars->v_full[j % C::kVStages], (j / C::kVStages) & 1, p.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer (one lane) ---------------------------------
    // tcgen05.mma issue blocks while the tensor pipe is busy, so the tensor core idles whenever
    // this thread does anything else: it only waits on barriers and issues.
    if (lane == 0) {
      // Test of the timeout path (off unless asked for): one bounded wait on a barrier that
      // nothing completes runs out, and the CTA takes the path of any wait that ran out.
      if (p.timeout_test_ns != 0) mbar_wait_limit(&bars->never, 0, p.timeout_test_ns, abort, p.err);
      bool ok = !*abort && mbar_wait(&bars->q_ready, 0, abort, p.err);
      tc_fence_after();
      // Descriptors are built once: a descriptor's low 14 bits hold its address >> 4, and shared
      // addresses stay below 256 KB, so adding a byte offset >> 4 moves it without carrying out of
      // the field. The thread shares its sub-partition with two softmax warps, so every scalar
      // instruction it saves shortens the time the tensor pipe waits for it.
      const uint64_t qdesc = sw128_desc(smem_u32(sQ), 16, 1024);
      const uint64_t kdesc = sw128_desc(smem_u32(sK), 16, 1024);
      const uint64_t vdesc = sw128_desc(smem_u32(sV), C::kBoxBytes, 1024);
      // S_j = Q K_j^T into S buffer j % B (B = kSBufs). Before P.V of tile jp, S of tiles up to jp
      // is issued (waiting for their K if need be: the softmax of tile jp needs S_jp), and S of
      // tiles up to jp + B - 1 only if their K has already landed, so that P.V never waits for a
      // later tile's K and each stage is released as soon as its P.V completes. S_{jp+B-1} goes
      // into the buffer that P.V of tile jp-1, issued before it, reads P from: MMAs run in issue
      // order.
      int next_s = 0;
      auto issue_s = [&](int j) {
        const int st = j % C::kKStages;
        tc_fence_after();
        const uint64_t kd = kdesc + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
        const uint32_t d_s = tbase + kColS + (j % C::kSBufs) * C::kKT;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t a = qdesc + static_cast<uint64_t>(((kk >> 2) * C::kQBoxBytes + (kk & 3) * 32) >> 4);
          const uint64_t bdesc = kd + static_cast<uint64_t>(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
          mma_ss(d_s, a, bdesc, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[j % C::kSBufs]);
        mma_commit(&bars->k_empty[st]);                 // S_j has read K_j
      };
      for (int jp = 0; ok && jp < w.nt; ++jp) {
        while (ok && next_s <= jp) {
          ok = mbar_wait(&bars->k_full[next_s % C::kKStages], (next_s / C::kKStages) & 1, abort, p.err);
          if (ok) issue_s(next_s++);
        }
        while (ok && next_s < w.nt && next_s <= jp + C::kSBufs - 1 &&
               mbar_test_wait(&bars->k_full[next_s % C::kKStages], (next_s / C::kKStages) & 1))
          issue_s(next_s++);
        if (!ok) break;
        // O_h += P_h V_h for tile jp over the keys [h kKH, (h + 1) kKH) of warpgroup h, which has
        // zeroed the V rows of its keys that lie outside every query's range before arriving.
        // V_jp has landed: a softmax warp waits for it before it arrives on the tile's P barrier.
        const int st = jp % C::kVStages;
        const uint64_t vd = vdesc + static_cast<uint64_t>((st * C::kTileBytes) >> 4);
        const int sb = jp % C::kSBufs;
        // One wait for both halves: the warpgroups finish a tile's P together, and every wait
        // costs the issuer about as much as two MMAs of the tile, with the tensor pipe idle.
        ok = mbar_wait(&bars->p_full[sb], (jp / C::kSBufs) & 1, abort, p.err);
        if (!ok) break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < C::kKH / 16; ++kk) {
            const uint64_t bdesc = vd + static_cast<uint64_t>(((h * C::kKH + 16 * kk) * 128) >> 4);
            mma_ts(tbase + kColO + h * 128, tbase + kColS + sb * C::kKT + h * C::kKH + kk * 8, bdesc, idesc_pv,
                   (jp > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_full[h][jp & 1]);
        }
        mma_commit(&bars->v_empty[st]);
        if (jp == w.nt - 1) mma_commit(&bars->o_done);
      }
      // Every MMA issued above completes before TMEM is freed.
      mma_commit(&bars->drain);
      mbar_drain(&bars->drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax / epilogue (warps 0-7) ------------------------
    const int wg = warp >> 2;                          // warpgroup: which 32 keys of a tile
    const int quarter = warp & 3;                      // TMEM lane quarter
    const int mrow = quarter * 32 + lane;              // TMEM lane and Q smem row
    const int lr = lane + (quarter == 2 ? 96 : quarter == 3 ? 64 : quarter * 32);   // tile row of this lane
    const bool active = __any_sync(0xffffffffu, lr < w.rows);  // the warp holds a row of the block
    const bool rv = lr < w.rows;
    const int r = w.row0 + lr;                         // block row: query r / G, q-head r % G
    const unsigned ug = static_cast<unsigned>(p.group);   // unsigned division: fewer instructions
    const int qi = rv ? static_cast<int>(static_cast<unsigned>(r) / ug) : 0;
    const int g = rv ? static_cast<int>(static_cast<unsigned>(r) % ug) : 0;
    // Q row -> swizzled smem (the 128-byte swizzle TMA would apply: chunk c of row m at c ^ (m & 7)).
    // Each warpgroup stages half of the row's 16-byte chunks.
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(w.q0 + qi) * p.hq + static_cast<size_t>(w.h) * p.group + g) * HD);
      constexpr int kHalf = HD / 16;
      uint4 qv[kHalf];
#pragma unroll
      for (int c = 0; c < kHalf; ++c) qv[c] = rv ? __ldg(src + wg * kHalf + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < kHalf; ++c) {
        const int cg = wg * kHalf + c;
        const int bx = cg >> 3, cc = cg & 7;
        *reinterpret_cast<uint4*>(sQ + bx * C::kQBoxBytes + mrow * 128 + ((cc ^ (mrow & 7)) << 4)) = qv[c];
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->q_ready);
    }
    const int p_i = w.L - w.nq + qi;                   // this row's query position
    const uint32_t lane_base = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int KH = C::kKH;                         // keys of a tile this warpgroup takes
    const int cw = C::kCPT == 2 ? wg : 0;              // the chunk that holds them
    const int kofs = C::kCPT == 2 ? 0 : wg * KH;       // and the first one's index in that chunk
    const uint32_t col_s = kColS + wg * KH;            // their S columns within a buffer
    const uint32_t col_o = kColO + wg * 128;           // this warpgroup's O accumulator
    float m_ref = -INFINITY;                           // this half's reference maximum
    float l_half = 0.f;                                // this half's row sum
    bool ok = true;
    for (int j = 0; j < w.nt; ++j) {
      const int sb = j % C::kSBufs;
      // The tile's geometry comes from the K producer through its ring, written before the tile's
      // copies are issued, so it is read (with this row's key interval) while S_j is computed.
      // The entry is rewritten for tile j + kGeo only after S_{j + kGeo - kKStages} has read its
      // K; that S needed its buffer back from P.V of tile j + kGeo - kKStages - kSBufs >= j, which
      // waits for this warpgroup's P of that tile. So the entry is still this tile's, and its
      // barrier is not a phase ahead.
      const int gs = j % kGeo;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->geo_full[gs], (j / kGeo) & 1, abort, p.err));
      if (!ok) break;
      Tile t;
      t.base = bars->tile_base[gs][cw];
      t.valid = bars->tile_valid[gs][cw] != 0;
      int klo = 0, khi = kChunk - 1;
      if (rv) key_interval<RING>(p, w, t, p_i, &klo, &khi);
      klo -= kofs;
      khi -= kofs;
      // Rows past the block (padding lanes) see Q = 0; their P and O rows are never read.
      const bool whole = __all_sync(0xffffffffu, klo <= 0 && khi >= KH - 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (j / C::kSBufs) & 1, abort, p.err));
      if (!ok) break;
      tc_fence_after();
      if (active) {
        // (A warp without rows of the block only keeps the barrier protocol: its P and O lanes are
        // never read.)
        float sv[KH];
        {
          uint32_t sr[KH];
          if constexpr (KH == 32)
            tmem_ld32(lane_base + col_s + sb * C::kKT, sr);
          else
            tmem_ld64(lane_base + col_s + sb * C::kKT, sr);
#pragma unroll
          for (int k = 0; k < KH; ++k) sv[k] = __uint_as_float(sr[k]);
        }
        if (!whole) {
#pragma unroll
          for (int k = 0; k < KH; ++k) sv[k] = (k >= klo && k <= khi) ? sv[k] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = sv[u];
#pragma unroll
        for (int k = 8; k < KH; ++k) mx[k & 7] = fmaxf(mx[k & 7], sv[k]);
        const float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
        bool need_o = false;
        float alpha = 1.f;
        if (m_tile > m_ref + kRescaleLog2) {
          need_o = m_ref != -INFINITY;                // O_h already holds weighted values
          alpha = ex2_approx(m_ref - m_tile);         // 0 when m_ref = -inf
          l_half *= alpha;
          m_ref = m_tile;
        }
        if (__any_sync(0xffffffffu, need_o)) {
          // O_h holds the sum over tiles < j: wait for its P.V of tile j-1, then scale it. S_j was
          // issued after P.V of tile j - kSBufs (S_j needs the buffer it read) and has completed,
          // so that P.V has too, and P.V of tile j+1 needs this tile's P: the barrier of odd or
          // even tiles o_full[h][(j-1) & 1] is in phase (j-1)/2 or the one after, so the parity
          // wait for phase (j-1)/2 is exact.
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bars->o_full[wg][(j - 1) & 1], ((j - 1) >> 1) & 1, abort, p.err));
          if (!ok) break;
          tc_fence_after();
          const float a = need_o ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + col_o + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st32(lane_base + col_o + c * 32, o);
          }
        }
        // p = 2^(s * scale * log2e - m_ref); masked keys carry s = -inf and give exactly 0. A row
        // that has seen no key yet (m_ref = -inf) has only masked keys here, and uses 0 as
        // reference.
        const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
        uint32_t pk[KH / 2];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < KH / 2; ++e) {
          const float p0 = ex2_approx(fmaf(sv[2 * e], p.scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(sv[2 * e + 1], p.scale_log2, neg_m));
          ps[e & 3] += p0 + p1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        if (rv) l_half += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // P_h over the first half of this warpgroup's own S columns
        if constexpr (KH == 32)
          tmem_st16(lane_base + col_s + sb * C::kKT, pk);
        else
          tmem_st32(lane_base + col_s + sb * C::kKT, pk);
      }
      tc_fence_before();
      if (bars->tile_zero[gs]) {
        // Keys outside every query's range may hold anything (stale ring slots, the unused tail
        // of the last chunk, a chunk the sequence lacks). P is 0 there, but 0 * NaN is NaN on the
        // tensor core, so the V rows of this half's such keys are zeroed (whole 128-byte rows:
        // the swizzle permutes 16-byte chunks within a row) before P.V reads them.
        const int sv_st = j % C::kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[sv_st], (j / C::kVStages) & 1, abort, p.err));
        if (!ok) break;
        constexpr int kTPR = 128 / KH;                 // threads per key row
        constexpr int kPerT = C::kBoxes * 8 / kTPR;    // 16-byte chunks each of them zeroes
        const int tw = threadIdx.x & 127;
        const int kz = tw / kTPR;
        int pos;
        if (!key_in_union<RING>(p, w, t, kofs + kz, &pos)) {
          uint8_t* vt = sV + sv_st * C::kTileBytes;
          const int row = wg * KH + kz;                // the key's row in the tile
#pragma unroll
          for (int c = (tw % kTPR) * kPerT; c < (tw % kTPR + 1) * kPerT; ++c)
            *reinterpret_cast<uint4*>(vt + (c >> 3) * C::kBoxBytes + row * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      if (warp == kVRelayWarp) {
        // This warp's arrival on the P barrier waits for V_j, so the issuer's one wait for P
        // covers V too. In a block of at most 96 rows it is a warp without rows; otherwise its
        // wait overlaps the other warps' softmax.
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&bars->v_full[j % C::kVStages], (j / C::kVStages) & 1, abort, p.err));
        if (!ok) break;
      }
      mbar_arrive(&bars->p_full[sb]);
    }
    // ---- epilogue: merge the two halves into the split's partial (m, l, unnormalised O) ----
    float m_w[2] = {-INFINITY, -INFINITY}, l_w[2] = {0.f, 0.f};
    if (ok) {
      bars->xm[wg][mrow] = l_half > 0.f ? m_ref : -INFINITY;
      bars->xl[wg][mrow] = l_half;
      mbar_arrive(&bars->xchg_l[quarter]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->xchg_l[quarter], 0, abort, p.err));
      if (ok) {
        m_w[0] = bars->xm[0][mrow];
        m_w[1] = bars->xm[1][mrow];
        l_w[0] = bars->xl[0][mrow];
        l_w[1] = bars->xl[1][mrow];
      }
    }
    const float m_row = fmaxf(m_w[0], m_w[1]);
    const float w0 = l_w[0] > 0.f ? ex2_approx(m_w[0] - m_row) : 0.f;
    const float w1 = l_w[1] > 0.f ? ex2_approx(m_w[1] - m_row) : 0.f;
    const float l_sum = w0 * l_w[0] + w1 * l_w[1];
    // A parity wait on o_full cannot tell phase nt-1 from nt-3 when P.V_{nt-2} is still running,
    // so the last P.V has a barrier of its own.
    if (ok && w.nt > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done, 0, abort, p.err));
      tc_fence_after();
    }
    if constexpr (MERGE) {
      // Each softmax thread sends its row's half of the columns, [h d/2, (h + 1) d/2) for
      // warpgroup h, straight from registers into the receive area of the row's owner, split rank
      // r % n: bf16 normalised by the split's row sum l, eight 16-byte stores; warpgroup 0 also
      // sends the (m, l) pair (fp32). A split without data for a row sends (-inf, 0) and no O.
      const int n = static_cast<int>(cluster_nctarank());
      const int rank = static_cast<int>(cluster_ctarank());
      const uint32_t recv = smem_u32(smem + C::kRecvOffset);
      const uint32_t recv_ml = smem_u32(smem + C::kRecvMlOffset);
      const unsigned rq = static_cast<unsigned>(lr) / static_cast<unsigned>(n);
      const int e = static_cast<int>(rq) * n + rank;     // entry in the owner's receive area
      const uint32_t owner = static_cast<uint32_t>(lr - static_cast<int>(rq) * n);
      if (rv && wg == 0)
        st_dsmem_f2(dsmem_addr(recv_ml + e * 8, owner), make_float2(l_sum > 0.f ? m_row : -INFINITY, l_sum));
      if (ok && w.nt > 0) {
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const uint32_t row_at = recv + e * HD * 2 + wg * HD;   // this half's bytes of the entry
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32x2(lane_base + kColO + wg * (HD / 2) + c * 32, lane_base + kColO + 128 + wg * (HD / 2) + c * 32,
                      o0, o1);
          if (rv && l_sum > 0.f) {
#pragma unroll
            for (int x = 0; x < 32; x += 8) {
              uint32_t pk[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float a = (w0 * __uint_as_float(o0[x + 2 * q]) + w1 * __uint_as_float(o1[x + 2 * q])) * inv;
                const float b =
                    (w0 * __uint_as_float(o0[x + 2 * q + 1]) + w1 * __uint_as_float(o1[x + 2 * q + 1])) * inv;
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
                pk[q] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              st_dsmem_u4(dsmem_addr(row_at + (c * 32 + x) * 2, owner), make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
          }
        }
      }
    } else if constexpr (DIRECT) {
      // A single split: this CTA holds every key of its rows, so it normalises O and writes it,
      // bf16, with the LSE; no combine follows. (A variant of its own: the same branch, untaken,
      // in the kernel the 40-layer pass runs made its full layers 2.7 us slower.) Warpgroup h writes
      // columns [h d/2, (h + 1) d/2). A row without an attended key gets O = 0, LSE = -inf.
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const unsigned br = static_cast<unsigned>(r);
      const unsigned bq = br / static_cast<unsigned>(p.group);
      const int t = w.q0 + static_cast<int>(bq);
      const int hq = w.h * p.group + static_cast<int>(br - bq * static_cast<unsigned>(p.group));
      const bool wr = ok && rv && t < p.token_cap;
      uint16_t* dst = p.out + (static_cast<size_t>(wr ? t : 0) * p.hq + hq) * HD + wg * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t o0[32], o1[32];
        if (ok && w.nt > 0) {
          tmem_ld32(lane_base + kColO + wg * (HD / 2) + c * 32, o0);
          tmem_ld32(lane_base + kColO + 128 + wg * (HD / 2) + c * 32, o1);
        }
        if (wr) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a = 0.f, b = 0.f;
            if (w.nt > 0 && l_sum > 0.f) {
              a = (w0 * __uint_as_float(o0[2 * e]) + w1 * __uint_as_float(o1[2 * e])) * inv;
              b = (w0 * __uint_as_float(o0[2 * e + 1]) + w1 * __uint_as_float(o1[2 * e + 1])) * inv;
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
            pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<uint4*>(dst + c * 32 + 2 * e) = make_uint4(pk[e], pk[e + 1], pk[e + 2], pk[e + 3]);
        }
      }
      if (wr && wg == 0 && p.lse != nullptr)
        p.lse[static_cast<size_t>(t) * p.hq + hq] =
            l_sum > 0.f ? (m_row + __log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
    } else if (ok) {
      // warpgroup h writes columns [h d/2, (h + 1) d/2) of the merged O
      float* dst = p.part_o + (pidx * kMaxRows + lr) * HD + wg * (HD / 2);
      if (w.nt > 0) {
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          uint32_t o0[32], o1[32];
          tmem_ld32(lane_base + kColO + wg * (HD / 2) + c * 32, o0);
          tmem_ld32(lane_base + kColO + 128 + wg * (HD / 2) + c * 32, o1);
          if (rv && l_sum > 0.f) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + c * 32 + e) =
                  make_float4(w0 * __uint_as_float(o0[e]) + w1 * __uint_as_float(o1[e]),
                              w0 * __uint_as_float(o0[e + 1]) + w1 * __uint_as_float(o1[e + 1]),
                              w0 * __uint_as_float(o0[e + 2]) + w1 * __uint_as_float(o1[e + 2]),
                              w0 * __uint_as_float(o0[e + 3]) + w1 * __uint_as_float(o1[e + 3]));
          }
        }
      }
      if (rv && wg == 0) {
        float2* ml = reinterpret_cast<float2*>(p.part_ml) + pidx * kMaxRows + lr;
        *ml = make_float2(l_sum > 0.f ? m_row : -INFINITY, l_sum);
      }
    }
  }
  if constexpr (MERGE) {
    // ---- cluster merge: the CTAs of the cluster are the splits of this (b, h), in rank order.
    // After the barrier every owner holds, in its own shared memory, all splits' (m, l, o) of its
    // rows rank + n k; one warp merges one row and writes its bf16 output and log-sum-exp:
    //   O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  LSE = ln2 * (M + log2 sum_s 2^(m_s - M) l_s)
    // No CTA touches another's shared memory after the barrier, so each exits when done.
    __syncwarp();
    cluster_sync_all();
    const int n = static_cast<int>(cluster_nctarank());
    const int rank = static_cast<int>(cluster_ctarank());
    constexpr int kPer = HD / 32;                      // columns per lane
    const uint16_t* recv = reinterpret_cast<const uint16_t*>(smem + C::kRecvOffset);
    const float2* recv_ml = reinterpret_cast<const float2*>(smem + C::kRecvMlOffset);
    for (int k = warp;; k += kThreads / 32) {
      const int r = rank + n * k;
      if (r >= w.rows) break;
      // Every lane reads all n (m, l) pairs of the row (same address across the warp) and the
      // lane's columns of every split's row, in one batch, and weighs them itself: no shuffles. A
      // split without data for the row sent no O row: its entry holds anything, and its zero weight
      // selects it out.
      const float2* mlk = recv_ml + k * n;
      const uint16_t* rowk = recv + static_cast<size_t>(k * n) * HD + lane * kPer;
      float2 mls[kMaxClusterSplits];
      uint32_t u[kMaxClusterSplits][kPer / 2];
#pragma unroll
      for (int s = 0; s < kMaxClusterSplits; ++s) {
        if (s < n) {
          mls[s] = mlk[s];
          if constexpr (kPer == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(rowk + s * HD);
            u[s][0] = v.x;
            u[s][1] = v.y;
          } else {
            u[s][0] = *reinterpret_cast<const uint32_t*>(rowk + s * HD);
          }
        } else {
          mls[s] = make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int x = 0; x < kPer / 2; ++x) u[s][x] = 0u;
        }
      }
      float mm = -INFINITY;
#pragma unroll
      for (int s = 0; s < kMaxClusterSplits; ++s) mm = mls[s].y > 0.f ? fmaxf(mm, mls[s].x) : mm;
      float lsum = 0.f;
      float acc[kPer];
#pragma unroll
      for (int x = 0; x < kPer; ++x) acc[x] = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxClusterSplits; ++s) {
        // the rows are normalised by their split's l: weight 2^(m - M) l
        const bool use = mls[s].y > 0.f;
        const float ws = use ? ex2_approx(mls[s].x - mm) * mls[s].y : 0.f;
        lsum += ws;
#pragma unroll
        for (int x = 0; x < kPer / 2; ++x) {
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[s][x]));
          acc[2 * x] = use ? fmaf(ws, a.x, acc[2 * x]) : acc[2 * x];
          acc[2 * x + 1] = use ? fmaf(ws, a.y, acc[2 * x + 1]) : acc[2 * x + 1];
        }
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const unsigned br = static_cast<unsigned>(w.row0 + r);   // r is the row within this tile
      const unsigned bq = br / static_cast<unsigned>(p.group);
      const int t = w.q0 + static_cast<int>(bq);
      const int hq = w.h * p.group + static_cast<int>(br - bq * static_cast<unsigned>(p.group));
      if (t < p.token_cap) {
        uint16_t* dst = p.out + (static_cast<size_t>(t) * p.hq + hq) * HD + lane * kPer;
        if constexpr (kPer == 4) {
          const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
          const __nv_bfloat162 c = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
          uint2 w2;
          w2.x = *reinterpret_cast<const uint32_t*>(&a);
          w2.y = *reinterpret_cast<const uint32_t*>(&c);
          *reinterpret_cast<uint2*>(dst) = w2;
        } else {
          const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
          *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&a);
        }
        if (p.lse != nullptr && lane == 0)
          p.lse[static_cast<size_t>(t) * p.hq + hq] =
              lsum > 0.f ? (mm + __log2f(lsum)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------ split combine ---------------------------------------------------
// One 128-thread CTA per output row (token t, q-head hq). Warp w takes splits w, w + 4, ...; each
// lane loads the (m, l) of one of them and 16 bytes of every one of them's O row, all loads in
// one batch. The warp merges its splits against its own maximum (shuffles), then warp 0 merges the
// four warps through shared memory:
//   O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  LSE = ln2 * (M + log2 sum_s 2^(m_s - M) l_s)
constexpr int kCombineMaxPerWarp = 16;   // splits per warp (64 splits per row at most)

template <int HD>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  constexpr int kPer = HD / 32;
  using Vec = typename std::conditional<kPer == 4, float4, float2>::type;
  __shared__ float s_m[4];
  __shared__ float s_l[4];
  __shared__ float s_acc[4][HD];
  pdl_launch_dependents();
  // The row's sequence comes from per-step metadata: read before the dependency wait when the
  // caller has declared it stable, after it otherwise. The partials are read after it.
  if (!p.stable_metadata) pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = static_cast<int>(blockIdx.x / p.hq);
  const int hq = static_cast<int>(blockIdx.x % p.hq);
  // One round trip for a one-sequence batch: its values are loaded with the batch's token count
  // (all in bounds: cu_q has B + 1 entries, seq_len B). A batch searches for its sequence.
  const int total = p.cu_q[p.num_seqs];
  int b = 0;
  int c0 = p.cu_q[0], c1 = p.cu_q[1], len = p.seq_len[0];
  if (p.num_seqs > 1 && t < p.token_cap && t < total) {
    while (b + 1 < p.num_seqs && p.cu_q[b + 1] <= t) ++b;
    c0 = p.cu_q[b];
    c1 = p.cu_q[b + 1];
    len = p.seq_len[b];
  }
  if (p.stable_metadata) pdl_wait();
  if (t >= p.token_cap || t >= total) return;
  const int i = t - c0;
  const int nq = c1 - c0;
  if (i < 0 || nq < 0 || nq > p.max_q || len < nq) return;   // skipped by the attention kernel too
  const int h = static_cast<int>(static_cast<unsigned>(hq) / static_cast<unsigned>(p.group));
  const int rg = i * p.group + (hq - h * p.group);        // block row
  const int rt = rg / kMaxRows;                           // its row tile
  const int r = rg - rt * kMaxRows;                       // and its row within the tile
  const size_t p0 = ((static_cast<size_t>(b) * p.row_tiles + rt) * p.hkv + h) * p.num_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);

  // this warp's splits: s = warp + 4 u, u < nsub
  const int nsub = min(kCombineMaxPerWarp, (p.num_splits - warp + 3) / 4);
  float2 my_ml = make_float2(-INFINITY, 0.f);
  if (lane < nsub) my_ml = __ldcg(ml + (p0 + warp + 4 * lane) * kMaxRows + r);
  // The O rows are loaded in the same batch as (m, l): a split without data for this row may hold
  // anything there, and its weight selects it out below (never multiplied in).
  Vec v[kCombineMaxPerWarp];
#pragma unroll
  for (int u = 0; u < kCombineMaxPerWarp; ++u) {
    if (u < nsub)
      v[u] = __ldcg(reinterpret_cast<const Vec*>(p.part_o + ((p0 + warp + 4 * u) * kMaxRows + r) * HD) + lane);
    else if constexpr (kPer == 4)
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    else
      v[u] = make_float2(0.f, 0.f);
  }
  float m_w = my_ml.y > 0.f ? my_ml.x : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m_w = fmaxf(m_w, __shfl_xor_sync(0xffffffffu, m_w, o));
  const float wgt = (my_ml.y > 0.f) ? ex2_approx(my_ml.x - m_w) : 0.f;
  float l_w = wgt * my_ml.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l_w += __shfl_xor_sync(0xffffffffu, l_w, o);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
#pragma unroll
  for (int u = 0; u < kCombineMaxPerWarp; ++u) {
    const float wk = __shfl_sync(0xffffffffu, wgt, u);
    const bool use = wk != 0.f;
    if constexpr (kPer == 4) {
      acc[0] = use ? fmaf(wk, v[u].x, acc[0]) : acc[0];
      acc[1] = use ? fmaf(wk, v[u].y, acc[1]) : acc[1];
      acc[2] = use ? fmaf(wk, v[u].z, acc[2]) : acc[2];
      acc[3] = use ? fmaf(wk, v[u].w, acc[3]) : acc[3];
    } else {
      acc[0] = use ? fmaf(wk, v[u].x, acc[0]) : acc[0];
      acc[1] = use ? fmaf(wk, v[u].y, acc[1]) : acc[1];
    }
  }
  if (lane == 0) {
    s_m[warp] = m_w;
    s_l[warp] = l_w;
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) s_acc[warp][lane * kPer + e] = acc[e];
  __syncthreads();
  if (warp != 0) return;
  const float mmax = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
  float sc[4];
  float lsum = 0.f;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    sc[x] = (s_l[x] > 0.f) ? ex2_approx(s_m[x] - mmax) : 0.f;
    lsum += sc[x] * s_l[x];
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  float o[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    float a = 0.f;
#pragma unroll
    for (int x = 0; x < 4; ++x) a = fmaf(sc[x], s_acc[x][lane * kPer + e], a);
    o[e] = a * inv;
  }
  uint16_t* dst = p.out + (static_cast<size_t>(t) * p.hq + hq) * HD + lane * kPer;
  if constexpr (kPer == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 c = __floats2bfloat162_rn(o[2], o[3]);
    uint2 w2;
    w2.x = *reinterpret_cast<const uint32_t*>(&a);
    w2.y = *reinterpret_cast<const uint32_t*>(&c);
    *reinterpret_cast<uint2*>(dst) = w2;
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]);
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(&a);
  }
  if (p.lse != nullptr && lane == 0) {
    p.lse[static_cast<size_t>(t) * p.hq + hq] =
        lsum > 0.f ? (mmax + __log2f(lsum)) * 0.6931471805599453f : -INFINITY;
  }
}

}  // namespace

// Largest cluster of merging attend_kernel CTAs that can be resident on the current device (one
// CTA per SM: the cluster must fit in one GPC), cached per device.
template <int HD, bool RING>
static int merge_cluster_limit() {
  static int limit[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (limit[dev] != 0) return limit[dev];
  auto kern = attend_kernel<HD, RING, true, false>;
  constexpr int kSmem = Cfg<HD, RING, true, false>::kSmemBytes;
  static size_t done[64] = {};
  if (ensure_smem_limit(kern, kSmem, done) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kMaxClusterSplits, 1, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  int n = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  limit[dev] = n < 1 ? 1 : (n > kMaxClusterSplits ? kMaxClusterSplits : n);
  return limit[dev];
}

template <int HD, bool RING, bool MERGE, bool WIDE, bool DIRECT = false>
static cudaError_t launch_attend_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                   int num_seqs, cudaStream_t stream) {
  static size_t done[64] = {};
  auto kern = attend_kernel<HD, RING, MERGE, WIDE, DIRECT>;
  constexpr int kSmem = Cfg<HD, RING, MERGE, WIDE>::kSmemBytes;
  cudaError_t e = ensure_smem_limit(kern, kSmem, done);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.hkv, num_seqs * p.row_tiles);
  if constexpr (!MERGE) {
    return launch_pdl(kern, grid, dim3(kThreads), kSmem, stream, p, tk, tv);
  } else {
    if (p.num_splits > merge_cluster_limit<HD, RING>()) return cudaErrorNotSupported;
    return launch_pdl_cluster(kern, grid, dim3(kThreads), kSmem, p.num_splits, stream, p, tk, tv);
  }
}

int attend_merge_limit(bool ring, int head_dim) {
  if (head_dim == 128) return ring ? merge_cluster_limit<128, true>() : merge_cluster_limit<128, false>();
  return ring ? merge_cluster_limit<64, true>() : merge_cluster_limit<64, false>();
}

template <int HD>
static cudaError_t launch_attend_hd(bool ring, AttnTiles tiles, const AttnParams& p, const CUtensorMap& tk,
                                    const CUtensorMap& tv, int num_seqs, cudaStream_t stream) {
  if (ring)
    return tiles == AttnTiles::kMerge ? launch_attend_t<HD, true, true, false>(p, tk, tv, num_seqs, stream)
                                      : launch_attend_t<HD, true, false, false>(p, tk, tv, num_seqs, stream);
  switch (tiles) {
    case AttnTiles::kMerge: return launch_attend_t<HD, false, true, false>(p, tk, tv, num_seqs, stream);
    case AttnTiles::kWide: return launch_attend_t<HD, false, false, true>(p, tk, tv, num_seqs, stream);
    case AttnTiles::kWideDirect: return launch_attend_t<HD, false, false, true, true>(p, tk, tv, num_seqs, stream);
    default: return launch_attend_t<HD, false, false, false>(p, tk, tv, num_seqs, stream);
  }
}

cudaError_t launch_attend(bool ring, int head_dim, AttnTiles tiles, const AttnParams& p, const CUtensorMap& tk,
                          const CUtensorMap& tv, int num_seqs, cudaStream_t stream) {
  if (ring && (tiles == AttnTiles::kWide || tiles == AttnTiles::kWideDirect)) return cudaErrorInvalidValue;
  if (head_dim == 128) return launch_attend_hd<128>(ring, tiles, p, tk, tv, num_seqs, stream);
  return launch_attend_hd<64>(ring, tiles, p, tk, tv, num_seqs, stream);
}

cudaError_t launch_combine(int head_dim, const CombineParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.token_cap) * p.hq;
  dim3 grid(static_cast<unsigned>(rows));
  if (head_dim == 128) return launch_pdl(combine_kernel<128>, grid, dim3(128), 0, stream, p);
  return launch_pdl(combine_kernel<64>, grid, dim3(128), 0, stream, p);
}

}  // namespace vfy
