// Chunk-residency top-k with slot reconciliation and the page-in list.
// Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "Three optimizations", item 1: the pool
// keeps 8K of the context on the GPU as 64-token chunks, and a drafter scores which chunks deserve
// residency. Selection rule (a reading; the pages name none): the k best scores, ties to the lower
// chunk index, -0 == +0, NaN below every number.
//
// One 1024-thread CTA per sequence. Scores become 32-bit keys that sort like the scores; a 4-pass
// radix select (8 bits per pass, shared-memory histograms) finds the k-th largest key t and how
// many entries equal to t to take; those are the lowest-index ones. Block-wide prefix sums then
// give every chosen chunk its output position, its rank among the equal keys, and, for chunks
// not yet resident, its rank among the newcomers, which indexes the ascending list of free slots.
#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kThreads = 1024;
constexpr int kPre = 4;      // owned chunks whose slots stay in registers (n <= 4096 at 1024 threads)

__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;           // NaN: below everything
  if (u == 0x80000000u) u = 0u;                              // -0 ties +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);         // -inf -> 0x007fffff > 0
}

// Exclusive block-wide prefix sum of one value per thread; returns the prefix, *total the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int s = warp_sums[lane];
    int t = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t - s;                                 // exclusive warp offsets
    if (lane == 31) warp_sums[32] = t;
  }
  __syncthreads();
  const int result = warp_sums[warp] + x - v;
  *total = warp_sums[32];
  __syncthreads();
  return result;
}

__global__ void __launch_bounds__(kThreads) select_kernel(const SelectParams p) {
  extern __shared__ uint32_t keys[];                         // [max(max_n, 2k)]
  __shared__ int hist[256];
  __shared__ int scan_buf[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  __shared__ int s_whole;       // the chosen digit's bin is taken whole: the threshold is found
  __shared__ int s_out0;
  __shared__ int s_flag;

  pdl_wait();
  const int b = blockIdx.x;
  const int k = p.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = p.cu_chunks[b];
  const int n = p.cu_chunks[b + 1] - c0;
  if (threadIdx.x == 0) {
    int o = 0;
    for (int bb = 0; bb < b; ++bb) {
      const int nb = p.cu_chunks[bb + 1] - p.cu_chunks[bb];
      if (nb >= 0 && nb <= p.max_n) o += min(k, nb);
    }
    s_out0 = o;
    s_flag = 0;
  }
  __syncthreads();
  const int out0 = s_out0;
  if (n < 0 || n > p.max_n || c0 < 0) {
    if (threadIdx.x == 0) {
      atomicOr(p.err, kErrDeviceInput);
      p.cu_res[b + 1] = out0;
      p.pagein_count[b] = 0;
      if (b == 0) p.cu_res[0] = 0;
    }
    return;
  }
  const int kk = min(k, n);

  // Each thread owns a contiguous run of `per` (<= 32) chunks, so thread order is chunk order.
  const int per = (n + kThreads - 1) / kThreads;
  const int j0 = min(n, static_cast<int>(threadIdx.x) * per);
  const int j1 = min(n, j0 + per);

  // The previous slots of the first kPre owned chunks are loaded with the scores, into
  // registers (the slot reconciliation needs them after the selection): one round trip for both.
  int prev_r[kPre];
#pragma unroll
  for (int t = 0; t < kPre; ++t) prev_r[t] = j0 + t < j1 ? p.slot_of_chunk[c0 + j0 + t] : -1;
  for (int j = j0; j < j1; ++j) keys[j] = score_key(p.scores[c0 + j]);
  __syncthreads();
  // owned chunk t's previous slot (registers for t < kPre)
  auto prev_slot = [&](int t) {
    int v = t < kPre ? prev_r[0] : p.slot_of_chunk[c0 + j0 + t];
#pragma unroll
    for (int u = 1; u < kPre; ++u) v = t == u ? prev_r[u] : v;
    return v;
  };

  // ---- radix select of the kk-th largest key ----
  uint32_t thr = 0u;
  int take_eq = 0;          // entries equal to thr to take (lowest indices first)
  const bool all = kk >= n;
  if (!all) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = kk;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (threadIdx.x < 256) hist[threadIdx.x] = 0;
      __syncthreads();
      // Lanes with the same digit add once per warp (the leading bytes of nearby scores agree,
      // so plain atomics would queue on a few bins). `per` is the same for every thread.
      for (int t = 0; t < per; ++t) {
        const int j = j0 + t;
        const bool valid = j < j1 && (keys[j] & mask) == prefix;
        if (!__any_sync(0xffffffffu, valid)) continue;   // later passes: most warps hold no candidate
        const uint32_t bin = valid ? (keys[j] >> shift) & 255u : 0xffffffffu;
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // Lane l holds bins 255-8l .. 248-8l (descending). A scan over the lanes gives the count
        // of keys in the bins above each lane's group; the lane whose group holds the
        // remaining-th largest key finds the digit: the largest d whose bins >= d hold at least
        // `remaining` keys (d = 255 when nothing remains to take).
        int c[8];
        int sum = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          c[u] = hist[255 - 8 * lane - u];
          sum += c[u];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int above_group = incl - sum;
        if ((remaining <= 0 && lane == 0) || (above_group < remaining && remaining <= incl)) {
          int above = above_group;
          int u = 0;
          for (; u < 7; ++u) {
            if (above + c[u] >= remaining) break;
            above += c[u];
          }
          s_remaining = remaining - above;
          s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - u) << shift);
          s_whole = (u < 8 ? c[u] : 0) == remaining - above && remaining > above;
        }
      }
      __syncthreads();
      remaining = s_remaining;
      prefix = s_prefix;
      mask |= 255u << shift;
      if (s_whole) {
        // Every key of the bin is chosen: they are exactly the keys >= prefix among the
        // candidates, so no lower digit is needed and no tie has to be broken.
        remaining = 0x7fffffff;
        break;
      }
    }
    thr = prefix;
    take_eq = remaining;
  }

  // ---- chosen flags, output positions ----
  int n_eq_before = 0;
  {
    int cnt_eq = 0;
    if (!all)
      for (int j = j0; j < j1; ++j) cnt_eq += keys[j] == thr;
    int tot;
    n_eq_before = block_exclusive_scan(cnt_eq, scan_buf, &tot);
  }
  uint32_t chosen = 0u;      // bit (j - j0) for every owned chunk chosen
  {
    int eq_rank = n_eq_before;
    for (int j = j0; j < j1; ++j) {
      bool c;
      if (all) {
        c = true;
      } else {
        const uint32_t u = keys[j];
        c = u > thr || (u == thr && eq_rank < take_eq);
        eq_rank += u == thr;
      }
      if (c) chosen |= 1u << (j - j0);
    }
  }
  int tot_chosen;
  const int pos0 = block_exclusive_scan(__popc(chosen), scan_buf, &tot_chosen);

  // ---- slot reconciliation ----
  // keys[] is reused: keys[s] = "slot s of the range is kept" (s < k), then keys[k + i] = the
  // i-th free slot of the range.
  __syncthreads();
  const int slot_base = b * k;
  for (int s = threadIdx.x; s < k; s += kThreads) keys[s] = 0u;
  __syncthreads();
  uint32_t kept = 0u;
  for (int j = j0; j < j1; ++j) {
    if (!((chosen >> (j - j0)) & 1u)) continue;
    const int prev = prev_slot(j - j0);
    if (prev >= slot_base && prev < slot_base + k) {
      if (atomicExch(&keys[prev - slot_base], 1u) != 0u) s_flag = 1;   // two chunks, one slot
      kept |= 1u << (j - j0);
    }
  }
  __syncthreads();
  const int sper = (k + kThreads - 1) / kThreads;
  const int s0 = min(k, static_cast<int>(threadIdx.x) * sper);
  const int s1 = min(k, s0 + sper);
  int nfree = 0;
  for (int s = s0; s < s1; ++s) nfree += keys[s] == 0u;
  int tot_free;
  int free_rank = block_exclusive_scan(nfree, scan_buf, &tot_free);
  uint32_t free_bits = 0u;
  for (int s = s0; s < s1; ++s)
    if (keys[s] == 0u) free_bits |= 1u << (s - s0);
  __syncthreads();
  for (int s = s0; s < s1; ++s)
    if ((free_bits >> (s - s0)) & 1u) keys[k + free_rank++] = static_cast<uint32_t>(s);
  __syncthreads();

  const uint32_t newcomers = chosen & ~kept;
  int tot_new;
  int new_rank = block_exclusive_scan(__popc(newcomers), scan_buf, &tot_new);

  // ---- outputs ----
  int pos = pos0;
  int32_t* list = p.pagein_list + static_cast<size_t>(b) * k * 2;
  int slot_r[kPre];                 // the new slots of the first kPre owned chunks (-1: not chosen)
#pragma unroll
  for (int t = 0; t < kPre; ++t) slot_r[t] = -1;
  for (int j = j0; j < j1; ++j) {
    const uint32_t bit = 1u << (j - j0);
    if (!(chosen & bit)) continue;
    int slot;
    if (kept & bit) {
      slot = prev_slot(j - j0);
    } else {
      slot = slot_base + static_cast<int>(keys[k + new_rank]);
      list[2 * new_rank] = c0 + j;
      list[2 * new_rank + 1] = slot;
      ++new_rank;
    }
    p.res_ids[out0 + pos] = j;
    p.res_slots[out0 + pos] = slot;
#pragma unroll
    for (int u = 0; u < kPre; ++u) slot_r[u] = j - j0 == u ? slot : slot_r[u];
    ++pos;
  }
  __syncthreads();   // every read of slot_of_chunk is done before it is rewritten
  {
    int opos = pos0;
    for (int j = j0; j < j1; ++j) {
      const int t = j - j0;
      int v = -1;
      if ((chosen >> t) & 1u) {
        if (t < kPre) {
          v = slot_r[0];
#pragma unroll
          for (int u = 1; u < kPre; ++u) v = t == u ? slot_r[u] : v;
        } else {
          v = p.res_slots[out0 + opos];
        }
        ++opos;
      }
      p.slot_of_chunk[c0 + j] = v;
    }
  }
  if (threadIdx.x == 0) {
    p.cu_res[b + 1] = out0 + kk;
    if (b == 0) p.cu_res[0] = 0;
    p.pagein_count[b] = tot_new;
    if (s_flag) atomicOr(p.err, kErrDeviceInput);
  }
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
  // keys[] holds max(n, 2k) words: the score keys first, then the slot table and the free list.
  const size_t words = static_cast<size_t>(p.max_n > 2 * p.k ? p.max_n : 2 * p.k);
  const size_t smem = (words > 0 ? words : 1) * sizeof(uint32_t);
  static size_t done[64] = {};
  cudaError_t e = ensure_smem_limit(select_kernel, smem, done);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(p.num_seqs), dim3(kThreads), smem, stream, p);
}

}  // namespace vfy
