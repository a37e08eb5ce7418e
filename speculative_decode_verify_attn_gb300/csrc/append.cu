// Block K/V append: the verify block's K/V rows of one layer, written where later steps read them.
// Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "Three optimizations": item 1 (a pool of
// 64-token chunks whose cold chunks live in host RAM bit-exact) and item 3 (window layers keep a
// position ring, slot = pos mod 2048).
//
// Full layers: block token i of sequence b (position p = L_b - q_b + i) goes to row p mod 64 of
// chunk cu_chunks[b] + p / 64 of the chunk store, and to the same row of the chunk's pool slot
// when it has one. Writing through to the store keeps every chunk's host copy bit-exact, so a
// chunk that leaves the pool needs no page-out. Window layers: slot (p + phi_b) mod R of the ring.
//
// One CTA per block token; its threads move the token's K and V rows of every KV head in 16-byte
// words (the store may be pinned host memory, written over the host link).
#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kThreads = 128;

template <bool RING>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
  pdl_launch_dependents();   // the next kernel may launch; it still waits for this grid
  pdl_wait();
  const int t = blockIdx.x;
  const int total = p.cu_q[p.num_seqs];
  if (t >= total || t >= p.token_cap) return;
  int b = 0;                                    // the sequence owning token t (cu_q ascending)
  {
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  const int q0 = p.cu_q[b];
  const int nq = p.cu_q[b + 1] - q0;
  const int L = p.seq_len[b];
  const int i = t - q0;
  if (nq < 1 || nq > p.max_q || L < nq || i < 0 || i >= nq) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrDeviceInput);
    return;
  }
  const long long pos = static_cast<long long>(L) - nq + i;
  const int w_head = p.head_dim / 8;            // 16-byte words per head row
  const int words = p.hkv * w_head;             // per K (or V) row of the token
  const uint4* kn = reinterpret_cast<const uint4*>(p.k_new) + static_cast<size_t>(t) * words;
  const uint4* vn = reinterpret_cast<const uint4*>(p.v_new) + static_cast<size_t>(t) * words;
  if (RING) {
    const int R = p.ring_len;
    const int phi = ((p.ring_off[b] % R) + R) % R;
    const long long slot = (pos + phi) % R;
    for (int x = threadIdx.x; x < 2 * words; x += kThreads) {
      const bool isv = x >= words;
      const int w = isv ? x - words : x;
      const int h = w / w_head, c = w - h * w_head;
      const size_t dst = ((static_cast<size_t>(b) * p.hkv + h) * R + slot) * w_head + c;
      uint4* ring = reinterpret_cast<uint4*>(isv ? p.v_dst : p.k_dst);
      ring[dst] = isv ? vn[w] : kn[w];
    }
  } else {
    const long long chunk = static_cast<long long>(p.cu_chunks[b]) + pos / kChunk;
    const int row = static_cast<int>(pos % kChunk);
    if (chunk < 0 || chunk >= p.num_host_chunks) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrDeviceInput);
      return;
    }
    const int slot = p.slot_of_chunk[chunk];
    const bool resident = slot >= 0 && slot < p.num_slots;
    for (int x = threadIdx.x; x < 2 * words; x += kThreads) {
      const bool isv = x >= words;
      const int w = isv ? x - words : x;
      const int h = w / w_head, c = w - h * w_head;
      const uint4 val = isv ? vn[w] : kn[w];
      const size_t off_row = (static_cast<size_t>(h) * kChunk + row) * w_head + c;
      uint4* store = reinterpret_cast<uint4*>(isv ? p.host_v : p.host_k);
      store[static_cast<size_t>(chunk) * p.hkv * kChunk * w_head + off_row] = val;
      if (resident) {
        uint4* pool = reinterpret_cast<uint4*>(isv ? p.v_dst : p.k_dst);
        pool[static_cast<size_t>(slot) * p.hkv * kChunk * w_head + off_row] = val;
      }
    }
  }
}

}  // namespace

cudaError_t launch_append(bool ring, const AppendParams& p, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(p.token_cap));
  if (ring) return launch_pdl(append_kernel<true>, grid, dim3(kThreads), 0, stream, p);
  return launch_pdl(append_kernel<false>, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace vfy
