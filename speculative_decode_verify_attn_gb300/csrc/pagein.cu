// Page-in: bit-exact copy of newly resident chunks from pinned host memory into pool slots.
// Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "Three optimizations", item 1 ("cold
// 64-token chunks page to host RAM bit-exact").
// The device reads the host store directly (zero-copy over the host link), so the (chunk, slot)
// list can stay in device memory and the copy can live inside a captured CUDA graph. Grid:
// x = list entry (sequence b, entry i < k), y = part of the chunk (1 to 4 CTAs per chunk, set per
// call); entries past pagein_count[b] return at once. Each thread keeps 2 x 2 independent 16-byte
// loads in flight. The copy is bound by the host link's latency, and host reads in flight slow the
// attention kernels that run beside it. Measured in the 40-layer pass on GB300 against 2 CTAs per
// chunk: 3 or 4 cost the pass 2 and 12 us; 1 for the page-ins after the first was 0.1 us/layer
// faster on one box and 0.02 slower on another; half the loads in flight per thread made the
// later page-ins late for their layers.
#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

__global__ void __launch_bounds__(kThreads) page_in_kernel(const PageInParams p) {
  pdl_wait();
  const int e = blockIdx.x;
  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.k));
  const int i = e - b * p.k;
  if (b >= p.num_seqs || i >= p.count[b]) return;
  const int chunk = p.list[2 * e];
  const int slot = p.list[2 * e + 1];
  if (chunk < 0 || chunk >= p.num_host_chunks || slot < 0 || slot >= p.num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, kErrDeviceInput);
    return;
  }
  const long long n16 = p.chunk_elems / 8;                   // 16-byte words per chunk
  const long long per = (n16 + gridDim.y - 1) / gridDim.y;
  const long long w0 = blockIdx.y * per;
  const long long w1 = min(n16, w0 + per);
  const uint4* sk = reinterpret_cast<const uint4*>(p.host_k + chunk * p.chunk_elems);
  const uint4* sv = reinterpret_cast<const uint4*>(p.host_v + chunk * p.chunk_elems);
  uint4* dk = reinterpret_cast<uint4*>(p.k_pool + static_cast<long long>(slot) * p.chunk_elems);
  uint4* dv = reinterpret_cast<uint4*>(p.v_pool + static_cast<long long>(slot) * p.chunk_elems);
  for (long long w = w0 + threadIdx.x; w < w1; w += static_cast<long long>(kThreads) * kUnroll) {
    uint4 a[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long x = w + static_cast<long long>(u) * kThreads;
      if (x < w1) {
        a[u] = __ldcs(sk + x);
        c[u] = __ldcs(sv + x);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long x = w + static_cast<long long>(u) * kThreads;
      if (x < w1) {
        dk[x] = a[u];
        dv[x] = c[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_page_in(const PageInParams& p, cudaStream_t stream) {
  if (p.parts < 1 || p.parts > kMaxPageInCtas) return cudaErrorInvalidValue;
  dim3 grid(p.num_seqs * p.k, p.parts);
  return launch_pdl(page_in_kernel, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace vfy
