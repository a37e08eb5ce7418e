// Fused argmax + greedy acceptance.
// Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "The model, fast MoE with a drafter in the
// box" (commit only tokens the target itself would emit) and "The Death of the Compute-Moat ...",
// "DFlash Drafters and the End of Speculative Loss" (verify, commit, fall back to the target's
// own token when no draft survives).
//
// Phase 1 (every CTA): a vocabulary segment of one logit row is scanned with 16-byte loads and
// reduced to one 64-bit key per row, combined across CTAs with atomicMax. The key orders a row's
// entries exactly like the greedy rule: high 32 bits = the fp32 value mapped to an unsigned
// integer that sorts like the value (every NaN maps to the top, -0 to +0), low 32 bits = the
// complement of the index (so equal values prefer the lower index).
// Phase 2 (the last CTA to finish, by an atomic ticket; no CTA ever waits for another): decode
// the argmax of every row, find each sequence's first draft mismatch with a warp ballot, write
// the accepted length, the bonus token and the committed tokens, then zero the keys and the
// ticket for the next call.
#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;     // float4 loads in flight per thread

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0xffffffffu;  // NaN: above everything
  if (u == 0x80000000u) u = 0u;                              // -0 ties +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack(float x, int idx) {
  return (static_cast<unsigned long long>(order_key(x)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ int unpack_index(unsigned long long key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key & 0xffffffffull));
}

// max that returns NaN when either operand is NaN (fmaxf returns the other operand)
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

template <bool VEC4>
__global__ void __launch_bounds__(kThreads) accept_kernel(const AcceptParams p) {
  __shared__ unsigned long long warp_best[kThreads / 32];
  __shared__ bool is_last;
  pdl_launch_dependents();   // the next kernel may launch; it still waits for this grid
  // The row count is per-step metadata: read before the dependency wait when the caller has
  // declared it stable, after it otherwise. The logits are read after it.
  if (!p.stable_metadata) pdl_wait();
  const int total_rows = p.cu_rows[p.num_seqs];
  if (p.stable_metadata) pdl_wait();
  const int row = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows_done = min(total_rows, p.max_rows);

  // Warp w loads sequence w's row range and its first 32 drafts now, with the logits: only the
  // finishing CTA uses them, but which CTA finishes is known only at the end, and loading them
  // then would add a dependent round trip to the tail of the step.
  int f_r0 = -1, f_r1 = -1, f_draft = -1;
  if (warp < p.num_seqs) {
    f_r0 = p.cu_rows[warp];
    f_r1 = p.cu_rows[warp + 1];
    const int depth = f_r1 - f_r0 - 1;
    if (f_r0 >= 0 && depth >= 0 && f_r1 <= rows_done && lane < depth) f_draft = p.drafts[f_r0 - warp + lane];
  }

  if (row < total_rows && row < p.max_rows) {
    const int v0 = blockIdx.x * p.seg;
    const int v1 = min(p.vocab, v0 + p.seg);
    const float* src = p.logits + static_cast<size_t>(row) * p.vocab;
    unsigned long long best = 0ull;
    if (VEC4) {
      // v0 and the row start are multiples of 4 floats (16 bytes). All of a thread's loads of a
      // round are issued before any is used, so the segment costs about one memory round trip.
      const float4* s4 = reinterpret_cast<const float4*>(src + v0);
      const int n4 = v1 > v0 ? (v1 - v0) >> 2 : 0;
      for (int i0 = threadIdx.x; i0 < n4; i0 += kThreads * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (i0 + u * kThreads < n4) v[u] = __ldcs(s4 + i0 + u * kThreads);
          else v[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        // The round's best key without packing every entry: the largest value by a NaN-propagating
        // max (NaN iff the round holds one), then the lowest index holding that value (a float
        // compare: -0 == +0, the two keys' tie) or, with a NaN, the lowest NaN's index. Padding
        // entries hold -inf at indices past the segment, so they never win a tie.
        float m = -INFINITY;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          m = max_nan(m, max_nan(max_nan(v[u].x, v[u].y), max_nan(v[u].z, v[u].w)));
        int at = 0x7fffffff;
        if (m == m) {
#pragma unroll
          for (int u = kUnroll - 1; u >= 0; --u) {
            const int base = v0 + 4 * (i0 + u * kThreads);
            at = v[u].w == m ? base + 3 : at;
            at = v[u].z == m ? base + 2 : at;
            at = v[u].y == m ? base + 1 : at;
            at = v[u].x == m ? base : at;
          }
        } else {
          m = __uint_as_float(0x7fffffffu);
#pragma unroll
          for (int u = kUnroll - 1; u >= 0; --u) {
            const int base = v0 + 4 * (i0 + u * kThreads);
            at = v[u].w != v[u].w ? base + 3 : at;
            at = v[u].z != v[u].z ? base + 2 : at;
            at = v[u].y != v[u].y ? base + 1 : at;
            at = v[u].x != v[u].x ? base : at;
          }
        }
        if (at != 0x7fffffff) best = umax64(best, pack(m, at));
      }
      for (int i = v0 + 4 * n4 + threadIdx.x; i < v1; i += kThreads) best = umax64(best, pack(src[i], i));
    } else {
      for (int i = v0 + threadIdx.x; i < v1; i += kThreads) best = umax64(best, pack(src[i], i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long b = warp_best[0];
      for (int w = 1; w < kThreads / 32; ++w) b = umax64(b, warp_best[w]);
      atomicMax(p.keys + row, b);
    }
  } else if (threadIdx.x == 0 && row == 0 && blockIdx.x == 0 && total_rows > p.max_rows) {
    atomicOr(p.err, kErrDeviceInput);
  }

  // Ticket: the last CTA of the grid does the acceptance. The add has release semantics (this
  // CTA's key is visible before its ticket); the finishing CTA acquires.
  if (threadIdx.x == 0) {
    const unsigned int total = gridDim.x * gridDim.y;
    unsigned int ticket;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(p.counter) : "memory");
    is_last = (ticket == total - 1);
  }
  __syncthreads();
  if (!is_last) {
    return;
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");

  for (int b = warp; b < p.num_seqs; b += kThreads / 32) {
    const bool pre = b == warp;                      // this warp's preloaded sequence
    const int r0 = pre ? f_r0 : p.cu_rows[b];
    const int r1 = pre ? f_r1 : p.cu_rows[b + 1];
    const int depth = r1 - r0 - 1;
    if (r0 < 0 || depth < 0 || r1 > rows_done) {
      if (lane == 0) atomicOr(p.err, kErrDeviceInput);
      continue;
    }
    const int d0 = r0 - b;   // drafts of sequence b start after the D_b' of earlier sequences
    // Lane j holds the greedy token of row r0 + j and draft j, both loaded in one round trip;
    // the bonus token comes from the lane of the first mismatch (or of row D_b).
    int n = depth, bonus = 0;
    for (int j0 = 0; j0 <= depth; j0 += 32) {
      const int j = j0 + lane;
      const int a = j <= depth ? unpack_index(__ldcg(p.keys + r0 + j)) : -1;
      const int dj = j < depth ? (pre && j0 == 0 ? f_draft : p.drafts[d0 + j]) : -1;
      const unsigned ballot = __ballot_sync(0xffffffffu, j < depth && a != dj);
      if (ballot != 0u) {
        n = j0 + __ffs(ballot) - 1;
        bonus = __shfl_sync(0xffffffffu, a, n - j0);
        break;
      }
      if (depth < j0 + 32) {             // every draft matched: row D_b gives the bonus
        bonus = __shfl_sync(0xffffffffu, a, depth - j0);
        break;
      }
    }
    for (int j = lane; j <= depth; j += 32) {
      int tok = -1;
      if (j < n) tok = pre && j < 32 ? f_draft : p.drafts[d0 + j];   // lane j holds draft j
      else if (j == n) tok = bonus;
      p.committed[r0 + j] = tok;
    }
    if (lane == 0) {
      p.accepted_len[b] = n;
      p.bonus[b] = bonus;
    }
  }
  __syncthreads();
  // Leave the workspace as this call found it: all keys zero, ticket zero.
  // (The kernel's completion makes these writes visible to the next call.)
  for (int r = threadIdx.x; r < p.max_rows; r += kThreads) p.keys[r] = 0ull;
  if (threadIdx.x == 0) *p.counter = 0u;
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, bool vec4, cudaStream_t stream) {
  dim3 grid(p.parts, p.max_rows);
  if (vec4) return launch_pdl(accept_kernel<true>, grid, dim3(kThreads), 0, stream, p);
  return launch_pdl(accept_kernel<false>, grid, dim3(kThreads), 0, stream, p);
}

}  // namespace vfy
