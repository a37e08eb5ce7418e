// Internal declarations shared by the host API (api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "vfy.h"

namespace vfy {

constexpr int kChunk = 64;          // tokens per pool chunk and per attention tile
constexpr int kMaxRowTiles = 32;   // row tiles of 128 per (sequence, KV head): q * G <= 4096
constexpr int kMaxRows = 128;       // block rows of one row tile: the M = 128 side of the MMA
constexpr int kMaxSelectChunks = 32768;
constexpr int kMaxSelectK = 4096;

// ------------------------------ attention ---------------------------------------------------
struct AttnParams {
  const uint16_t* q;          // [T][Hq][d]
  const int32_t* cu_q;        // [B+1]
  const int32_t* seq_len;     // [B]
  // full layers: resident list
  const int32_t* res_ids;
  const int32_t* res_slots;
  const int32_t* cu_res;
  int num_slots;
  // window layers: ring
  const int32_t* ring_off;    // [B]
  int ring_len;
  int window;
  // shapes
  int hq, hkv, group;
  int num_splits;
  int max_q;
  int row_tiles;              // ceil(max_q * G / 128): grid z = B * row_tiles
  float scale_log2;           // softmax scale * log2(e)
  // split partials (workspace)
  float* part_o;              // [B][Hkv][splits][128][d]
  float* part_ml;             // [B][Hkv][splits][128][2] (m in log2 units, l)
  // cluster-merged launches only: the splits of one (b, h) merge in the kernel and write these
  uint16_t* out;              // [T][Hq][d]
  float* lse;                 // [T][Hq] or null
  int token_cap;              // host bound on cu_q[B]
  unsigned long long timeout_test_ns;  // != 0: each CTA first waits that long on a barrier
                                       // nothing completes (the timeout path's test)
  int stable_metadata;        // read the work item before the dependency wait
  int* err;
};

// Splits of one (sequence, KV head) that one cluster can merge in the attention kernel (the
// largest non-portable cluster).
constexpr int kMaxClusterSplits = 16;
constexpr int kMaxPageInCtas = 4;     // CTAs per chunk of a page-in

struct CombineParams {
  const int32_t* cu_q;
  const int32_t* seq_len;
  int num_seqs;
  int hq, hkv, group;
  int num_splits;
  int max_q;
  int row_tiles;
  int token_cap;              // host bound on cu_q[B]
  int stable_metadata;        // read cu_q / seq_len before the dependency wait
  const float* part_o;
  const float* part_ml;
  uint16_t* out;              // [T][Hq][d]
  float* lse;                 // [T][Hq] or null
  int* err;
};

// How an attention launch tiles and finishes its work:
//  kNarrow  one 64-token chunk per tile; the splits' partials go to the combine kernel
//  kWide    two chunks per tile (full layers whose splits hold many chunks: fewer, larger steps
//           for the same bytes); partials go to the combine kernel
//  kMerge   one chunk per tile; the grid's x dimension (the splits) is one cluster, which merges
//           the splits and writes p.out / p.lse itself (no combine launch follows). Returns
//           cudaErrorNotSupported, before launching anything, when such a cluster cannot be
//           resident on this device.
//  kWideDirect  kWide with a single split: the kernel normalises O and writes p.out / p.lse
//           itself (no combine launch)
enum class AttnTiles { kNarrow, kWide, kMerge, kWideDirect };
// A split of a full layer takes wide tiles from this many resident chunks on.
constexpr int kWideMinChunks = 8;
cudaError_t launch_attend(bool ring, int head_dim, AttnTiles tiles, const AttnParams& p, const CUtensorMap& tk,
                          const CUtensorMap& tv, int num_seqs, cudaStream_t stream);
cudaError_t launch_combine(int head_dim, const CombineParams& p, cudaStream_t stream);
// The most splits one merging launch can take on the current device (0 on error).
int attend_merge_limit(bool ring, int head_dim);

// ------------------------------ acceptance --------------------------------------------------
struct AcceptParams {
  const float* logits;
  int vocab;
  const int32_t* drafts;
  const int32_t* cu_rows;
  int num_seqs;
  int max_rows;
  int parts;                  // CTAs per row
  int seg;                    // vocab entries per CTA (multiple of 4)
  int32_t* accepted_len;
  int32_t* bonus;
  int32_t* committed;
  unsigned long long* keys;   // [max_rows] workspace, zero between calls
  unsigned int* counter;      // workspace, zero between calls
  int stable_metadata;        // read cu_rows[num_seqs] before the dependency wait
  int* err;
};
cudaError_t launch_accept(const AcceptParams& p, bool vec4, cudaStream_t stream);

// ------------------------------ residency ---------------------------------------------------
struct SelectParams {
  const float* scores;
  const int32_t* cu_chunks;
  int num_seqs;
  int max_n;
  int k;
  int32_t* slot_of_chunk;
  int32_t* res_ids;
  int32_t* res_slots;
  int32_t* cu_res;
  int32_t* pagein_list;
  int32_t* pagein_count;
  int* err;
};
cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);

struct PageInParams {
  const uint16_t* host_k;
  const uint16_t* host_v;
  long long num_host_chunks;
  uint16_t* k_pool;
  uint16_t* v_pool;
  int num_slots;
  const int32_t* list;
  const int32_t* count;
  int num_seqs;
  int k;
  long long chunk_elems;      // Hkv * 64 * d
  int* err;
  int parts;                  // CTAs per chunk, 1 .. kMaxPageInCtas
};
cudaError_t launch_page_in(const PageInParams& p, cudaStream_t stream);

// ------------------------------ block K/V append ---------------------------------------------
struct AppendParams {
  const uint16_t* k_new;      // [T][Hkv][d]
  const uint16_t* v_new;
  const int32_t* cu_q;        // [B+1]
  const int32_t* seq_len;     // [B]
  int num_seqs;
  int max_q;
  int token_cap;              // host bound on cu_q[B]: the grid
  int hkv, head_dim;
  // full layers: chunk store (write-through) and pool
  const int32_t* cu_chunks;   // [B+1]
  const int32_t* slot_of_chunk;
  uint16_t* host_k;           // [chunks][Hkv][64][d]
  uint16_t* host_v;
  long long num_host_chunks;
  int num_slots;
  // window layers: ring
  const int32_t* ring_off;    // [B]
  int ring_len;
  uint16_t* k_dst;            // pool [slots][Hkv][64][d] or ring [B][Hkv][R][d]
  uint16_t* v_dst;
  int* err;
};
cudaError_t launch_append(bool ring, const AppendParams& p, cudaStream_t stream);

// Launch with the programmatic-stream-serialization attribute so that a kernel's prologue can
// overlap the tail of the kernel before it; every kernel calls griddepcontrol.wait before it
// touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with the grid's x dimension split into clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                               cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the dynamic shared-memory limit of `kernel` once per device (the attribute is per device).
template <typename K>
cudaError_t ensure_smem_limit(K kernel, size_t bytes, size_t* done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (bytes <= 48 * 1024) return cudaSuccess;
  if (dev >= 0 && dev < 64 && done_per_device[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done_per_device[dev] = bytes;
  return e;
}

}  // namespace vfy
