// Host side of the C ABI: context and workspace, argument validation, tensor maps, launches.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "ptx.cuh"
#include "vfy_internal.cuh"

struct vfy_ctx {
  vfy_config cfg;
  int device;
  int num_sms;
  float scale;
  // split partials
  float* part_o;
  float* part_ml;
  // acceptance workspace
  unsigned long long* accept_keys;
  int accept_rows_cap;
  unsigned int* accept_counter;
  // sticky device error word
  int* err;
  int full_splits;   // 0 = automatic
  int swa_splits;
  unsigned long long launches;   // kernels enqueued through this context
  int row_tiles;                 // ceil(max_queries_per_seq * G / 128)
  unsigned long long timeout_test_ns;   // see vfy_test_wait_timeout
  int stable_metadata;                // see vfy_set_stable_metadata
  int pagein_ctas;                    // see vfy_set_pagein_ctas (0 = 2)
};

namespace {

using vfy::kChunk;
using vfy::kMaxRows;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D view [rows][d] of a bf16 array; 64 x 64 boxes (128 bytes wide) with the 128-byte swizzle.
bool make_tmap(CUtensorMap* map, const void* base, uint64_t rows, int d) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Makes the context's device current for the duration of a call and restores the caller's.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      prev = -1;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

}  // namespace

#define VFY_REQUIRE(c)           \
  do {                           \
    if (!(c)) return VFY_EINVAL; \
  } while (0)

#define VFY_CUDA(call)           \
  do {                           \
    if ((call) != cudaSuccess) { \
      (void)cudaGetLastError();  \
      return VFY_ECUDA;          \
    }                            \
  } while (0)

extern "C" {

unsigned long long vfy_launch_count(const vfy_ctx* ctx) { return ctx != nullptr ? ctx->launches : 0ull; }

const char* vfy_strerror(vfy_status s) {
  switch (s) {
    case VFY_OK: return "ok";
    case VFY_EINVAL: return "invalid argument";
    case VFY_ECUDA: return "CUDA runtime error";
    case VFY_ENOMEM: return "out of device memory";
    case VFY_EUNSUPPORTED: return "unsupported device or configuration";
    case VFY_EDEVICE_INPUT: return "a device-side list or length was out of range (element skipped)";
    case VFY_EDEVICE_TIMEOUT: return "a bounded device wait ran out";
  }
  return "unknown status";
}

vfy_status vfy_create(const vfy_config* cfg_in, int device, vfy_ctx** out) {
  VFY_REQUIRE(cfg_in != nullptr && out != nullptr);
  *out = nullptr;
  const vfy_config cfg = *cfg_in;
  VFY_REQUIRE(cfg.num_q_heads >= 1 && cfg.num_kv_heads >= 1 && cfg.num_q_heads % cfg.num_kv_heads == 0);
  VFY_REQUIRE(cfg.head_dim == 64 || cfg.head_dim == 128);
  VFY_REQUIRE(cfg.chunk_tokens == kChunk);
  VFY_REQUIRE(cfg.max_seqs >= 1 && cfg.max_queries_per_seq >= 1 && cfg.max_splits >= 1);
  VFY_REQUIRE(cfg.max_splits <= 64 && cfg.max_seqs <= 65535 && cfg.num_kv_heads <= 65535);
  const int group = cfg.num_q_heads / cfg.num_kv_heads;
  VFY_REQUIRE(static_cast<long long>(cfg.max_queries_per_seq) * group <= static_cast<long long>(kMaxRows) * vfy::kMaxRowTiles);
  VFY_REQUIRE(cfg.window >= 1 && cfg.ring_len >= kChunk && cfg.ring_len % kChunk == 0);
  // The ring must hold the union window of a block plus one tile of slack, so that the
  // slot-aligned tiles covering it are distinct.
  VFY_REQUIRE(static_cast<long long>(cfg.window) + cfg.max_queries_per_seq - 1 + kChunk <= cfg.ring_len);
  VFY_REQUIRE(cfg.softmax_scale >= 0.f && std::isfinite(cfg.softmax_scale));

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    (void)cudaGetLastError();
    return VFY_EINVAL;
  }
  cudaDeviceProp prop;
  VFY_CUDA(cudaGetDeviceProperties(&prop, device));
  if (!(prop.major == 10 && prop.minor == 3)) return VFY_EUNSUPPORTED;   // sm_103 only

  DeviceGuard guard(device);
  if (!guard.ok) return VFY_ECUDA;
  if (get_encode() == nullptr) return VFY_EUNSUPPORTED;
  vfy_ctx* ctx = new (std::nothrow) vfy_ctx();
  if (ctx == nullptr) return VFY_ENOMEM;
  ctx->cfg = cfg;
  ctx->device = device;
  ctx->num_sms = prop.multiProcessorCount;
  ctx->scale = cfg.softmax_scale > 0.f ? cfg.softmax_scale : 1.0f / std::sqrt(static_cast<float>(cfg.head_dim));

  ctx->row_tiles = ceil_div(static_cast<long long>(cfg.max_queries_per_seq) * group, kMaxRows);
  const size_t parts =
      static_cast<size_t>(cfg.max_seqs) * ctx->row_tiles * cfg.num_kv_heads * cfg.max_splits * kMaxRows;
  ctx->accept_rows_cap = cfg.max_seqs * cfg.max_queries_per_seq;
  bool ok = cudaMalloc(&ctx->part_o, parts * cfg.head_dim * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&ctx->part_ml, parts * 2 * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&ctx->accept_keys, ctx->accept_rows_cap * sizeof(unsigned long long)) == cudaSuccess &&
            cudaMalloc(&ctx->accept_counter, sizeof(unsigned int)) == cudaSuccess &&
            cudaMalloc(&ctx->err, sizeof(int)) == cudaSuccess;
  if (ok)
    ok = cudaMemset(ctx->accept_keys, 0, ctx->accept_rows_cap * sizeof(unsigned long long)) == cudaSuccess &&
         cudaMemset(ctx->accept_counter, 0, sizeof(unsigned int)) == cudaSuccess &&
         cudaMemset(ctx->err, 0, sizeof(int)) == cudaSuccess &&
         cudaMemset(ctx->part_ml, 0, parts * 2 * sizeof(float)) == cudaSuccess &&
         cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    (void)cudaGetLastError();
    vfy_destroy(ctx);
    return VFY_ENOMEM;
  }
  *out = ctx;
  return VFY_OK;
}

void vfy_destroy(vfy_ctx* ctx) {
  if (ctx == nullptr) return;
  {
    DeviceGuard guard(ctx->device);
    cudaDeviceSynchronize();
    cudaFree(ctx->part_o);
    cudaFree(ctx->part_ml);
    cudaFree(ctx->accept_keys);
    cudaFree(ctx->accept_counter);
    cudaFree(ctx->err);
    (void)cudaGetLastError();
  }
  delete ctx;
}

vfy_status vfy_get_status(vfy_ctx* ctx, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  VFY_CUDA(cudaStreamSynchronize(s));
  VFY_CUDA(cudaMemcpy(&word, ctx->err, sizeof(int), cudaMemcpyDeviceToHost));
  VFY_CUDA(cudaMemset(ctx->err, 0, sizeof(int)));
  VFY_CUDA(cudaDeviceSynchronize());
  if (word & vfy::kErrTimeout) return VFY_EDEVICE_TIMEOUT;
  if (word & vfy::kErrDeviceInput) return VFY_EDEVICE_INPUT;
  return VFY_OK;
}

vfy_status vfy_set_splits(vfy_ctx* ctx, int full_splits, int swa_splits) {
  VFY_REQUIRE(ctx != nullptr);
  VFY_REQUIRE(full_splits >= 0 && full_splits <= ctx->cfg.max_splits);
  VFY_REQUIRE(swa_splits >= 0 && swa_splits <= ctx->cfg.max_splits);
  ctx->full_splits = full_splits;
  ctx->swa_splits = swa_splits;
  return VFY_OK;
}

vfy_status vfy_set_pagein_ctas(vfy_ctx* ctx, int ctas_per_chunk) {
  VFY_REQUIRE(ctx != nullptr && ctas_per_chunk >= 0 && ctas_per_chunk <= vfy::kMaxPageInCtas);
  ctx->pagein_ctas = ctas_per_chunk;
  return VFY_OK;
}

vfy_status vfy_test_wait_timeout(vfy_ctx* ctx, uint64_t limit_ns) {
  VFY_REQUIRE(ctx != nullptr);
  ctx->timeout_test_ns = limit_ns;
  return VFY_OK;
}

vfy_status vfy_set_stable_metadata(vfy_ctx* ctx, int stable) {
  VFY_REQUIRE(ctx != nullptr && (stable == 0 || stable == 1));
  ctx->stable_metadata = stable;
  return VFY_OK;
}

vfy_status vfy_select_resident(vfy_ctx* ctx, const float* scores, const int32_t* cu_chunks, int num_seqs,
                               int max_chunks_per_seq, int k, int32_t* slot_of_chunk, int32_t* resident_ids,
                               int32_t* resident_slots, int32_t* cu_resident, int32_t* pagein_list,
                               int32_t* pagein_count, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && scores != nullptr && cu_chunks != nullptr && slot_of_chunk != nullptr);
  VFY_REQUIRE(resident_ids != nullptr && resident_slots != nullptr && cu_resident != nullptr);
  VFY_REQUIRE(pagein_list != nullptr && pagein_count != nullptr);
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  VFY_REQUIRE(k >= 1 && k <= vfy::kMaxSelectK);
  VFY_REQUIRE(max_chunks_per_seq >= 0 && max_chunks_per_seq <= vfy::kMaxSelectChunks);
  VFY_REQUIRE(static_cast<long long>(num_seqs) * k <= INT_MAX / 2);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  vfy::SelectParams p;
  p.scores = scores;
  p.cu_chunks = cu_chunks;
  p.num_seqs = num_seqs;
  p.max_n = max_chunks_per_seq;
  p.k = k;
  p.slot_of_chunk = slot_of_chunk;
  p.res_ids = resident_ids;
  p.res_slots = resident_slots;
  p.cu_res = cu_resident;
  p.pagein_list = pagein_list;
  p.pagein_count = pagein_count;
  p.err = ctx->err;
  VFY_CUDA(vfy::launch_select(p, reinterpret_cast<cudaStream_t>(stream)));
  ++ctx->launches;
  return VFY_OK;
}

// Outside stream capture: check that a caller's "host" buffers are addressable by the device
// (pinned, managed or device memory) and translate pinned host pointers to their device
// addresses. During capture the check is skipped (the pointers are used as given).
static vfy_status device_view(cudaStream_t s, void** ptrs, int n) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return VFY_ECUDA;
  if (cap != cudaStreamCaptureStatusNone) return VFY_OK;
  for (int i = 0; i < n; ++i) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
      (void)cudaGetLastError();
      return VFY_EINVAL;
    }
    if (a.type == cudaMemoryTypeUnregistered) return VFY_EINVAL;
    if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) ptrs[i] = a.devicePointer;
  }
  return VFY_OK;
}

vfy_status vfy_page_in(vfy_ctx* ctx, const uint16_t* host_k, const uint16_t* host_v, int64_t num_host_chunks,
                       uint16_t* k_pool, uint16_t* v_pool, int num_slots, const int32_t* pagein_list,
                       const int32_t* pagein_count, int num_seqs, int k, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && host_k != nullptr && host_v != nullptr && k_pool != nullptr && v_pool != nullptr);
  VFY_REQUIRE(pagein_list != nullptr && pagein_count != nullptr);
  VFY_REQUIRE(aligned16(host_k) && aligned16(host_v) && aligned16(k_pool) && aligned16(v_pool));
  VFY_REQUIRE(num_host_chunks >= 1 && num_host_chunks <= INT_MAX && num_slots >= 1);
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs && k >= 1 && k <= vfy::kMaxSelectK);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* dev_ptr[2] = {const_cast<uint16_t*>(host_k), const_cast<uint16_t*>(host_v)};
  const vfy_status st = device_view(s, dev_ptr, 2);
  if (st != VFY_OK) return st;
  vfy::PageInParams p;
  p.host_k = static_cast<const uint16_t*>(dev_ptr[0]);
  p.host_v = static_cast<const uint16_t*>(dev_ptr[1]);
  p.num_host_chunks = num_host_chunks;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.num_slots = num_slots;
  p.list = pagein_list;
  p.count = pagein_count;
  p.num_seqs = num_seqs;
  p.k = k;
  p.chunk_elems = static_cast<long long>(ctx->cfg.num_kv_heads) * kChunk * ctx->cfg.head_dim;
  p.err = ctx->err;
  p.parts = ctx->pagein_ctas > 0 ? ctx->pagein_ctas : 2;
  VFY_CUDA(vfy::launch_page_in(p, s));
  ++ctx->launches;
  return VFY_OK;
}

vfy_status vfy_append_full(vfy_ctx* ctx, const uint16_t* k_new, const uint16_t* v_new, const int32_t* cu_q,
                           const int32_t* seq_len, const int32_t* cu_chunks, const int32_t* slot_of_chunk,
                           uint16_t* host_k, uint16_t* host_v, int64_t num_host_chunks, uint16_t* k_pool,
                           uint16_t* v_pool, int num_slots, int num_seqs, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && k_new != nullptr && v_new != nullptr && cu_q != nullptr && seq_len != nullptr);
  VFY_REQUIRE(cu_chunks != nullptr && slot_of_chunk != nullptr && host_k != nullptr && host_v != nullptr);
  VFY_REQUIRE(k_pool != nullptr && v_pool != nullptr);
  VFY_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned16(host_k) && aligned16(host_v) &&
              aligned16(k_pool) && aligned16(v_pool));
  VFY_REQUIRE(num_host_chunks >= 1 && num_host_chunks <= INT_MAX && num_slots >= 1);
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* store[2] = {host_k, host_v};
  const vfy_status st = device_view(s, store, 2);
  if (st != VFY_OK) return st;
  vfy::AppendParams p = {};
  p.k_new = k_new;
  p.v_new = v_new;
  p.cu_q = cu_q;
  p.seq_len = seq_len;
  p.num_seqs = num_seqs;
  p.max_q = ctx->cfg.max_queries_per_seq;
  p.token_cap = num_seqs * ctx->cfg.max_queries_per_seq;
  p.hkv = ctx->cfg.num_kv_heads;
  p.head_dim = ctx->cfg.head_dim;
  p.cu_chunks = cu_chunks;
  p.slot_of_chunk = slot_of_chunk;
  p.host_k = static_cast<uint16_t*>(store[0]);
  p.host_v = static_cast<uint16_t*>(store[1]);
  p.num_host_chunks = num_host_chunks;
  p.num_slots = num_slots;
  p.k_dst = k_pool;
  p.v_dst = v_pool;
  p.err = ctx->err;
  VFY_CUDA(vfy::launch_append(false, p, s));
  ++ctx->launches;
  return VFY_OK;
}

vfy_status vfy_append_swa(vfy_ctx* ctx, const uint16_t* k_new, const uint16_t* v_new, const int32_t* cu_q,
                          const int32_t* seq_len, const int32_t* ring_offset, uint16_t* k_ring, uint16_t* v_ring,
                          int num_seqs, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && k_new != nullptr && v_new != nullptr && cu_q != nullptr && seq_len != nullptr);
  VFY_REQUIRE(ring_offset != nullptr && k_ring != nullptr && v_ring != nullptr);
  VFY_REQUIRE(aligned16(k_new) && aligned16(v_new) && aligned16(k_ring) && aligned16(v_ring));
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  vfy::AppendParams p = {};
  p.k_new = k_new;
  p.v_new = v_new;
  p.cu_q = cu_q;
  p.seq_len = seq_len;
  p.num_seqs = num_seqs;
  p.max_q = ctx->cfg.max_queries_per_seq;
  p.token_cap = num_seqs * ctx->cfg.max_queries_per_seq;
  p.hkv = ctx->cfg.num_kv_heads;
  p.head_dim = ctx->cfg.head_dim;
  p.ring_off = ring_offset;
  p.ring_len = ctx->cfg.ring_len;
  p.k_dst = k_ring;
  p.v_dst = v_ring;
  p.err = ctx->err;
  VFY_CUDA(vfy::launch_append(true, p, reinterpret_cast<cudaStream_t>(stream)));
  ++ctx->launches;
  return VFY_OK;
}

static vfy_status attend_common(vfy_ctx* ctx, bool ring, const uint16_t* q, const int32_t* cu_q,
                                const uint16_t* k_src, const uint16_t* v_src, uint64_t src_rows,
                                const int32_t* ids, const int32_t* slots, const int32_t* cu_res, int num_slots,
                                int max_res, const int32_t* ring_offset, const int32_t* seq_len, uint16_t* out,
                                float* lse, int num_seqs, vfy_stream_t stream) {
  const vfy_config& c = ctx->cfg;
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  CUtensorMap tk, tv;
  if (!make_tmap(&tk, k_src, src_rows, c.head_dim) || !make_tmap(&tv, v_src, src_rows, c.head_dim))
    return VFY_EINVAL;
  const int hkv = c.num_kv_heads;
  int splits;
  if (!ring) {
    splits = ctx->full_splits;
    if (splits == 0) {
      if (ctx->row_tiles > 1) {
        // Blocks of several row tiles (prefill-shaped) have (KV head, row tile) items enough to
        // fill the SMs with few splits, and a long split keeps the tensor pipe busier: at most one
        // wave. Measured with 1024 queries over 128 chunks (128 items): 1 split 121 us, 2 splits
        // 130, 3 138, 4 146, 5 (four waves) 155.
        splits = ctx->num_sms / (hkv * num_seqs * ctx->row_tiles);
      } else {
        // One wave of CTAs for one sequence; several waves for a batch, so that the hardware
        // scheduler can balance sequences of different lengths.
        const int target = ctx->num_sms * (num_seqs > 1 ? 4 : 1);
        splits = ceil_div(target, static_cast<long long>(hkv) * num_seqs);
      }
      splits = clampi(splits, 1, max_res > 0 ? max_res : 1);
    }
  } else {
    splits = ctx->swa_splits;
    if (splits == 0) {
      // a row tile's queries: at most 128 / G of them
      const int tile_q = std::min(c.max_queries_per_seq, ceil_div(kMaxRows, c.num_q_heads / hkv));
      const int max_tiles = ceil_div(static_cast<long long>(kChunk - 1) + c.window + tile_q - 1, kChunk);
      const int by_sms = ceil_div(ctx->num_sms, static_cast<long long>(hkv) * num_seqs * ctx->row_tiles);
      splits = clampi(by_sms, 1, max_tiles);
      // With SMs to spare (one tile per split), two more splits than tiles: the splits without a
      // tile only take their share of the cluster merge. Measured on the 40-layer pass (10
      // tiles: 12 splits 10.27-10.29 us/layer against 10.40-10.51 for 10, 11, 13, 14 and 16).
      if (by_sms > max_tiles && max_tiles + 2 <= vfy::kMaxClusterSplits) splits = std::min(max_tiles + 2, by_sms);

    }
  }
  splits = clampi(splits, 1, c.max_splits);

  vfy::AttnParams p;
  p.q = q;
  p.cu_q = cu_q;
  p.seq_len = seq_len;
  p.res_ids = ids;
  p.res_slots = slots;
  p.cu_res = cu_res;
  p.num_slots = num_slots;
  p.ring_off = ring_offset;
  p.ring_len = c.ring_len;
  p.window = c.window;
  p.hq = c.num_q_heads;
  p.hkv = hkv;
  p.group = c.num_q_heads / hkv;
  p.num_splits = splits;
  p.max_q = c.max_queries_per_seq;
  p.row_tiles = ctx->row_tiles;
  p.scale_log2 = ctx->scale * 1.4426950408889634f;
  p.part_o = ctx->part_o;
  p.part_ml = ctx->part_ml;
  p.timeout_test_ns = ctx->timeout_test_ns;
  p.stable_metadata = ctx->stable_metadata;
  p.err = ctx->err;
  // Full-layer splits over many resident chunks take wide tiles (their combine is a small part
  // of a long split). Otherwise up to kMaxClusterSplits splits (and no more than one GPC holds)
  // merge inside the attention kernel, as one thread-block cluster per (sequence, KV head, row
  // tile); more go through the combine.
  const bool wide = !ring && ceil_div(max_res > 0 ? max_res : 1, splits) >= vfy::kWideMinChunks;
  // A single split of a long block writes O itself (no combine launch).
  const bool direct = wide && splits == 1;
  const bool merge = !direct && !wide && splits <= vfy::kMaxClusterSplits &&
                     splits <= vfy::attend_merge_limit(ring, c.head_dim);
  const vfy::AttnTiles tiles = merge    ? vfy::AttnTiles::kMerge
                              : direct ? vfy::AttnTiles::kWideDirect
                              : wide   ? vfy::AttnTiles::kWide
                                       : vfy::AttnTiles::kNarrow;
  p.out = merge || direct ? out : nullptr;
  p.lse = merge || direct ? lse : nullptr;
  p.token_cap = num_seqs * c.max_queries_per_seq;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  VFY_CUDA(vfy::launch_attend(ring, c.head_dim, tiles, p, tk, tv, num_seqs, s));
  ++ctx->launches;
  if (merge || direct) return VFY_OK;

  vfy::CombineParams cp;
  cp.cu_q = cu_q;
  cp.seq_len = seq_len;
  cp.num_seqs = num_seqs;
  cp.hq = c.num_q_heads;
  cp.hkv = hkv;
  cp.group = p.group;
  cp.num_splits = splits;
  cp.max_q = c.max_queries_per_seq;
  cp.row_tiles = ctx->row_tiles;
  cp.token_cap = num_seqs * c.max_queries_per_seq;
  cp.stable_metadata = ctx->stable_metadata;
  cp.part_o = ctx->part_o;
  cp.part_ml = ctx->part_ml;
  cp.out = out;
  cp.lse = lse;
  cp.err = ctx->err;
  VFY_CUDA(vfy::launch_combine(c.head_dim, cp, s));
  ++ctx->launches;
  return VFY_OK;
}

vfy_status vfy_attend_full(vfy_ctx* ctx, const uint16_t* q, const int32_t* cu_q, const uint16_t* k_pool,
                           const uint16_t* v_pool, int num_slots, const int32_t* resident_ids,
                           const int32_t* resident_slots, const int32_t* cu_resident, int max_resident_per_seq,
                           const int32_t* seq_len, uint16_t* out, float* lse, int num_seqs,
                           vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && q != nullptr && cu_q != nullptr && k_pool != nullptr && v_pool != nullptr);
  VFY_REQUIRE(resident_ids != nullptr && resident_slots != nullptr && cu_resident != nullptr);
  VFY_REQUIRE(seq_len != nullptr && out != nullptr);
  VFY_REQUIRE(aligned16(q) && aligned16(k_pool) && aligned16(v_pool) && aligned16(out));
  VFY_REQUIRE(lse == nullptr || (reinterpret_cast<uintptr_t>(lse) & 3u) == 0);
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  VFY_REQUIRE(num_slots >= 1 && max_resident_per_seq >= 0);
  const uint64_t rows = static_cast<uint64_t>(num_slots) * ctx->cfg.num_kv_heads * kChunk;
  VFY_REQUIRE(rows <= static_cast<uint64_t>(INT_MAX));
  return attend_common(ctx, false, q, cu_q, k_pool, v_pool, rows, resident_ids, resident_slots, cu_resident,
                       num_slots, max_resident_per_seq, nullptr, seq_len, out, lse, num_seqs, stream);
}

vfy_status vfy_attend_swa(vfy_ctx* ctx, const uint16_t* q, const int32_t* cu_q, const uint16_t* k_ring,
                          const uint16_t* v_ring, const int32_t* ring_offset, const int32_t* seq_len,
                          uint16_t* out, float* lse, int num_seqs, vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && q != nullptr && cu_q != nullptr && k_ring != nullptr && v_ring != nullptr);
  VFY_REQUIRE(ring_offset != nullptr && seq_len != nullptr && out != nullptr);
  VFY_REQUIRE(aligned16(q) && aligned16(k_ring) && aligned16(v_ring) && aligned16(out));
  VFY_REQUIRE(lse == nullptr || (reinterpret_cast<uintptr_t>(lse) & 3u) == 0);
  VFY_REQUIRE(num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  const uint64_t rows = static_cast<uint64_t>(num_seqs) * ctx->cfg.num_kv_heads * ctx->cfg.ring_len;
  VFY_REQUIRE(rows <= static_cast<uint64_t>(INT_MAX));
  return attend_common(ctx, true, q, cu_q, k_ring, v_ring, rows, nullptr, nullptr, nullptr, 0, 0, ring_offset,
                       seq_len, out, lse, num_seqs, stream);
}

vfy_status vfy_accept(vfy_ctx* ctx, const float* logits, int vocab, const int32_t* drafts, const int32_t* cu_rows,
                      int max_rows, int32_t* accepted_len, int32_t* bonus, int32_t* committed, int num_seqs,
                      vfy_stream_t stream) {
  VFY_REQUIRE(ctx != nullptr && logits != nullptr && drafts != nullptr && cu_rows != nullptr);
  VFY_REQUIRE(accepted_len != nullptr && bonus != nullptr && committed != nullptr);
  VFY_REQUIRE(vocab >= 1 && num_seqs >= 1 && num_seqs <= ctx->cfg.max_seqs);
  VFY_REQUIRE(max_rows >= 1 && max_rows <= ctx->accept_rows_cap && max_rows <= 65535);
  VFY_REQUIRE((reinterpret_cast<uintptr_t>(logits) & 3u) == 0);
  DeviceGuard guard(ctx->device);
  if (!guard.ok) return VFY_ECUDA;
  vfy::AcceptParams p;
  p.logits = logits;
  p.vocab = vocab;
  p.drafts = drafts;
  p.cu_rows = cu_rows;
  p.num_seqs = num_seqs;
  p.max_rows = max_rows;
  // About two CTAs per SM over all rows; each CTA scans a whole number of 16-byte words.
  int parts = ceil_div(2LL * ctx->num_sms, max_rows);
  parts = clampi(parts, 1, ceil_div(vocab, 1024));
  int seg = ceil_div(vocab, parts);
  seg = (seg + 3) & ~3;
  p.parts = ceil_div(vocab, seg);
  p.seg = seg;
  p.accepted_len = accepted_len;
  p.bonus = bonus;
  p.committed = committed;
  p.keys = ctx->accept_keys;
  p.counter = ctx->accept_counter;
  p.stable_metadata = ctx->stable_metadata;
  p.err = ctx->err;
  const bool vec4 = (vocab % 4 == 0) && aligned16(logits);
  VFY_CUDA(vfy::launch_accept(p, vec4, reinterpret_cast<cudaStream_t>(stream)));
  ++ctx->launches;
  return VFY_OK;
}

}  // extern "C"
