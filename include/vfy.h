/*
 * vfy.h -- C ABI of libvfy.so, the GB300 (sm_103a) speculative-decoding verify step.
 *
 * One decode step of speculative decoding verifies a block of q = D + 1 tokens (the last
 * committed token plus D drafted tokens) in one batched target forward and commits only the
 * tokens the target itself would emit ("Laguna XS 2.1 33B on a RTX 3090: 296 tok/s peak,
 * 152 tok/s at 256K context" (lucebox), section "The model, fast MoE with a drafter in the box";
 * "The Death of the Compute-Moat ...", section "DFlash Drafters and the End of Speculative Loss").
 * This library holds the data-parallel hot path of that step:
 *
 *   vfy_select_resident  residency top-k over per-chunk scores + slot reconciliation
 *   vfy_page_in          bit-exact copy of newly resident chunks from pinned host memory
 *   vfy_append_full/_swa the block's K/V rows into the chunk store, pool slot or ring
 *   vfy_attend_full      full-attention layer over the resident chunks of a KVFlash-style pool
 *   vfy_attend_swa       sliding-window layer over a position ring
 *   vfy_accept           fused argmax + greedy acceptance
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers named host_* are host pointers; every other pointer is DEVICE memory on the
 *    context's device. All memory is owned by the caller. The library owns only the context and
 *    the workspace it allocates in vfy_create (split partials, counters, an error word).
 *  - No call allocates memory or synchronises the host, except vfy_create, vfy_destroy and
 *    vfy_get_status. Every other call only enqueues kernels on `stream`, so it can be captured
 *    in a CUDA graph. Per-step values (lengths, lists, offsets, counts) are read from device
 *    memory, so one captured graph serves every step.
 *  - A context's workspace is shared by its calls: calls on one context must be ordered (one
 *    stream, or streams joined by events). Use one context per concurrent stream.
 *  - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16). Indices are int32.
 *  - Host-detectable errors (null pointers, misalignment, sizes beyond the context's capacities)
 *    return VFY_EINVAL and launch nothing. A failed launch returns VFY_ECUDA. Errors found on the
 *    device (an out-of-range chunk id or slot in a device list, a sequence longer than a
 *    capacity) skip the offending element, set a sticky device error word and are reported by
 *    the next vfy_get_status as VFY_EDEVICE_INPUT. Device code never traps.
 *  - Every device-side wait is bounded; a wait that runs out sets VFY_EDEVICE_TIMEOUT in the
 *    error word and the kernel returns.
 */
#ifndef VFY_H
#define VFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VFY_API __attribute__((visibility("default")))
#else
#define VFY_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* vfy_stream_t; /* the same handle as cudaStream_t / CUstream */

typedef enum vfy_status {
  VFY_OK = 0,
  VFY_EINVAL = 1,          /* bad argument; nothing was launched */
  VFY_ECUDA = 2,           /* a CUDA runtime call failed */
  VFY_ENOMEM = 3,          /* vfy_create could not allocate its workspace */
  VFY_EUNSUPPORTED = 4,    /* device is not sm_103 / configuration not supported */
  VFY_EDEVICE_INPUT = 5,   /* a device-side list held an out-of-range entry (it was skipped) */
  VFY_EDEVICE_TIMEOUT = 6  /* a bounded device wait ran out */
} vfy_status;

typedef struct vfy_ctx vfy_ctx; /* opaque, owned by the library */

/* Capacities and shapes, fixed for the life of a context. */
typedef struct vfy_config {
  int num_q_heads;          /* Hq (16 for the Laguna XS shape; 4 in the tiny case) */
  int num_kv_heads;         /* Hkv (4; 1); Hq must be a multiple of Hkv, G = Hq / Hkv */
  int head_dim;             /* d: 64 or 128 */
  int chunk_tokens;         /* pool chunk length: must be 64 ("cold 64-token chunks") */
  int window;               /* sliding-window width in positions, self included (512) */
  int ring_len;             /* ring slots per sequence and KV head (2048), multiple of 64 */
  int max_seqs;             /* largest num_seqs of any call */
  int max_queries_per_seq;  /* largest q (D + 1 for a verify block; up to a prefill-sized block):
                               q * G <= 4096. Each 128 of the q * G rows is one row tile,
                               with CTAs and split partials of its own */
  int max_splits;           /* split-KV partitions per (sequence, KV head) the workspace holds,
                               1..64 */
  float softmax_scale;      /* 0 -> 1 / sqrt(head_dim) */
} vfy_config;

/* Create a context on `device` (which must be an sm_103 GPU) and allocate its workspace.
 * Returns VFY_EINVAL for an invalid config, VFY_EUNSUPPORTED for another GPU, VFY_ENOMEM. */
VFY_API vfy_status vfy_create(const vfy_config* cfg, int device, vfy_ctx** out);

/* Free the context and its workspace (synchronises the device). NULL is ignored. */
VFY_API void vfy_destroy(vfy_ctx* ctx);

/* Synchronise `stream`, read and clear the sticky device error word and return what it held
 * (VFY_OK, VFY_EDEVICE_INPUT or VFY_EDEVICE_TIMEOUT). Not capturable (it synchronises). */
VFY_API vfy_status vfy_get_status(vfy_ctx* ctx, vfy_stream_t stream);

/* A static string naming a status. */
VFY_API const char* vfy_strerror(vfy_status status);

/* Number of kernels the calls on this context have enqueued so far (a captured call counts once,
 * however often its graph is replayed); 0 for NULL. Host-side bookkeeping, no device work. */
VFY_API unsigned long long vfy_launch_count(const vfy_ctx* ctx);

/* Override the split counts chosen automatically (0 = automatic; at most max_splits). Tuning
 * knob; the results agree up to rounding for every split count. Full-layer splits over at least
 * 8 resident chunks stream two chunks per pipeline step and finish in a second, combine kernel.
 * Otherwise a layer whose splits per (sequence, KV head) fit one thread-block cluster (at most
 * 16, and what one GPC holds) merges them inside its attention kernel; more splits also go
 * through the combine kernel. */
VFY_API vfy_status vfy_set_splits(vfy_ctx* ctx, int full_splits, int swa_splits);

/* CTAs that copy each chunk in the vfy_page_in calls enqueued afterwards: 1 to 4, or 0 (the
 * default) for 2. Tuning knob; the copy is bit-exact either way. More CTAs keep more host reads in
 * flight, so a page-in alone finishes sooner, but beside running attention kernels the reads in
 * flight slow those kernels down. */
VFY_API vfy_status vfy_set_pagein_ctas(vfy_ctx* ctx, int ctas_per_chunk);

/* Test of the timeout path (0, the default, turns it off). With limit_ns != 0, every CTA of
 * the attention kernels enqueued afterwards first waits on a barrier that nothing completes, for
 * limit_ns nanoseconds. That wait runs out exactly as a pipeline wait that ran out would: it sets
 * VFY_EDEVICE_TIMEOUT in the device error word and the abort flag, the CTA's other waits give up,
 * the copies and MMAs it issued land (under the default limit), it frees its tensor memory and
 * returns; the call's outputs are undefined. The context stays usable: vfy_get_status reports and
 * clears the error, and calls enqueued after the test is turned off produce correct results. No
 * GPU fault, trap or hang is involved. */
VFY_API vfy_status vfy_test_wait_timeout(vfy_ctx* ctx, uint64_t limit_ns);

/* Declare (1) or withdraw (0, the default) that the per-step metadata the attention calls of
 * this context read -- cu_q, seq_len, ring_offset, resident_ids, resident_slots, cu_resident --
 * is written only by work that has completed before those calls' kernels start: host copies made
 * before the calls are enqueued, or kernels joined to the stream through an event wait or a
 * synchronisation. Not by a kernel earlier on the same stream: under programmatic dependent
 * launch a kernel starts while the kernels before it still run. The attention kernels then read
 * that metadata before they wait for the previous kernel, which takes one memory round trip per
 * layer off the critical path. Q, the K/V data and the resident lists' entries beyond the
 * per-sequence offsets are read after that wait. The 40-layer
 * pass meets the condition (its residency lists come from a side stream that the layer chain
 * joins by events). Applies to calls enqueued afterwards. */
VFY_API vfy_status vfy_set_stable_metadata(vfy_ctx* ctx, int stable);

/*
 * vfy_select_resident -- chunk-residency top-k and slot reconciliation.
 * Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "Three optimizations", item 1: the pool
 * holds 8K of the context on the GPU in 64-token chunks, cold chunks page to host RAM, and a
 * drafter scores which chunks deserve residency. The pages name no selection rule; this call
 * keeps the k best-scored chunks of each sequence.
 *
 *  scores        fp32 [cu_chunks[B]]   residency score of every chunk of every sequence.
 *                Order: higher first; ties to the lower chunk index; -0 == +0; NaN below all
 *                numbers. (Callers give the chunks holding the verify block the score +inf.)
 *  cu_chunks     int32 [B+1]           chunk offsets of the sequences (device)
 *  num_seqs      B (host) <= max_seqs
 *  max_chunks_per_seq  host bound on cu_chunks[b+1]-cu_chunks[b] (<= 32768)
 *  k             resident budget per sequence (host) in [1, 4096]. Sequence b owns pool slots
 *                [b*k, b*k + k).
 *  slot_of_chunk int32 [cu_chunks[B]]  IN/OUT: pool slot of every chunk, -1 if not resident.
 *                A chosen chunk whose slot lies in its sequence's range keeps it; the other chosen
 *                chunks, ascending, take the free slots of the range, ascending; chunks not
 *                chosen get -1. An entry outside the range counts as not resident.
 *  resident_ids  int32 [sum_b min(k, n_b)] OUT: chosen chunk indices (sequence-local),
 *                ascending within each sequence, sequences concatenated
 *  resident_slots int32 [same]         OUT: their pool slots
 *  cu_resident   int32 [B+1]           OUT: offsets into resident_ids / resident_slots
 *  pagein_list   int32 [B*k][2]        OUT: for sequence b, entries [b*k, b*k + pagein_count[b])
 *                hold (global chunk index = cu_chunks[b] + local id, slot) of newly resident
 *                chunks in ascending chunk order
 *  pagein_count  int32 [B]             OUT
 * Device errors: a sequence longer than max_chunks_per_seq, or two chunks holding the same
 * slot, sets VFY_EDEVICE_INPUT (the sequence's outputs are then unspecified).
 */
VFY_API vfy_status vfy_select_resident(vfy_ctx* ctx, const float* scores, const int32_t* cu_chunks,
                                       int num_seqs, int max_chunks_per_seq, int k,
                                       int32_t* slot_of_chunk, int32_t* resident_ids,
                                       int32_t* resident_slots, int32_t* cu_resident,
                                       int32_t* pagein_list, int32_t* pagein_count,
                                       vfy_stream_t stream);

/*
 * vfy_page_in -- bit-exact copy of newly resident chunks into their pool slots.
 * Source: same page, item 1 ("cold 64-token chunks page to host RAM bit-exact").
 *
 *  host_k, host_v  bf16 [num_host_chunks][Hkv][64][d] pinned host memory (cudaHostAlloc /
 *                  cudaMallocHost / torch pin_memory), readable by the device. Owned by caller.
 *  k_pool, v_pool  bf16 [num_slots][Hkv][64][d] device pool of one layer
 *  pagein_list, pagein_count, num_seqs, k: as written by vfy_select_resident
 * Each listed (chunk, slot) copies host chunk `chunk` (all KV heads, K and V) into pool slot
 * `slot`. Entries with chunk or slot out of range are skipped (VFY_EDEVICE_INPUT).
 * Pointers must be 16-byte aligned. Outside stream capture the call checks that the host store
 * is pinned (or device / managed) memory and returns VFY_EINVAL for pageable memory.
 */
VFY_API vfy_status vfy_page_in(vfy_ctx* ctx, const uint16_t* host_k, const uint16_t* host_v,
                               int64_t num_host_chunks, uint16_t* k_pool, uint16_t* v_pool,
                               int num_slots, const int32_t* pagein_list,
                               const int32_t* pagein_count, int num_seqs, int k,
                               vfy_stream_t stream);

/*
 * vfy_attend_full -- verify attention of one full-attention layer over the resident chunks.
 * Source: same page, "The model ..." (the block of 16 drafts + 1 is verified in one batched
 * forward) and item 1 (the pool). Sequence b's block query i sits at position
 * p_i = seq_len[b] - q_b + i and attends every resident position p <= p_i:
 *     O = softmax(scale * Q K^T) V,  q-head g reads KV head g / G.
 *
 *  q              bf16 [cu_q[B]][Hq][d]   block queries, sequence b owns rows cu_q[b]..cu_q[b+1]
 *  cu_q           int32 [B+1]            (device) q_b = cu_q[b+1]-cu_q[b] <= max_queries_per_seq
 *  k_pool, v_pool bf16 [num_slots][Hkv][64][d]   16-byte aligned
 *  resident_ids, resident_slots, cu_resident   as written by vfy_select_resident, or any list of
 *                 (chunk index, slot) per sequence (e.g. every chunk, for an all-resident pool)
 *  max_resident_per_seq  host bound on cu_resident[b+1]-cu_resident[b] (sets the split count)
 *  seq_len        int32 [B]              L_b, counting the block
 *  out            bf16 [cu_q[B]][Hq][d]  OUT
 *  lse            fp32 [cu_q[B]][Hq]     OUT, natural-log sum-exp of the scaled scores;
 *                 NULL to skip. A row that attends no position gets out = 0, lse = -inf.
 * Values at positions some block query attends must be finite (a masked entry contributes
 * P = 0, and 0 * inf is NaN on the tensor core). Rows past seq_len and chunks not in the list
 * may hold anything.
 * Device errors: a slot outside [0, num_slots) or q_b beyond capacity: element skipped,
 * VFY_EDEVICE_INPUT.
 */
VFY_API vfy_status vfy_attend_full(vfy_ctx* ctx, const uint16_t* q, const int32_t* cu_q,
                                   const uint16_t* k_pool, const uint16_t* v_pool, int num_slots,
                                   const int32_t* resident_ids, const int32_t* resident_slots,
                                   const int32_t* cu_resident, int max_resident_per_seq,
                                   const int32_t* seq_len, uint16_t* out, float* lse,
                                   int num_seqs, vfy_stream_t stream);

/*
 * vfy_attend_swa -- verify attention of one sliding-window layer read from a position ring.
 * Source: same page, item 3 ("Ring caches for the sliding-window layers": a 512-token window
 * kept in a small position ring, slot = pos mod 2048). Position p of sequence b sits in slot
 * (p + ring_offset[b]) mod ring_len; block query i (position p_i) attends positions
 * [max(0, p_i - window + 1), p_i].
 *
 *  q, cu_q, seq_len, out, lse  as in vfy_attend_full
 *  k_ring, v_ring bf16 [B][Hkv][ring_len][d]; slots outside the block's window may hold anything
 *  ring_offset    int32 [B]  (device) write-head offset phi_b (taken mod ring_len)
 */
VFY_API vfy_status vfy_attend_swa(vfy_ctx* ctx, const uint16_t* q, const int32_t* cu_q,
                                  const uint16_t* k_ring, const uint16_t* v_ring,
                                  const int32_t* ring_offset, const int32_t* seq_len,
                                  uint16_t* out, float* lse, int num_seqs, vfy_stream_t stream);

/*
 * vfy_append_full -- write the verify block's K/V rows of one full-attention layer where later
 * steps read them. Source: "Laguna XS 2.1 33B on a RTX 3090" (lucebox), "Three optimizations"
 * item 1 (a pool of 64-token chunks; cold chunks page to host RAM bit-exact).
 * Block token i of sequence b sits at position p = seq_len[b] - q_b + i. Its K and V rows (all
 * KV heads) go to row p mod 64 of chunk cu_chunks[b] + p / 64 of the chunk store and, when that
 * chunk holds a pool slot, to the same row of the slot. Writing through to the store keeps every
 * chunk's host copy bit-exact with the pool, so a chunk that vfy_select_resident evicts needs no
 * page-out: its slot is simply reassigned.
 *
 *  k_new, v_new   bf16 [cu_q[B]][Hkv][d]   the block's K/V rows (sequence b owns rows cu_q[b]..)
 *  cu_q, seq_len  as in vfy_attend_full
 *  cu_chunks      int32 [B+1] (device)     sequence b's chunks are cu_chunks[b].. of the store
 *  slot_of_chunk  int32 [cu_chunks[B]] (device)   pool slot of each chunk, -1 if not resident
 *  host_k, host_v bf16 [num_host_chunks][Hkv][64][d]   the chunk store: pinned host memory (written
 *                 over the host link) or device memory; outside capture, pageable memory is
 *                 rejected with VFY_EINVAL
 *  k_pool, v_pool bf16 [num_slots][Hkv][64][d]
 * Pointers must be 16-byte aligned. Call it before the layer's vfy_attend_full.
 * Device errors: a chunk index outside [0, num_host_chunks), or q_b beyond capacity: the token
 * is skipped, VFY_EDEVICE_INPUT.
 */
VFY_API vfy_status vfy_append_full(vfy_ctx* ctx, const uint16_t* k_new, const uint16_t* v_new,
                                   const int32_t* cu_q, const int32_t* seq_len, const int32_t* cu_chunks,
                                   const int32_t* slot_of_chunk, uint16_t* host_k, uint16_t* host_v,
                                   int64_t num_host_chunks, uint16_t* k_pool, uint16_t* v_pool,
                                   int num_slots, int num_seqs, vfy_stream_t stream);

/*
 * vfy_append_swa -- write the verify block's K/V rows of one sliding-window layer into its ring.
 * Source: same page, item 3 (slot = pos mod 2048, here (pos + ring_offset[b]) mod ring_len).
 *  k_new, v_new   bf16 [cu_q[B]][Hkv][d];  cu_q, seq_len, ring_offset as in vfy_attend_swa
 *  k_ring, v_ring bf16 [B][Hkv][ring_len][d]
 * Call it before the layer's vfy_attend_swa.
 * Device errors: q_b beyond capacity: the sequence's tokens are skipped, VFY_EDEVICE_INPUT.
 */
VFY_API vfy_status vfy_append_swa(vfy_ctx* ctx, const uint16_t* k_new, const uint16_t* v_new,
                                  const int32_t* cu_q, const int32_t* seq_len, const int32_t* ring_offset,
                                  uint16_t* k_ring, uint16_t* v_ring, int num_seqs, vfy_stream_t stream);

/*
 * vfy_gate_depths -- confidence-gated draft depths for a ragged verify batch (host function, no
 * device work, no context). Source: "Width vs. Depth: Speculating on the Margin" (draft depth
 * allocated unevenly by drafter confidence beats fixed depths; it needs ragged speculation).
 * Sequence b's drafted positions are each accepted with probability confidence[b] in [0, 1],
 * independently, so depth D commits 1 + c + ... + c^D tokens in expectation. The depths
 * maximise that sum under sum_b (depths[b] + 1) <= row_budget and 0 <= depths[b] <= max_depth
 * (rows are handed out one at a time to the largest gain c^(D+1), ties to the lower index).
 *  confidence  fp32 [num_seqs] host;  depths  int32 [num_seqs] host, OUT
 * Returns VFY_EINVAL for a confidence outside [0, 1] (or NaN) or a negative count.
 */
VFY_API vfy_status vfy_gate_depths(const float* confidence, int num_seqs, int row_budget, int max_depth,
                                   int32_t* depths);

/*
 * vfy_accept -- fused argmax over fp32 logits + greedy acceptance.
 * Source: same page, "The model ..." (commit only tokens the target itself would emit) and
 * "The Death of the Compute-Moat", "DFlash Drafters ..." (verify, commit, fallback).
 * a_r = argmax_v logits[r][v] (ties to the lowest index; a NaN is the maximum, first NaN wins).
 * For sequence b with rows r = cu_rows[b] .. cu_rows[b+1]-1 (D_b + 1 rows) and drafts
 * d_j = drafts[cu_rows[b] - b + j], j < D_b:
 *     n_b = length of the longest prefix with a_{cu_rows[b]+j} == d_j
 *     accepted_len[b] = n_b, bonus[b] = a_{cu_rows[b]+n_b}
 *     committed[cu_rows[b] + j] = d_j (j < n_b), bonus (j == n_b), -1 (j > n_b)
 *
 *  logits    fp32 [cu_rows[B]][vocab]
 *  vocab     host int, >= 1
 *  drafts    int32 [cu_rows[B] - B]
 *  cu_rows   int32 [B+1] (device)
 *  max_rows  host bound on cu_rows[B] (sets the grid), <= max_seqs * max_queries_per_seq
 */
VFY_API vfy_status vfy_accept(vfy_ctx* ctx, const float* logits, int vocab, const int32_t* drafts,
                              const int32_t* cu_rows, int max_rows, int32_t* accepted_len,
                              int32_t* bonus, int32_t* committed, int num_seqs,
                              vfy_stream_t stream);

/*
 * vfy_accept_static -- vfy_accept for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point: it exists for integration. Some callers
 * cannot call cudaMalloc: code running inside an allocator or memory pool it must not re-enter,
 * plug-ins whose host owns every device allocation, and deployments whose device memory budget is
 * fixed before decoding starts. vfy_accept needs a context, and vfy_create allocates; this call
 * needs neither. Its scratch (argmax keys, a CTA ticket, an error word) is one fixed 8 KiB array in
 * the library's device memory, held by every GPU that loads the library until the process exits.
 *
 * Arguments and results are those of vfy_accept, on the CURRENT device (`stream` must belong to
 * it), with max_rows (a host bound on cu_rows[B]) at most 1024: a larger max_rows returns
 * VFY_EINVAL and launches nothing. device_error (nullable) is a caller-owned device int32 that
 * receives VFY device error bits (1 = out-of-range list, 2 = timeout) OR-ed in; the caller clears it.
 * With device_error NULL, device errors go to a word inside the scratch array that the next
 * call clears and no call reads: they are discarded, and the outputs of a call that hit one are
 * unspecified. Pass a word to see them.
 *  - The first call on a device looks up the scratch array's device address
 *    (cudaGetSymbolAddress) with that device current. Make that first call before any stream
 *    capture. The address is cached per device; a call that finds another context current on
 *    the device (after cudaDeviceReset, say) looks it up again, so make the first call after a
 *    reset outside capture too. Device ordinals of 64 and above return VFY_EUNSUPPORTED.
 *  - Each call clears the scratch on `stream` (cudaMemsetAsync) and then launches the kernel; it
 *    calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every call on a device shares the one array: calls whose work overlaps on the GPU (other
 *    streams, other host threads) race and give wrong results. Order them.
 */
VFY_API vfy_status vfy_accept_static(const float* logits, int vocab, const int32_t* drafts,
                                     const int32_t* cu_rows, int num_seqs, int max_rows,
                                     int32_t* accepted_len, int32_t* bonus, int32_t* committed,
                                     int32_t* device_error, vfy_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VFY_H */
