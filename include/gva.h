/*
 * gva.h - C ABI of the gapped variable-length attention forward for GB300 (sm_103a).
 *
 * The operation (cosmos-framework PR #302 "fix(mot): gapped replay on GPUs
 * FlashAttention-4 has no kernels for (sm120)", section "What"; the FA4 varlen
 * forward with seqused_q / seqused_k it replaces):
 *
 *   Segment b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1] and key rows
 *   cu_seqlens_k[b] .. cu_seqlens_k[b+1]. Only its first seqused_q[b] query rows
 *   attend, and only to its first seqused_k[b] keys. For every such row r and query
 *   head h (KV head h / (Hq/Hkv), contiguous GQA groups):
 *       O[r,h,:]  = softmax_j(s * <Q[r,h,:], K[j,hkv,:]>) . V[j,hkv,:]
 *       LSE[h,r]  = ln sum_j exp(s * <Q[r,h,:], K[j,hkv,:]>)     (natural log, FP32)
 *   Rows past a segment's used length are not written (O and LSE). A segment with
 *   seqused_k[b] = 0 gets O = +0 and LSE = -inf on its used rows. Keys past
 *   seqused_k[b] (gap or zero padding) never enter the softmax: each attended zero
 *   key would add exp(0) = 1 to the denominator (TensorRT-LLM issue #18687,
 *   "actual behavior").
 *
 * Layouts (all tensors contiguous, row-major, device memory):
 *   Q, O : [total_q, Hq, d]      Q bf16; O bf16 or fp32 (gva_dtype)
 *   K, V : [total_k, Hkv, d]     bf16
 *   LSE  : [Hq, total_q]         fp32 (the PyTorch unpadded-varlen LSE layout named
 *                                in the review of PR #302)
 *   total_q = cu_seqlens_q[B], total_k = cu_seqlens_k[B] (rows of the buffers).
 *
 * Entry points:
 *   plans        gva_plan (used prefixes), gva_plan_ranges (several key ranges per
 *                segment), gva_plan_causal (block-causal), gva_plan_get_info,
 *                gva_plan_inspect (the work lists, host only), gva_plan_destroy
 *   forward      gva_forward, gva_forward_noalloc (no plan, no allocation)
 *   merge        gva_lse_merge (FP32 LSE merge of partial results)
 *   backward     gva_backward_workspace_size, gva_backward (dQ, dK, dV)
 *   status       gva_device_status, gva_status_string, gva_last_error
 *
 * Conventions:
 *   - Every function returns a gva_status and never throws. On failure,
 *     gva_last_error() gives a human-readable reason (thread-local).
 *   - gva_forward, gva_lse_merge and gva_backward are asynchronous on `stream`,
 *     allocate nothing, and do not synchronise the host. gva_plan allocates and
 *     uploads a small device work list once per geometry (from host ints: no
 *     device-to-host read).
 *   - The caller owns every tensor. A plan owns only its device work list and is
 *     released by gva_plan_destroy; no launch that uses it may still be in flight.
 *   - Two launches that share a plan may run concurrently: a plan holds no per-call
 *     state except a device error word (see gva_device_status).
 */
#ifndef GVA_H_
#define GVA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define GVA_API __attribute__((visibility("default")))
#else
#define GVA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GVA_OK = 0,
  GVA_ERR_INVALID_ARG = 1,  /* bad geometry, null / misaligned pointer, bad count */
  GVA_ERR_UNSUPPORTED = 2,  /* head_dim, head grouping or device not supported */
  GVA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
  GVA_ERR_DEVICE_CHECK = 4  /* a kernel reported a device-side check failure */
} gva_status;

typedef enum { GVA_BF16 = 0, GVA_FP32 = 1 } gva_dtype;

typedef struct gva_plan* gva_plan_t;

/* Geometry summary of a plan (for tests and benchmarks). */
typedef struct {
  int32_t num_segments, num_heads_q, num_heads_kv, head_dim;
  int64_t total_q, total_k;
  int32_t num_work_items;   /* forward work items (segment, kv head, 2 x 128-row Q tiles) */
  int32_t num_merge_units;  /* merge work units (up to 16 used rows of one segment, sized so
                               that the units fill whole waves of about 4 CTAs per SM) */
  int32_t grid_ctas;        /* persistent CTAs one forward launch uses */
  int32_t sm_count;
  double used_flops;        /* 4 * d * Hq * sum_b seqused_q[b] * seqused_k[b] */
} gva_plan_info;

/*
 * gva_plan - validate one launch's segment geometry and build its work list.
 *
 * Cites: PR #302 "What" (cu_seqlens / seqused semantics) and its review (build the
 * gather plan from the runtime's host ints, with no device sync inside the op).
 *
 *   cu_seqlens_q, cu_seqlens_k : HOST int32 [num_segments + 1], non-negative and
 *                                non-decreasing (segment capacities are differences;
 *                                a first offset above 0 lets a visibility partition
 *                                address a sub-range of the same K/V buffers)
 *   seqused_q, seqused_k       : HOST int32 [num_segments], 0 <= used <= capacity
 *   num_heads_q % num_heads_kv == 0, group g = num_heads_q / num_heads_kv <= 128,
 *   num_heads_q <= 256; a 128-row Q tile folds floor(128 / g) tokens of the g query
 *   heads of one KV head (GQA folding, PR #312 "Problem and behavior"), so any g up
 *   to 128 is accepted (rows past floor(128 / g) * g of a tile are idle)
 *   head_dim in {64, 128}
 *
 * The plan is bound to the current CUDA device, which must be sm_103 (GB300).
 * Errors: GVA_ERR_INVALID_ARG for bad geometry (checked before any CUDA call),
 * GVA_ERR_UNSUPPORTED for head_dim / grouping / device, GVA_ERR_CUDA if the upload
 * fails. On error *out_plan is set to NULL.
 */
GVA_API gva_status gva_plan(const int32_t* cu_seqlens_q, const int32_t* seqused_q, const int32_t* cu_seqlens_k,
                    const int32_t* seqused_k, int32_t num_segments, int32_t num_heads_q, int32_t num_heads_kv,
                    int32_t head_dim, gva_plan_t* out_plan);

/*
 * gva_plan_ranges - like gva_plan, but each segment's keys are several row ranges of
 * K/V, attended as one softmax over their concatenation.
 *
 * Cites: cosmos-framework PR #312, "Problem and behavior" (visibility partitions of
 * one launch, normally merged with an FP32 LSE merge: here they run as one launch
 * with no merge), and TensorRT-LLM issue #18687, "additional notes" (after an
 * all-to-all the valid keys of a sample are not a prefix: rank-major order).
 *
 *   cu_seqlens_q, seqused_q : HOST int32, as for gva_plan
 *   key_range_offsets       : HOST int32 [num_segments + 1], starts at 0,
 *                             non-decreasing: segment b owns ranges
 *                             key_range_offsets[b] .. key_range_offsets[b+1]
 *   key_range_starts/lengths: HOST int32 [key_range_offsets[num_segments]]: K/V rows
 *                             start .. start + length, each inside [0, total_k)
 *   total_k                 : rows of the K and V buffers
 * A segment whose ranges hold no key is keyless (O = 0, LSE = -inf on used rows).
 * Ranges may lie anywhere (also overlapping other segments' ranges). gva_forward and
 * gva_lse_merge take a plan from either builder. Errors as for gva_plan.
 */
GVA_API gva_status gva_plan_ranges(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                                   const int32_t* key_range_offsets, const int32_t* key_range_starts,
                                   const int32_t* key_range_lengths, int64_t total_k, int32_t num_heads_q,
                                   int32_t num_heads_kv, int32_t head_dim, gva_plan_t* out_plan);

/*
 * gva_plan_causal - like gva_plan, with block-causal masking inside each segment.
 *
 * Cites: cosmos-framework PR #312, "Problem and behavior" (causal replay split into
 * maskless visibility partitions merged by an FP32 LSE merge) and PR #302, "What" (the
 * FA4 varlen forward it stands in for also takes a causal flag): here one launch
 * applies the mask.
 *
 * Row token i of segment b (i < seqused_q[b]) sits at key position
 * pos = i + seqused_k[b] - seqused_q[b] (the queries are the last positions of the
 * segment's key sequence) and attends keys j < min(seqused_k[b],
 * (floor(pos / causal_block) + 1) * causal_block); causal_block = 1 is token-causal. A
 * row that sees no key gets O = +0 and LSE = -inf. Each work item only loads the key
 * blocks its last row sees. causal_block >= 1, else GVA_ERR_INVALID_ARG; other
 * arguments and errors as for gva_plan.
 */
GVA_API gva_status gva_plan_causal(const int32_t* cu_seqlens_q, const int32_t* seqused_q,
                                   const int32_t* cu_seqlens_k, const int32_t* seqused_k, int32_t num_segments,
                                   int32_t causal_block, int32_t num_heads_q, int32_t num_heads_kv,
                                   int32_t head_dim, gva_plan_t* out_plan);

/*
 * gva_forward - the gapped varlen attention forward of one launch (one kernel).
 *
 * Cites: PR #302 "What" (used rows attend used keys; rows past the used length left
 * as they are; a keyless segment gets zero output and -inf LSE), TensorRT-LLM issue
 * #18687 "actual behavior" (padded keys must not enter the softmax denominator).
 *
 *   q, k, v   : DEVICE bf16, layouts above, 16-byte aligned, must not alias out/lse
 *   out       : DEVICE, out_dtype (GVA_BF16 or GVA_FP32), [total_q, Hq, d], 16-byte
 *               aligned (full tiles are written by TMA stores, which require it)
 *   lse       : DEVICE fp32 [Hq, total_q], 16-byte aligned
 *   softmax_scale : s in the formula; <= 0 selects 1/sqrt(head_dim)
 *   stream    : CUDA stream the kernel is enqueued on
 *
 * Only used rows of out / lse are written. Asynchronous; returns GVA_ERR_INVALID_ARG for a
 * NULL or misaligned pointer and GVA_ERR_CUDA if the launch fails. Device-side waits are bounded; a timeout is recorded in the plan's
 * error word (gva_device_status) instead of hanging.
 */
GVA_API gva_status gva_forward(gva_plan_t plan, const void* q, const void* k, const void* v, void* out,
                       gva_dtype out_dtype, float* lse, float softmax_scale, cudaStream_t stream);

/*
 * gva_lse_merge - combine partial forwards over disjoint key sets of the same rows.
 *
 * Cites: cosmos-framework PR #312, "Problem and behavior" (visibility partitions are
 * combined by an FP32 LSE merge). For every used row r and head h of `plan`'s query
 * geometry:
 *   L = max_p lses[p][h,r];  L = -inf  ->  out = +0, lse = -inf
 *   else w_p = exp(lses[p][h,r] - L), lse = L + ln sum_p w_p,
 *        out[r,h,:] = sum_p w_p outs[p][r,h,:] / sum_p w_p
 * A partition whose lse is -inf contributes nothing (its output is not read).
 *
 *   num_parts : 1 .. 8
 *   outs      : HOST array of num_parts DEVICE pointers, in_dtype, [total_q, Hq, d]
 *   lses      : HOST array of num_parts DEVICE fp32 pointers, [Hq, total_q]
 *   out, lse  : DEVICE outputs (out_dtype / fp32); out may alias outs[0] and lse may
 *               alias lses[0] (every element is read before it is written); rows past
 *               the used length are not written.
 * outs and out must be 16-byte aligned, lses and lse 4-byte aligned. Computed in FP32.
 * Asynchronous on `stream`; no allocation.
 * Errors: GVA_ERR_INVALID_ARG for a NULL plan or pointer, num_parts outside 1 .. 8, a bad
 * dtype, a misaligned pointer or a plan built on another device; GVA_ERR_CUDA if the
 * launch fails.
 */
GVA_API gva_status gva_lse_merge(gva_plan_t plan, int32_t num_parts, const void* const* outs, gva_dtype in_dtype,
                         const float* const* lses, void* out, gva_dtype out_dtype, float* lse,
                         cudaStream_t stream);

/*
 * gva_backward_workspace_size - bytes of device workspace gva_backward needs.
 *
 * Writes Hq * total_q * 4 (one fp32 D value per row and query head) to *bytes.
 */
GVA_API gva_status gva_backward_workspace_size(gva_plan_t plan, size_t* bytes);

/*
 * gva_backward - gradients of gva_forward with respect to Q, K and V.
 *
 * Cites: cosmos-framework PR #302, review (the FP32 fallback covers the forward only)
 * and PR #312, "Problem and behavior" (the SM120 path raises on backward): the
 * gradients the forward's definition implies. For each segment b, query head h (KV
 * head h_kv = h / (Hq/Hkv)), used row i and used key j, with P the softmax of the
 * forward recomputed from `lse`:
 *   dP_ij = <dO_i, V_j>,  D_i = <dO_i, O_i>,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = s sum_j dS_ij K_j
 *   dK_j = s sum_{i, h of the KV group} dS_ij Q_i,   dV_j = sum_{i, h} P_ij dO_i
 * For plans from gva_plan (maskless), gva_plan_causal (the gradients of the block-causal
 * forward: P is zero past each row's key limit, and a row that sees no key gets dQ = 0)
 * and gva_plan_ranges (segment b's keys are its ranges, as in the forward). Key ranges
 * may overlap, across segments or within one (TensorRT-LLM issue #18687, "additional
 * notes": after an all-to-all the valid keys are not a prefix): a K/V row's dK / dV is
 * then the sum of the contributions of every segment that attends it, counted once per
 * range of that segment that covers the row, as the forward counts them. The plan cuts
 * the union of the ranges where any range starts or ends and gives each piece (at most
 * 128 rows) one unit per KV head that walks the Q tiles of all its attending segments,
 * so each dK / dV row still has a single writer.
 *
 *   q, k, v   : DEVICE bf16, as given to gva_forward
 *   out, lse  : DEVICE, the forward's bf16 output [total_q, Hq, d] and fp32 LSE
 *               [Hq, total_q] (natural log) for the same inputs and scale
 *   d_out     : DEVICE bf16 [total_q, Hq, d], the gradient of the output
 *   dq        : DEVICE dq_dtype (GVA_BF16 / GVA_FP32) [total_q, Hq, d]
 *   dk, dv    : DEVICE dkv_dtype [total_k, Hkv, d]
 *   workspace : DEVICE, 16-byte aligned, >= gva_backward_workspace_size bytes; scratch
 *               for the duration of the call (stream order)
 *   softmax_scale : the forward's s; <= 0 selects 1/sqrt(head_dim)
 *   stream    : CUDA stream the kernels are enqueued on
 *
 * Rows written: dq on used rows (zero on the used rows of a keyless segment); dk / dv
 * on every K/V row some segment's keys include (zero where no attending segment has a
 * used row). Gap rows and
 * K/V rows outside every segment's keys are not written; their contents (even NaN) do not affect any
 * written value. Every pointer 16-byte aligned; inputs must not alias outputs. No
 * atomics: the result is deterministic. Asynchronous; bounded device waits as for
 * gva_forward (gva_device_status reports a timeout).
 */
GVA_API gva_status gva_backward(gva_plan_t plan, const void* q, const void* k, const void* v, const void* out,
                                const void* d_out, const float* lse, void* dq, gva_dtype dq_dtype, void* dk,
                                void* dv, gva_dtype dkv_dtype, void* workspace, size_t workspace_bytes,
                                float softmax_scale, cudaStream_t stream);

/*
 * gva_plan_inspect - the work lists a plan would hold, built on the host only.
 *
 * For tests and tuning: no CUDA call is made and no plan is created. The geometry is
 * that of gva_plan / gva_plan_causal (HOST arrays, same validation: cu_seqlens_k and
 * seqused_k, key_range_offsets NULL), or that of gva_plan_ranges (key_range_offsets,
 * key_range_starts, key_range_lengths and total_k; cu_seqlens_k / seqused_k are then
 * not read and causal_block must be 0). causal_block: 0 maskless, > 0 as
 * gva_plan_causal. grid (>= 1): the SM count the work lists (and the merge units,
 * summary->num_merge_units) are laid out for;
 * walk_list selects the list `walk` describes (0 forward items, 1 dQ items, 2 dK / dV
 * units). Fills *summary (backward_ok: always 1) and copies at most *_capacity records
 * into each non-NULL array (8 int32 per record; 2 for kv_segs; one per entry for walk):
 *   items     : forward work items {q_row0, q_rows, blk0, nblk, head_kv, n_tiles, k_len,
 *               q_pos0}, longest first;
 *   walk      : one int32 per entry of the chosen list as its kernel walks it (with
 *               g = min(grid, the list's length) CTAs, CTA c reads entry r * g + c in
 *               even rounds r and r * g + g - 1 - c in odd ones): the entry's index in
 *               the sorted list, or -1 for padding;
 *   bwd_items : backward dQ items, same layout, one Q tile each;
 *   kv_units  : backward dK / dV units {key_row0, keys, seg0, n_tiles, head_kv, tile0,
 *               key_pos0, pos_shift}, one per piece of at most 128 K/V rows and KV head:
 *               rows key_row0 .. key_row0 + keys, run against n_tiles Q tiles of the
 *               segments kv_segs[seg0 ..] (starting at tile tile0 of the first);
 *   kv_segs   : {q_row0, q_used} of the segments the units list (summary->num_kv_segs).
 * Errors: GVA_ERR_INVALID_ARG for a NULL summary, a negative causal_block, ranges with a
 * causal_block, grid < 1, walk_list outside 0 .. 2 or bad geometry; GVA_ERR_UNSUPPORTED
 * as gva_plan.
 */
typedef struct {
  int32_t num_work_items, num_key_blocks, num_merge_units, num_bwd_items, num_kv_units, backward_ok;
  double used_flops;
  int32_t num_walk_entries, num_kv_segs;
} gva_work_summary;
GVA_API gva_status gva_plan_inspect(const int32_t* cu_seqlens_q, const int32_t* seqused_q,
                                    const int32_t* cu_seqlens_k, const int32_t* seqused_k, int32_t num_segments,
                                    const int32_t* key_range_offsets, const int32_t* key_range_starts,
                                    const int32_t* key_range_lengths, int64_t total_k, int32_t causal_block,
                                    int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t grid,
                                    int32_t walk_list, gva_work_summary* summary, int32_t* items,
                                    int32_t items_capacity, int32_t* walk, int32_t walk_capacity,
                                    int32_t* bwd_items, int32_t bwd_items_capacity, int32_t* kv_units,
                                    int32_t kv_units_capacity, int32_t* kv_segs, int32_t kv_segs_capacity);

/* Release a plan's device memory. NULL is accepted. Synchronous with respect to the
 * host only through cudaFree. */
GVA_API gva_status gva_plan_destroy(gva_plan_t plan);

/* Fill *info with the plan's geometry summary. */
GVA_API gva_status gva_plan_get_info(gva_plan_t plan, gva_plan_info* info);

/* Synchronise the device, read and clear the plan's device error word. Returns
 * GVA_ERR_DEVICE_CHECK if a kernel of this plan recorded a bounded-wait timeout or a
 * check failure since the last call, GVA_OK otherwise. For tests and debugging; it
 * is not needed on the fast path.
 * With plan = NULL it does the same for the error word of gva_forward_noalloc's
 * scratch on the current device, which reports the last gva_forward_noalloc launch
 * there (each call clears the word before its launch); GVA_OK if none has run, and
 * GVA_ERR_UNSUPPORTED without a usable CUDA device. */
GVA_API gva_status gva_device_status(gva_plan_t plan);

/*
 * gva_forward_noalloc - gva_forward for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart for this entry point. It exists for callers that may
 * not call cudaMalloc: a serving runtime that hands out all device memory from its own
 * pool, code under a fixed memory budget, or a loop that must not take cudaMalloc's
 * implicit device synchronisation. gva_plan allocates a device work list; this call
 * instead builds the work list on the host and copies it, on `stream`, into a scratch
 * array that is part of the library image (GVA_NOALLOC_MAX_WORK_ITEMS work items of 32
 * bytes, GVA_NOALLOC_MAX_KEY_BLOCKS key blocks of 8 bytes and an error word, about
 * 1.5 MiB, held by every GPU that loads the library until the process exits). It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * Arguments: the geometry exactly as for gva_plan (HOST arrays, same rules), then the
 * tensors, scale and stream exactly as for gva_forward (the caller still owns and
 * passes inputs and outputs). A launch needing more than GVA_NOALLOC_MAX_WORK_ITEMS
 * work items (items = sum over segments of ceil(seqused_q / (2 * floor(128 / (Hq/Hkv)))) * Hkv)
 * or more than GVA_NOALLOC_MAX_KEY_BLOCKS key blocks (sum over segments of
 * ceil(seqused_k / 128)) is refused with GVA_ERR_INVALID_ARG before any GPU work.
 *
 * The first call on a device resolves the scratch array's address for that device
 * (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture. Every call overwrites the shared scratch and clears its error word
 * on `stream`: calls on one stream are ordered, but calls whose kernels may overlap on
 * the GPU (different streams without ordering) race on the scratch and must not be
 * made.
 *
 * Host wait: the work list is copied from a host staging array in ordinary (pageable)
 * memory, and the CUDA runtime starts such a copy only after the work already queued
 * on `stream` has finished. Each call therefore blocks the calling thread until that
 * earlier work is done (the kernel itself is then launched asynchronously).
 *
 * Device errors: a bounded wait that times out inside the kernel leaves rows
 * unwritten and records it in the scratch's error word, not in the return value;
 * gva_device_status(NULL) reads and clears that word for the current device.
 */
#define GVA_NOALLOC_MAX_WORK_ITEMS 32768
#define GVA_NOALLOC_MAX_KEY_BLOCKS 65536
GVA_API gva_status gva_forward_noalloc(const int32_t* cu_seqlens_q, const int32_t* seqused_q,
                                       const int32_t* cu_seqlens_k, const int32_t* seqused_k,
                                       int32_t num_segments, int32_t num_heads_q, int32_t num_heads_kv,
                                       int32_t head_dim, const void* q, const void* k, const void* v, void* out,
                                       gva_dtype out_dtype, float* lse, float softmax_scale, cudaStream_t stream);

/* Static description of a status code. */
GVA_API const char* gva_status_string(gva_status status);

/* Detail of the last error returned on the calling thread ("" if none). */
GVA_API const char* gva_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GVA_H_ */
