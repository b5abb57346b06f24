// Internal types shared by the host API and the kernels.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gva {

// Rows of one Q tile (one TMEM lane per row), keys per K/V block, Q tiles per work item.
constexpr int kTileRows = 128;
constexpr int kBlockKeys = 128;
constexpr int kTilesPerItem = 2;
// Used rows of one segment handled by one merge work unit.
constexpr int kMergeRows = 16;
constexpr int kMaxMergeParts = 8;

// One forward work item: up to 2 x 128 folded rows (tokens x the query heads of one KV
// head) of one segment, attending the segment's used keys. The keys are a list of key
// blocks (see KeyBlock) shared by every item of the segment.
struct alignas(16) WorkItem {
  int32_t q_row0;   // global token row of the item's first token
  int32_t q_rows;   // used tokens covered by the item (1 .. 2 * tokens_per_tile)
  int32_t blk0;     // first key block of the segment in the block table
  int32_t nblk;     // key blocks (0: keyless, epilogue only)
  int32_t head_kv;  // KV head; query heads head_kv * group .. + group - 1
  int32_t n_tiles;  // 1 or 2 Q tiles with used rows
  int32_t k_len;    // used keys in all (sum of the blocks' valid counts)
  int32_t q_pos0;   // block-causal plans: key position of the item's first token
};

// Up to kBlockKeys keys: K/V rows row0 .. row0 + valid (a key range is cut into such
// blocks; only its last block can be partial).
struct alignas(8) KeyBlock {
  int32_t row0;
  int32_t valid;
};

// One unit of the dK / dV kernel: up to kBlockKeys consecutive K/V rows for one KV head,
// run against every Q tile of every segment that attends them. The segments are a run
// of SegRef entries; a segment whose key ranges cover the rows m times appears m times
// (its rows attend each copy of those keys). Each K/V row belongs to exactly one unit
// per KV head, so dK and dV have one writer and need no atomics, even when key ranges
// of several segments (or of one segment) overlap.
struct alignas(16) KvUnit {
  int32_t key_row0;  // global K/V row of the block's first key
  int32_t keys;      // K/V rows in the block (1 .. kBlockKeys)
  int32_t seg0;      // first SegRef of the unit's segments
  int32_t n_tiles;   // Q tiles over all of them (0: no row attends the block, dK = dV = 0)
  int32_t head_kv;
  int32_t tile0;     // first Q tile of the first segment that sees the block (block-causal; else 0)
  int32_t key_pos0;  // block-causal (one segment): index of the block's first key within it
  int32_t pos_shift; // block-causal: key position of the segment's query row 0 (used_k - used_q)
};

// A segment attending a dK / dV unit's keys: its query rows (used rows > 0 only).
struct alignas(8) SegRef {
  int32_t q_row0;  // global token row of the segment's first query
  int32_t q_used;  // used query rows
};

struct alignas(8) MergeUnit {
  int32_t row0;   // global token row of the first row
  int32_t rows;   // used rows in this unit (1 .. kMergeRows)
};

struct FwdParams {
  const WorkItem* items;
  const KeyBlock* blocks;
  int32_t num_items;
  void* out;
  float* lse;
  int64_t total_q;
  int32_t num_heads_q;
  int32_t group;            // Hq / Hkv
  int32_t tokens_per_tile;  // kTileRows / group
  float scale_log2;         // softmax scale * log2(e)
  int32_t causal_block;     // > 0: block-causal masking within each segment
  int32_t out_wide;         // out is 32-byte aligned: rows are stored with 32-byte stores
  int32_t out_tma;          // out has a tensor map: full Q tiles leave through TMA stores
  int* error_flag;
};

struct MergeParams {
  const MergeUnit* units;
  int32_t num_units;
  int32_t num_parts;
  const void* outs[kMaxMergeParts];
  const float* lses[kMaxMergeParts];
  void* out;
  float* lse;
  int64_t total_q;
  int32_t num_heads_q;
  int32_t head_dim;
  int* error_flag;
};

struct BwdParams {
  const WorkItem* items;   // dQ work: one Q tile (up to 128 folded rows) per item
  const KeyBlock* blocks;
  int32_t num_items;
  const KvUnit* kv_units;  // dK / dV work
  const SegRef* kv_segs;   // the segments of each dK / dV unit
  int32_t num_kv_units;
  const float* lse;        // [Hq, total_q] from the forward
  const float* dvec;       // [Hq, total_q]: rowsum(dO * O)
  void* dq;                // [total_q, Hq, d]
  void* dk;                // [total_k, Hkv, d]
  void* dv;
  int64_t total_q;
  int32_t num_heads_q;
  int32_t num_heads_kv;
  int32_t group;
  int32_t tokens_per_tile;
  float scale;             // softmax scale s
  float scale_log2;        // s * log2(e)
  int32_t causal_block;    // > 0: gradients of the block-causal forward
  int* error_flag;
};

// Persistent schedule: in round r, CTA c of a grid of `grid` takes the work-list entry
// at r * grid + c in even rounds and r * grid + (grid - 1 - c) in odd ones. The host
// lays every work list out so that this walk hands each CTA the work it was assigned.
__host__ __device__ inline int item_index(int round, int cta, int grid) {
  return (round & 1) ? round * grid + (grid - 1 - cta) : round * grid + cta;
}

// Device error word bits.
constexpr int kErrWaitTimeout = 1;

// Launchers (defined in gva_fwd.cu / gva_merge.cu). They return the launch error.
// map_o (over out, laid out like map_q) is read only when p.out_tma is set.
cudaError_t launch_forward(int head_dim, bool out_f32, const FwdParams& p, const CUtensorMap& map_q,
                           const CUtensorMap& map_k, const CUtensorMap& map_v, const CUtensorMap& map_o, int grid,
                           cudaStream_t stream);
// The merge runs one persistent CTA per resident slot (as many as fit per SM x sm_count).
cudaError_t launch_merge(bool in_f32, bool out_f32, const MergeParams& p, int sm_count, cudaStream_t stream);
// Dynamic shared memory of the merge launch (and its chunk ring slots), or -1 when the
// partitions' weights leave no room for one chunk of every partition.
int merge_smem_bytes(bool in_f32, int num_parts, int num_heads_q, int* ring_slots);
int forward_smem_bytes(int head_dim);
// Backward: rowsum(dO * O) over used rows, then dQ, then dK / dV (gva_bwd.cu).
// Backward kernels take the block-causal variant when p.causal_block > 0. dq_grid and
// kv_grid are the CTA counts the plan's dQ and dK / dV lists were laid out for.
cudaError_t launch_backward(int head_dim, bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units,
                            int32_t num_units, const void* out, const void* d_out, float* dvec,
                            const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, int dq_grid, int kv_grid, int sm_count,
                            cudaStream_t stream);
// Raise kernel K's dynamic shared-memory limit to `bytes`, once per device: the
// attribute persists, and setting it on every launch is redundant work inside a CUDA
// graph capture. One flag word per kernel instantiation (bit d: device d < 64).
template <auto K>
inline cudaError_t ensure_smem_limit(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Set the calling thread's gva_last_error() text (defined in gva_api.cu).
void set_last_error(const char* message);

// Synchronise the current device, read and clear the error word of the last
// gva_forward_noalloc launch on it (defined in gva_noalloc.cu; GVA_OK if none ran).
// Returns a gva_status value.
int noalloc_device_status();

}  // namespace gva
