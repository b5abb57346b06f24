// gva_forward_noalloc: the gapped varlen forward for callers that cannot allocate
// device memory.
//
// gva_forward needs a plan, and gva_plan allocates the plan's device work list and
// error word with cudaMalloc. Some callers cannot do that: a serving runtime that owns
// all device memory through its own pool, code that runs under a fixed memory budget,
// or a hot loop that must not hit cudaMalloc's implicit device synchronisation. This
// entry point keeps the work list, the key-block table and the error word in one
// file-scope __device__ array instead. The array is part of the library image, so every
// GPU that loads the library holds it (kNoallocScratchBytes, about 1.5 MiB) until the
// process exits.
//
// Set-up: the first call on a device (with that device current) resolves the array's
// device address with cudaGetSymbolAddress and caches it; make that first call before
// any stream capture. Each call then copies its work list into the array and clears
// the error word, on the caller's stream. The copy comes from a host staging array in
// ordinary (pageable) memory, and the CUDA runtime starts such a copy only once the
// stream's earlier work has finished: each call therefore waits on the host for the
// work already queued on its stream. All calls share the one array, so calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on it
// and must be avoided; calls on one stream are ordered and safe.
//
// A bounded wait that times out inside the kernel leaves rows unwritten and sets the
// error word; gva_device_status(NULL) reads (and clears) that word for the current
// device after synchronising it.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "gva.h"
#include "gva_internal.h"

namespace {

constexpr int32_t kNoallocMaxItems = GVA_NOALLOC_MAX_WORK_ITEMS;
constexpr int32_t kNoallocMaxBlocks = GVA_NOALLOC_MAX_KEY_BLOCKS;
constexpr size_t kNoallocItemBytes = static_cast<size_t>(kNoallocMaxItems) * sizeof(gva::WorkItem);
constexpr size_t kNoallocBlockBytes = static_cast<size_t>(kNoallocMaxBlocks) * sizeof(gva::KeyBlock);
// work list, key blocks, then the error word
constexpr size_t kNoallocScratchBytes = kNoallocItemBytes + kNoallocBlockBytes + 256;
constexpr int kMaxDevices = 64;

// The scratch: [work items | key blocks | error word]. Host code must not use this name as an
// address; it uses the pointer cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
gva::WorkItem g_staging[kNoallocMaxItems];       // host staging of the work list (under g_mutex)
gva::KeyBlock g_staging_blocks[kNoallocMaxBlocks];  // host staging of the key blocks (under g_mutex)

// Errors are reported through gva_last_error(), like every other entry point.
gva_status fail(gva_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  gva::set_last_error(buf);
  return s;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A map over a packed [rows, heads, d] tensor (bf16, or fp32 with `f32`) whose box is 128
// bytes of d by box_rows by box_heads, 128-byte swizzled.
bool encode(CUtensorMap* m, const void* base, int64_t rows, int32_t heads, int32_t d, uint32_t box_rows,
            uint32_t box_heads, bool f32 = false) {
  auto enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(heads) * d * es, static_cast<cuuint64_t>(d) * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), box_rows, box_heads};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace gva {

// The error word of the last gva_forward_noalloc launch on the current device (behind
// gva_device_status(NULL)): synchronise, read it, clear it. GVA_OK when no call has
// run on this device yet.
int noalloc_device_status() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GVA_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GVA_ERR_UNSUPPORTED, "device ordinal %d is out of range", dev);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    base = g_scratch_ptr[dev];
  }
  if (base == nullptr) {
    set_last_error("");
    return GVA_OK;
  }
  int* d_error = reinterpret_cast<int*>(static_cast<unsigned char*>(base) + kNoallocItemBytes + kNoallocBlockBytes);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess)
    return fail(GVA_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
  int word = 0;
  if ((e = cudaMemcpy(&word, d_error, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail(GVA_ERR_CUDA, "reading the no-alloc error word: %s", cudaGetErrorString(e));
  if (word != 0) {
    cudaMemset(d_error, 0, sizeof(int));
    return fail(GVA_ERR_DEVICE_CHECK,
                "a gva_forward_noalloc kernel recorded device error bits 0x%x (1 = bounded wait timed out)", word);
  }
  set_last_error("");
  return GVA_OK;
}

}  // namespace gva

extern "C" GVA_API gva_status gva_forward_noalloc(
    const int32_t* cu_seqlens_q, const int32_t* seqused_q, const int32_t* cu_seqlens_k, const int32_t* seqused_k,
    int32_t num_segments, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, const void* q, const void* k,
    const void* v, void* out, gva_dtype out_dtype, float* lse, float softmax_scale, cudaStream_t stream) {
  gva::set_last_error("");
  // ---- geometry checks (same rules as gva_plan)
  if (num_segments < 0) return fail(GVA_ERR_INVALID_ARG, "num_segments = %d < 0", num_segments);
  if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr ||
      (num_segments > 0 && (seqused_q == nullptr || seqused_k == nullptr)))
    return fail(GVA_ERR_INVALID_ARG, "a geometry array is NULL");
  if (num_heads_q <= 0 || num_heads_kv <= 0 || num_heads_q % num_heads_kv != 0)
    return fail(GVA_ERR_INVALID_ARG, "bad head counts (Hq=%d, Hkv=%d)", num_heads_q, num_heads_kv);
  const int32_t group = num_heads_q / num_heads_kv;
  if (group > gva::kTileRows)
    return fail(GVA_ERR_UNSUPPORTED, "query heads per KV head (%d) must be at most %d", group, gva::kTileRows);
  if (head_dim != 64 && head_dim != 128) return fail(GVA_ERR_UNSUPPORTED, "head_dim=%d is not supported", head_dim);
  if (out_dtype != GVA_BF16 && out_dtype != GVA_FP32) return fail(GVA_ERR_INVALID_ARG, "bad out_dtype");
  if (!std::isfinite(softmax_scale)) return fail(GVA_ERR_INVALID_ARG, "softmax_scale is not finite");
  const int32_t* cus[2] = {cu_seqlens_q, cu_seqlens_k};
  const int32_t* useds[2] = {seqused_q, seqused_k};
  for (int s = 0; s < 2; ++s) {
    if (cus[s][0] < 0) return fail(GVA_ERR_INVALID_ARG, "first segment offset is negative");
    for (int32_t b = 0; b < num_segments; ++b) {
      if (cus[s][b + 1] < cus[s][b]) return fail(GVA_ERR_INVALID_ARG, "segment offsets decrease at %d", b);
      if (useds[s][b] < 0 || useds[s][b] > cus[s][b + 1] - cus[s][b])
        return fail(GVA_ERR_INVALID_ARG, "used length of segment %d is outside its capacity", b);
    }
  }
  // ---- count the work items first, so an oversized launch is refused before any work
  const int32_t tpt = gva::kTileRows / group;
  const int32_t tpi = tpt * gva::kTilesPerItem;
  int64_t count = 0;
  for (int32_t b = 0; b < num_segments; ++b) count += static_cast<int64_t>((seqused_q[b] + tpi - 1) / tpi) * num_heads_kv;
  if (count > kNoallocMaxItems)
    return fail(GVA_ERR_INVALID_ARG,
                "this launch needs %lld work items; gva_forward_noalloc holds at most %d (use gva_plan + gva_forward)",
                static_cast<long long>(count), kNoallocMaxItems);
  int64_t nblocks = 0;
  for (int32_t b = 0; b < num_segments; ++b) nblocks += (seqused_k[b] + gva::kBlockKeys - 1) / gva::kBlockKeys;
  if (nblocks > kNoallocMaxBlocks)
    return fail(GVA_ERR_INVALID_ARG,
                "this launch needs %lld key blocks; gva_forward_noalloc holds at most %d (use gva_plan + gva_forward)",
                static_cast<long long>(nblocks), kNoallocMaxBlocks);
  if (count == 0) return GVA_OK;  // no used rows: nothing to write
  const int64_t total_q = cu_seqlens_q[num_segments];
  const int64_t total_k = cu_seqlens_k[num_segments];
  if (total_k == 0) k = v = q;  // no keys at all: K and V are never read
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr)
    return fail(GVA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(GVA_ERR_INVALID_ARG, "q, k, v, out and lse must be 16-byte aligned");

  // ---- device and its scratch address (resolved once per device)
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GVA_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GVA_ERR_UNSUPPORTED, "device ordinal %d is out of range", dev);
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(GVA_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device %d is sm_%d%d", dev, major,
                minor);

  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(GVA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = ptr;
  }
  unsigned char* scratch = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  gva::WorkItem* d_items = reinterpret_cast<gva::WorkItem*>(scratch);
  gva::KeyBlock* d_blocks = reinterpret_cast<gva::KeyBlock*>(scratch + kNoallocItemBytes);
  int* d_error = reinterpret_cast<int*>(scratch + kNoallocItemBytes + kNoallocBlockBytes);

  // ---- work list in the host staging array: most key blocks first (the persistent
  // kernel hands items out in this order)
  // key blocks of each segment's used prefix, then the segment's work items
  int32_t nb = 0, n = 0;
  for (int32_t b = 0; b < num_segments; ++b) {
    const int32_t blk0 = nb;
    for (int32_t o = 0; o < seqused_k[b]; o += gva::kBlockKeys)
      g_staging_blocks[nb++] = gva::KeyBlock{cu_seqlens_k[b] + o, std::min(gva::kBlockKeys, seqused_k[b] - o)};
    const int32_t uq = seqused_q[b];
    for (int32_t hk = 0; hk < num_heads_kv; ++hk) {
      for (int32_t t0 = 0; t0 < uq; t0 += tpi) {
        gva::WorkItem& it = g_staging[n++];
        it = gva::WorkItem{};
        it.q_row0 = cu_seqlens_q[b] + t0;
        it.q_rows = std::min(tpi, uq - t0);
        it.blk0 = blk0;
        it.nblk = nb - blk0;
        it.k_len = seqused_k[b];
        it.head_kv = hk;
        it.n_tiles = it.q_rows > tpt ? 2 : 1;
      }
    }
  }
  auto cost = [](const gva::WorkItem& it) {
    return static_cast<int64_t>(it.nblk) * it.n_tiles * 4 + it.n_tiles;
  };
  // In place (std::sort allocates nothing); ties are broken by position so the order is
  // deterministic. The order only affects scheduling: each output row is computed by
  // exactly one item, with the same arithmetic wherever it runs.
  std::sort(g_staging, g_staging + n, [&](const gva::WorkItem& a, const gva::WorkItem& c) {
    const int64_t ca = cost(a), cc = cost(c);
    if (ca != cc) return ca > cc;
    if (a.q_row0 != c.q_row0) return a.q_row0 < c.q_row0;
    return a.head_kv < c.head_kv;
  });

  // Pageable-to-device copy: the staging array is free again once the call returns.
  e = cudaMemcpyAsync(d_items, g_staging, static_cast<size_t>(n) * sizeof(gva::WorkItem), cudaMemcpyHostToDevice,
                      stream);
  if (e != cudaSuccess) return fail(GVA_ERR_CUDA, "copying the work list: %s", cudaGetErrorString(e));
  if (nb > 0) {
    e = cudaMemcpyAsync(d_blocks, g_staging_blocks, static_cast<size_t>(nb) * sizeof(gva::KeyBlock),
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return fail(GVA_ERR_CUDA, "copying the key blocks: %s", cudaGetErrorString(e));
  }
  e = cudaMemsetAsync(d_error, 0, sizeof(int), stream);
  if (e != cudaSuccess) return fail(GVA_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));

  // the maps are host structures passed with the launch: nothing is allocated for them
  CUtensorMap mq, mk, mv, mo;
  const int64_t krows = total_k > 0 ? total_k : 1;
  if (!encode(&mq, q, total_q, num_heads_q, head_dim, tpt, group) ||
      !encode(&mk, k, krows, num_heads_kv, head_dim, gva::kBlockKeys, 1) ||
      !encode(&mv, v, krows, num_heads_kv, head_dim, gva::kBlockKeys, 1) ||
      !encode(&mo, out, total_q, num_heads_q, head_dim, tpt, group, out_dtype == GVA_FP32))
    return fail(GVA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  gva::FwdParams prm{};
  prm.items = d_items;
  prm.blocks = d_blocks;
  prm.num_items = n;
  prm.out = out;
  prm.out_wide = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  prm.out_tma = 1;
  prm.lse = lse;
  prm.total_q = total_q;
  prm.num_heads_q = num_heads_q;
  prm.group = group;
  prm.tokens_per_tile = tpt;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.error_flag = d_error;
  e = gva::launch_forward(head_dim, out_dtype == GVA_FP32, prm, mq, mk, mv, mo, std::min(n, sms), stream);
  if (e != cudaSuccess) return fail(GVA_ERR_CUDA, "launching the forward kernel: %s", cudaGetErrorString(e));
  return GVA_OK;
}
