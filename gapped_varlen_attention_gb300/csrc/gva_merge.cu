// FP32 log-sum-exp merge of partial attention results over disjoint key sets
// (cosmos-framework PR #312, "Problem and behavior": visibility partitions are
// combined by an FP32 LSE merge).
//
// For a used row r and head h:  L = max_p lse_p;  L = -inf -> O = 0, lse = -inf;
// otherwise w_p = exp(lse_p - L), lse = L + ln(sum w_p), O = sum_p w_p O_p / sum_p w_p.
//
// The merge streams every partial output once and is HBM-bound. A CTA takes a unit of
// up to 16 consecutive used rows of one segment: it first turns the partitions' LSEs of
// those rows (coalesced along rows) into normalised weights in shared memory, then
// streams the unit's contiguous [rows, Hq, d] block of every partition through a ring
// of shared-memory chunks filled by bulk asynchronous copies (cp.async.bulk, completing
// on one mbarrier per chunk slot): one thread keeps several chunks of every partition in
// flight while all threads combine the chunk that has landed and store the result with
// 16- or 32-byte vector stores. A partition with no weight anywhere in the unit (no keys
// for those rows) is not copied, and a zero weight never reads its partial, so values
// there cannot leak. Gap rows are never read or written. The output may alias the
// first partition: every element is copied in before it is overwritten.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdint>

#include "gva_device_common.cuh"
#include "gva_internal.h"
#include "sm103_ptx.cuh"

namespace gva {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;                        // elements per thread per chunk
constexpr int kChunkElems = kThreads * kVec;   // elements of one partition per chunk

// One bulk copy global -> shared memory completing `bytes` on `bar` (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load_smem(const void* ptr, float (&x)[8]) {
    const uint4 u = *static_cast<const uint4*>(ptr);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void store(void* ptr, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(x[2 * i + 1]), "f"(x[2 * i]));
    }
    *static_cast<uint4*>(ptr) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load_smem(const void* ptr, float (&x)[8]) {
    const float4 a = static_cast<const float4*>(ptr)[0], b = static_cast<const float4*>(ptr)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store(void* ptr, const float (&x)[8]) {
    float4* d = static_cast<float4*>(ptr);
    d[0] = make_float4(x[0], x[1], x[2], x[3]);
    d[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

// Shared memory: [ring_slots chunks][num_parts x Hq x kMergeRows weights][ring_slots
// mbarriers][live flags][abort flag]. Chunk slot g * num_parts + q holds partition q of
// the g-th chunk in flight; the CTA's chunks are numbered across its units (seq), so the
// slot group of chunk s is s % depth and the phase it completes is (s / depth) & 1.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) gva_lse_merge_kernel(const MergeParams p, const int ring_slots) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr uint32_t kChunkBytes = kChunkElems * sizeof(TIn);
  const int parts = p.num_parts;
  const int hq = p.num_heads_q;
  const int slots = hq * kMergeRows;
  unsigned char* ring = smem;
  float* w_smem = reinterpret_cast<float*>(smem + static_cast<size_t>(ring_slots) * kChunkBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(w_smem + parts * slots);  // parts * slots is a multiple of 16
  int* live = reinterpret_cast<int*>(full + ring_slots);
  int* abort_flag = live + kMaxMergeParts;
  const int depth = ring_slots / parts;  // chunks in flight (>= 1, checked on the host)
  if (threadIdx.x == 0) {
    for (int i = 0; i < ring_slots; ++i) mbar_init(&full[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Hq * d * kMergeRows < 2^31: the unit's element offsets fit 32 bits
  const uint32_t row_elems = static_cast<uint32_t>(hq) * p.head_dim;
  const int dshift = p.head_dim == 128 ? 7 : 6;
  uint32_t seq = 0;
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const MergeUnit mu = p.units[u];
    if (threadIdx.x < kMaxMergeParts) live[threadIdx.x] = 0;
    __syncthreads();  // also: the previous unit's chunks and weights are no longer read
    for (int i = threadIdx.x; i < slots; i += kThreads) {
      const int h = i / kMergeRows;
      const int r = i - h * kMergeRows;
      if (r >= mu.rows) continue;
      const int64_t li = static_cast<int64_t>(h) * p.total_q + mu.row0 + r;
      float lv[kMaxMergeParts];
      float big = -CUDART_INF_F;
      for (int q = 0; q < parts; ++q) {
        lv[q] = p.lses[q][li];
        big = fmaxf(big, lv[q]);
      }
      float merged;
      if (big == -CUDART_INF_F) {
        for (int q = 0; q < parts; ++q) w_smem[q * slots + i] = 0.0f;
        merged = -CUDART_INF_F;
      } else {
        float tot = 0.0f;
        for (int q = 0; q < parts; ++q) {
          lv[q] = (lv[q] == -CUDART_INF_F) ? 0.0f : expf(lv[q] - big);
          tot += lv[q];
        }
        const float inv = 1.0f / tot;
        for (int q = 0; q < parts; ++q) {
          const float w = lv[q] * inv;
          w_smem[q * slots + i] = w;
          if (w != 0.0f) live[q] = 1;
        }
        merged = big + logf(tot);
      }
      p.lse[li] = merged;
    }
    __syncthreads();
    const size_t base = static_cast<size_t>(mu.row0) * row_elems;
    const uint32_t n = static_cast<uint32_t>(mu.rows) * row_elems;
    const int nchunks = static_cast<int>((n + kChunkElems - 1) / kChunkElems);
    auto issue = [&](int c) {  // one thread: the copies of chunk c of every partition
      const int g = static_cast<int>((seq + c) % depth);
      const uint32_t e0 = static_cast<uint32_t>(c) * kChunkElems;
      const uint32_t bytes = min(static_cast<uint32_t>(kChunkElems), n - e0) * sizeof(TIn);
      for (int q = 0; q < parts; ++q) {
        uint64_t* bar = &full[g * parts + q];
        if (live[q]) {
          mbar_arrive_expect_tx(bar, bytes);
          bulk_load(ring + static_cast<size_t>(g * parts + q) * kChunkBytes,
                    static_cast<const TIn*>(p.outs[q]) + base + e0, bytes, bar);
        } else {
          mbar_arrive(bar);  // nothing to copy: the slot's phase completes at once
        }
      }
    };
    if (threadIdx.x == 0)
      for (int c = 0; c < min(depth, nchunks); ++c) issue(c);
    int c = 0;
    for (; c < nchunks; ++c) {
      const uint32_t s = seq + c;
      const int g = static_cast<int>(s % depth);
      const uint32_t parity = (s / depth) & 1u;
      bool ok = true;
      for (int q = 0; q < parts && ok; ++q) ok = wait_bar(&full[g * parts + q], parity, abort_flag, p.error_flag);
      const uint32_t e = static_cast<uint32_t>(c) * kChunkElems + threadIdx.x * kVec;
      if (ok && e < n) {
        const uint32_t r = e / row_elems;
        const uint32_t h = (e - r * row_elems) >> dshift;
        const int slot = static_cast<int>(h) * kMergeRows + static_cast<int>(r);
        float acc[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
        for (int q = 0; q < parts; ++q) {
          const float w = w_smem[q * slots + slot];
          if (w != 0.0f) {
            float x[kVec];
            Vec8<TIn>::load_smem(ring + static_cast<size_t>(g * parts + q) * kChunkBytes + threadIdx.x * kVec * sizeof(TIn), x);
#pragma unroll
            for (int i = 0; i < kVec; ++i) acc[i] = fmaf(w, x[i], acc[i]);
          }
        }
        Vec8<TOut>::store(static_cast<TOut*>(p.out) + base + e, acc);
      }
      if (__syncthreads_or(!ok)) break;  // every thread leaves together
      if (threadIdx.x == 0 && c + depth < nchunks) issue(c + depth);
    }
    if (c < nchunks) {
      // a wait gave up: let the copies already issued (chunks c .. c + depth - 1) land
      // before the CTA's shared memory is released
      if (threadIdx.x == 0) {
        for (int c2 = c; c2 < min(c + depth, nchunks); ++c2) {
          const uint32_t s = seq + c2;
          for (int q = 0; q < parts; ++q)
            drain_bar(&full[static_cast<int>(s % depth) * parts + q], (s / depth) & 1u, p.error_flag);
        }
      }
      return;
    }
    seq += static_cast<uint32_t>(nchunks);
  }
}

// Chunk ring per CTA. Measured on the text + video merge (2 FP32 partitions of Hq = 24,
// d = 128; 519 units): 32 or 48 KB rings (four or more CTAs per SM, two or three chunks
// of both partitions in flight each) took 43 us, as long as a device copy of the same
// bytes; 64 and 96 KB rings took 59-63 us and 192 KB 102 us (fewer CTAs per SM, and
// the units no longer fit one wave).
constexpr int kRingBytes = 48 * 1024;
constexpr int kMergeSmemCap = 227 * 1024;   // opt-in shared memory per CTA
constexpr int kSmemPerSm = 228 * 1024;      // shared memory per SM, 1 KB of it reserved per CTA

template <typename TIn, typename TOut>
cudaError_t launch_merge_impl(const MergeParams& p, int sm_count, cudaStream_t stream) {
  int ring_slots = 0;
  const int smem = merge_smem_bytes(sizeof(TIn) == 4, p.num_parts, p.num_heads_q, &ring_slots);
  if (smem <= 0) return cudaErrorInvalidValue;  // refused on the host before the launch
  cudaError_t e = ensure_smem_limit<gva_lse_merge_kernel<TIn, TOut>>(kMergeSmemCap);
  if (e != cudaSuccess) return e;
  const int per_sm = std::max(1, std::min(2048 / kThreads, kSmemPerSm / (smem + 1024)));
  const int grid = std::min(p.num_units, per_sm * sm_count);
  gva_lse_merge_kernel<TIn, TOut><<<grid, kThreads, smem, stream>>>(p, ring_slots);
  return cudaGetLastError();
}

}  // namespace

int merge_smem_bytes(bool in_f32, int num_parts, int num_heads_q, int* ring_slots) {
  const int chunk = kChunkElems * (in_f32 ? 4 : 2);
  const int fixed = num_parts * num_heads_q * kMergeRows * 4 + (kMaxMergeParts + 1) * 4;
  // slots: a whole number of chunk groups (one chunk of every partition), as many as
  // the ring budget holds but at least one, within the shared-memory cap
  const int cap_groups = (kMergeSmemCap - fixed) / ((chunk + 8) * num_parts);
  const int groups = std::min(std::max(kRingBytes / (chunk * num_parts), 1), cap_groups);
  if (groups < 1) return -1;
  const int slots = groups * num_parts;
  *ring_slots = slots;
  return slots * (chunk + 8) + fixed;
}

cudaError_t launch_merge(bool in_f32, bool out_f32, const MergeParams& p, int sm_count, cudaStream_t stream) {
  if (in_f32) {
    return out_f32 ? launch_merge_impl<float, float>(p, sm_count, stream)
                   : launch_merge_impl<float, __nv_bfloat16>(p, sm_count, stream);
  }
  return out_f32 ? launch_merge_impl<__nv_bfloat16, float>(p, sm_count, stream)
                 : launch_merge_impl<__nv_bfloat16, __nv_bfloat16>(p, sm_count, stream);
}

}  // namespace gva
