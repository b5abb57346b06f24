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
// streams the unit's contiguous [rows, Hq, d] block of every partition with 16- or
// 32-byte vector loads. Gap rows are never read or written. Plain (coherent) loads are
// used because the output may alias the first partition.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "gva_internal.h"

namespace gva {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;  // elements per vector access (Hq * d is a multiple of 8)

template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const void* base, int64_t e, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + e);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void store(void* base, int64_t e, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(x[2 * i + 1]), "f"(x[2 * i]));
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + e) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const void* base, int64_t e, float (&x)[8]) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store(void* base, int64_t e, const float (&x)[8]) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + e);
    p[0] = make_float4(x[0], x[1], x[2], x[3]);
    p[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) gva_lse_merge_kernel(const MergeParams p) {
  extern __shared__ float w_smem[];  // [num_parts][Hq][kMergeRows] normalised weights
  const int hq = p.num_heads_q;
  const int slots = hq * kMergeRows;
  const int64_t row_elems = static_cast<int64_t>(hq) * p.head_dim;
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const MergeUnit mu = p.units[u];
    for (int i = threadIdx.x; i < slots; i += kThreads) {
      const int h = i / kMergeRows;
      const int r = i - h * kMergeRows;
      if (r >= mu.rows) continue;
      const int64_t li = static_cast<int64_t>(h) * p.total_q + mu.row0 + r;
      float lv[kMaxMergeParts];
      float big = -CUDART_INF_F;
      for (int q = 0; q < p.num_parts; ++q) {
        lv[q] = p.lses[q][li];
        big = fmaxf(big, lv[q]);
      }
      float merged;
      if (big == -CUDART_INF_F) {
        for (int q = 0; q < p.num_parts; ++q) w_smem[q * slots + i] = 0.0f;
        merged = -CUDART_INF_F;
      } else {
        float tot = 0.0f;
        for (int q = 0; q < p.num_parts; ++q) {
          lv[q] = (lv[q] == -CUDART_INF_F) ? 0.0f : expf(lv[q] - big);
          tot += lv[q];
        }
        const float inv = 1.0f / tot;
        for (int q = 0; q < p.num_parts; ++q) w_smem[q * slots + i] = lv[q] * inv;
        merged = big + logf(tot);
      }
      p.lse[li] = merged;
    }
    __syncthreads();
    const int64_t base = static_cast<int64_t>(mu.row0) * row_elems;
    const int64_t n = static_cast<int64_t>(mu.rows) * row_elems;
    for (int64_t e = static_cast<int64_t>(threadIdx.x) * kVec; e < n; e += kThreads * kVec) {
      const int r = static_cast<int>(e / row_elems);
      const int h = static_cast<int>((e - r * row_elems) / p.head_dim);
      const int slot = h * kMergeRows + r;
      float acc[kVec];
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
      for (int q = 0; q < p.num_parts; ++q) {
        const float w = w_smem[q * slots + slot];
        if (w != 0.0f) {  // a partition without keys for this row is not read
          float x[kVec];
          Vec8<TIn>::load(p.outs[q], base + e, x);
#pragma unroll
          for (int i = 0; i < kVec; ++i) acc[i] = fmaf(w, x[i], acc[i]);
        }
      }
      Vec8<TOut>::store(p.out, base + e, acc);
    }
    __syncthreads();
  }
}

template <typename TIn, typename TOut>
cudaError_t launch_merge_impl(const MergeParams& p, int grid, cudaStream_t stream) {
  const int smem = p.num_parts * p.num_heads_q * kMergeRows * static_cast<int>(sizeof(float));
  auto kern = gva_lse_merge_kernel<TIn, TOut>;
  // the plan validation caps the weights at 200 KB; raise the limit to that once
  cudaError_t e = ensure_smem_limit<gva_lse_merge_kernel<TIn, TOut>>(200 * 1024);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(bool in_f32, bool out_f32, const MergeParams& p, int grid, cudaStream_t stream) {
  if (in_f32) {
    return out_f32 ? launch_merge_impl<float, float>(p, grid, stream)
                   : launch_merge_impl<float, __nv_bfloat16>(p, grid, stream);
  }
  return out_f32 ? launch_merge_impl<__nv_bfloat16, float>(p, grid, stream)
                 : launch_merge_impl<__nv_bfloat16, __nv_bfloat16>(p, grid, stream);
}

}  // namespace gva
