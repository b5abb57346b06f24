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
// 32-byte vector loads: each thread has two vectors of two partitions in flight before
// it accumulates, since the kernel is latency-bound at one load at a time. Gap rows are
// never read or written. Plain (coherent) loads are used because the output may alias
// the first partition.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdint>

#include "gva_internal.h"

namespace gva {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;  // elements per vector access (Hq * d is a multiple of 8)

// Loads of 8 elements that happen only when `live` (a partition with zero weight for the
// row is not read): predicated in PTX rather than branched around, so that the loads of
// every partition and unrolled vector are in flight together.
template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const void* base, uint32_t e, bool live, float (&x)[8]) {
    uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    const __nv_bfloat16* ptr = static_cast<const __nv_bfloat16*>(base) + e;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "@p ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%5];\n\t}"
        : "+r"(w0), "+r"(w1), "+r"(w2), "+r"(w3)
        : "r"(static_cast<uint32_t>(live)), "l"(ptr));
    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void store(void* base, uint32_t e, const float (&x)[8]) {
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
  static __device__ __forceinline__ void load(const void* base, uint32_t e, bool live, float (&x)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    const float* ptr = static_cast<const float*>(base) + e;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %8, 0;\n\t"
        "@p ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%9];\n\t"
        "@p ld.global.L1::no_allocate.v4.f32 {%4, %5, %6, %7}, [%9+16];\n\t}"
        : "+f"(x[0]), "+f"(x[1]), "+f"(x[2]), "+f"(x[3]), "+f"(x[4]), "+f"(x[5]), "+f"(x[6]), "+f"(x[7])
        : "r"(static_cast<uint32_t>(live)), "l"(ptr));
  }
  static __device__ __forceinline__ void store(void* base, uint32_t e, const float (&x)[8]) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + e);
    p[0] = make_float4(x[0], x[1], x[2], x[3]);
    p[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
};

// Measured on the text + video merge (2 FP32 partitions, 519 units): one vector per
// thread with both partitions' loads in flight ran at 52 us; two or four vectors per
// thread, or two or four CTAs sharing a unit, ran at 54-64 us.
constexpr int kUnroll = 1;     // vectors per thread per round
constexpr int kPartStep = 2;   // partitions loaded per round before their FMAs

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kThreads) gva_lse_merge_kernel(const MergeParams p) {
  extern __shared__ float w_smem[];  // [num_parts][Hq][kMergeRows] normalised weights
  const int hq = p.num_heads_q;
  const int slots = hq * kMergeRows;
  // Hq * d * kMergeRows < 2^31: the unit's element offsets fit 32 bits
  const uint32_t row_elems = static_cast<uint32_t>(hq) * p.head_dim;
  const int dshift = p.head_dim == 128 ? 7 : 6;
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
    // the unit's rows are one contiguous [rows, Hq, d] block in every tensor
    const size_t base = static_cast<size_t>(mu.row0) * row_elems;
    const uint32_t n = static_cast<uint32_t>(mu.rows) * row_elems;
    for (uint32_t e0 = threadIdx.x * kVec; e0 < n; e0 += kThreads * kVec * kUnroll) {
      uint32_t e[kUnroll];
      int slot[kUnroll];
      bool in[kUnroll];
      float acc[kUnroll][kVec];
#pragma unroll
      for (int v = 0; v < kUnroll; ++v) {
        e[v] = e0 + v * kThreads * kVec;
        in[v] = e[v] < n;
        const uint32_t r = in[v] ? e[v] / row_elems : 0;
        const uint32_t h = (e[v] - r * row_elems) >> dshift;
        slot[v] = static_cast<int>(h) * kMergeRows + static_cast<int>(r);
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[v][i] = 0.0f;
      }
      for (int q0 = 0; q0 < p.num_parts; q0 += kPartStep) {
        float x[kPartStep][kUnroll][kVec];
        float w[kPartStep][kUnroll];
#pragma unroll
        for (int j = 0; j < kPartStep; ++j) {
          const int q = q0 + j;
#pragma unroll
          for (int v = 0; v < kUnroll; ++v) {
            w[j][v] = (q < p.num_parts && in[v]) ? w_smem[q * slots + slot[v]] : 0.0f;
          }
        }
#pragma unroll
        for (int j = 0; j < kPartStep; ++j) {
          const int q = q0 + j < p.num_parts ? q0 + j : 0;
          const char* part = static_cast<const char*>(p.outs[q]) + base * sizeof(TIn);
#pragma unroll
          for (int v = 0; v < kUnroll; ++v) Vec8<TIn>::load(part, e[v], w[j][v] != 0.0f, x[j][v]);
        }
#pragma unroll
        for (int j = 0; j < kPartStep; ++j)
#pragma unroll
          for (int v = 0; v < kUnroll; ++v)
#pragma unroll
            for (int i = 0; i < kVec; ++i) acc[v][i] = fmaf(w[j][v], x[j][v][i], acc[v][i]);
      }
      char* outp = static_cast<char*>(p.out) + base * sizeof(TOut);
#pragma unroll
      for (int v = 0; v < kUnroll; ++v)
        if (in[v]) Vec8<TOut>::store(outp, e[v], acc[v]);
    }
    __syncthreads();
  }
}

template <typename TIn, typename TOut>
cudaError_t launch_merge_impl(const MergeParams& p, int max_grid, cudaStream_t stream) {
  const int smem = p.num_parts * p.num_heads_q * kMergeRows * static_cast<int>(sizeof(float));
  auto kern = gva_lse_merge_kernel<TIn, TOut>;
  // the plan validation caps the weights at 200 KB; raise the limit to that once
  cudaError_t e = ensure_smem_limit<gva_lse_merge_kernel<TIn, TOut>>(200 * 1024);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.num_units, max_grid);
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(bool in_f32, bool out_f32, const MergeParams& p, int max_grid, cudaStream_t stream) {
  if (in_f32) {
    return out_f32 ? launch_merge_impl<float, float>(p, max_grid, stream)
                   : launch_merge_impl<float, __nv_bfloat16>(p, max_grid, stream);
  }
  return out_f32 ? launch_merge_impl<__nv_bfloat16, float>(p, max_grid, stream)
                 : launch_merge_impl<__nv_bfloat16, __nv_bfloat16>(p, max_grid, stream);
}

}  // namespace gva
