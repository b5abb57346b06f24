// Device helpers shared by the forward and backward kernels: bounded mbarrier waits,
// work-list loads and row stores.
#pragma once

#include <cuda_bf16.h>

#include "gva_internal.h"
#include "sm103_ptx.cuh"

namespace gva {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

// Wait for the phase of `bar` with parity `parity` to complete. Gives up (returning
// false) when another role has aborted or after kWaitLimitNs, recording the timeout.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}

// Same, ignoring the abort flag: used to drain copies and MMAs already in flight.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, int* err) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrWaitTimeout);
      return;
    }
  }
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ WorkItem load_item(const WorkItem* items, int idx) {
  const int4* p = reinterpret_cast<const int4*>(items + idx);
  const int4 a = __ldg(p), b = __ldg(p + 1);
  WorkItem it;
  it.q_row0 = a.x; it.q_rows = a.y; it.blk0 = a.z; it.nblk = a.w;
  it.head_kv = b.x; it.n_tiles = b.y; it.k_len = b.z; it.q_pos0 = b.w;
  return it;
}

__device__ __forceinline__ KeyBlock load_block(const KeyBlock* blocks, int idx) {
  const int2 v = __ldg(reinterpret_cast<const int2*>(blocks) + idx);
  return KeyBlock{v.x, v.y};
}

template <typename TOut>
__device__ __forceinline__ void store_row32(TOut* dst, const float (&x)[32]);

template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* dst, const float (&x)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d[i] = make_uint4(pack_bf16x2(x[8 * i + 0], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                      pack_bf16x2(x[8 * i + 4], x[8 * i + 5]), pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
  }
}

template <>
__device__ __forceinline__ void store_row32<float>(float* dst, const float (&x)[32]) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) d[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
}

// The same rows with 32-byte stores (st.global.v8.b32, sm_100 and later): half the
// store instructions. A warp's 32 rows are 32 different rows of the output, so every
// store instruction touches 32 lines and the epilogue is bound by the number of store
// instructions. `dst` must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

template <typename TOut>
__device__ __forceinline__ void store_row32_wide(TOut* dst, const float (&x)[32]);

template <>
__device__ __forceinline__ void store_row32_wide<__nv_bfloat16>(__nv_bfloat16* dst, const float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float* y = x + 16 * i;
    st_global_v8(dst + 16 * i, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                 pack_bf16x2(y[6], y[7]), pack_bf16x2(y[8], y[9]), pack_bf16x2(y[10], y[11]),
                 pack_bf16x2(y[12], y[13]), pack_bf16x2(y[14], y[15]));
  }
}

template <>
__device__ __forceinline__ void store_row32_wide<float>(float* dst, const float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float* y = x + 8 * i;
    st_global_v8(dst + 8 * i, __float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]),
                 __float_as_uint(y[3]), __float_as_uint(y[4]), __float_as_uint(y[5]), __float_as_uint(y[6]),
                 __float_as_uint(y[7]));
  }
}

// MMA issue. One thread issues every tcgen05.mma, so the issue path must be short:
// the shared-memory descriptors are built once per operand buffer, and each K step only
// adds its byte offset (in 16-byte units) to the start-address field (bits 0-13; every
// address here is below 256 KB, so the field never carries). Building a 64-bit
// descriptor per MMA instead costs more issue time than a 128x128x16 MMA executes.
// Operand tiles are 128 rows of 128-byte swizzled rows per 64-column chunk.
constexpr uint32_t kChunkBytes = 128 * 128;
static_assert(kTileRows == 128 && kBlockKeys == 128, "tiles of 128 rows");

// D[128 x 128] = A[128 x D] B[128 x D]^T with both operands K-major in shared memory
// (S = Q K^T in the forward; S, dP, S^T and dP^T in the backward).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = make_idesc_bf16(kTileRows, kBlockKeys, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4;
    umma_bf16_ss(tmem_s, q_desc + off, k_desc + off, idesc, kk > 0);
  }
}

// D[128 x D] (+)= A[128 x 128] B[128 x D] with A (bf16 pairs) in TMEM and B MN-major in
// shared memory (O += P V in the forward; dQ += dS K, dV += P^T dO, dK += dS^T Q).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, uint32_t accumulate) {
  constexpr uint32_t idesc = make_idesc_bf16(kTileRows, D, true);
  umma_bf16_ts(tmem_o, tmem_p, v_desc, idesc, accumulate);
#pragma unroll
  for (int kk = 1; kk < kBlockKeys / 16; ++kk)
    umma_bf16_ts(tmem_o, tmem_p + kk * 8, v_desc + ((kk * 16 * 128) >> 4), idesc, 1u);
}

}  // namespace gva
