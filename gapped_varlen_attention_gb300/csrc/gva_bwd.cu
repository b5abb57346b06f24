// Backward of the gapped variable-length attention forward, sm_103a.
//
// The pages mark the backward as missing on the non-FA4 paths (cosmos-framework PR #302
// review: the torch fallback is forward only; PR #312 "Problem and behavior": SM120
// backward raises). From the forward's definition, for each used row i of a segment,
// query head h and used key j, with P the softmax recomputed from the saved LSE:
//
//   dP_ij = <dO_i, V_j>,  D_i = <dO_i, O_i> (= sum_j P_ij dP_ij),  dS_ij = P_ij (dP_ij - D_i)
//   dQ_i = s sum_j dS_ij K_j,  dK_j = s sum_i dS_ij Q_i,  dV_j = sum_i P_ij dO_i
//
// (the dK / dV sums run over the g query heads of the KV group as well). Three launches:
//   1. gva_bwd_dvec_kernel: D = rowsum(dO * O) for every used row and head.
//   2. gva_bwd_dq_kernel: one 128-row Q tile (folded GQA rows, as in the forward) per
//      work item, streaming the segment's key blocks: S = Q K^T and dP = dO V^T into
//      TMEM, P and dS by one thread per row, dQ += dS K with dS read from TMEM.
//   3. gva_bwd_dkdv_kernel: one key block of one KV head per unit, streaming the
//      segment's Q / dO tiles: S^T = K Q^T and dP^T = V dO^T into TMEM, P^T and dS^T by
//      one thread per key, dV += P^T dO and dK += dS^T Q accumulated in TMEM, then
//      written once. No atomics anywhere.
// Operand rows past the used lengths (gaps, padding, possibly NaN) are zeroed in shared
// memory before an MMA could multiply them by a zero weight.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "gva_device_common.cuh"
#include "gva_internal.h"
#include "sm103_ptx.cuh"

namespace gva {
namespace {

constexpr int kBwdThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 compute
constexpr uint32_t kBwdTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTileRows * D * 2;  // a Q, dO, K or V tile of 128 rows
  static constexpr int kSlots = 4;                      // dQ kernel K/V ring
  static constexpr int kSmemDq = 2 * kTileBytes + kSlots * kTileBytes + 1024;
  static constexpr int kSmemDkv = 2 * kTileBytes + 2 * 2 * kTileBytes + 1024;
  static_assert(kSmemDq <= 227 * 1024 && kSmemDkv <= 227 * 1024, "shared memory budget");
};

// Zero the 128-byte rows `rows` of a 128-row tile (all column chunks); the swizzle only
// permutes 16-byte pieces within a row, so whole rows are cleared position-free.
template <int D>
__device__ __forceinline__ void zero_tile_row(uint8_t* tile, int row) {
#pragma unroll
  for (int ch = 0; ch < D / 64; ++ch) {
    uint4* r = reinterpret_cast<uint4*>(tile + ch * kChunkBytes + row * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ KvUnit load_unit(const KvUnit* units, int idx) {
  const int4* p = reinterpret_cast<const int4*>(units + idx);
  const int4 a = __ldg(p);
  KvUnit u;
  u.key_row0 = a.x; u.keys = a.y; u.q_row0 = a.z; u.q_used = a.w;
  u.head_kv = __ldg(reinterpret_cast<const int*>(p + 1));
  u.pad0 = u.pad1 = u.pad2 = 0;
  return u;
}

struct BwdCtrl {
  float xl[2][kTileRows];  // dK / dV kernel: per-column log2-LSE of the current Q tile
  float xd[2][kTileRows];  //                 per-column D
  uint64_t a_full, a_empty;            // dQ: Q + dO tiles;   dK/dV: K + V blocks
  uint64_t r_full[4], r_empty[4];      // dQ: K/V ring;       dK/dV: Q/dO slots (2)
  uint64_t zero_bar;                   // partial tiles: the producer's own copy wait
  uint64_t s_full, p_full, acc_full, mma_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void init_ctrl(BwdCtrl& c, int ring) {
  mbar_init(&c.a_full, 1);
  mbar_init(&c.a_empty, 1);
  for (int i = 0; i < ring; ++i) {
    mbar_init(&c.r_full[i], 1);
    mbar_init(&c.r_empty[i], 1);
  }
  mbar_init(&c.zero_bar, 1);
  mbar_init(&c.s_full, 1);
  mbar_init(&c.p_full, 128);
  mbar_init(&c.acc_full, 1);
  mbar_init(&c.mma_done, 1);
  c.abort = 0;
  fence_barrier_init();
}

// ---------------------------------------------------------------------------------
// 1. D = rowsum(dO * O)
// ---------------------------------------------------------------------------------
// Eight threads per (row, head) pair; each reads 16 bf16 of dO and O per pass.
template <int D>
__global__ void __launch_bounds__(256) gva_bwd_dvec_kernel(const MergeUnit* units, int32_t num_units,
                                                           const __nv_bfloat16* out, const __nv_bfloat16* d_out,
                                                           float* dvec, int64_t total_q, int32_t hq) {
  const int sub = threadIdx.x & 7;
  const int warp_pair0 = (threadIdx.x >> 5) * 4;  // 4 pairs per warp, 32 per block pass
  const int pair_in_warp = (threadIdx.x >> 3) & 3;
  for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
    const MergeUnit mu = units[u];
    const int pairs = mu.rows * hq;
    for (int base = warp_pair0; base < pairs; base += 32) {  // uniform over the warp
      const int pr = base + pair_in_warp;
      const bool live = pr < pairs;
      const int r = pr / hq, h = pr - r * hq;
      const int64_t row = mu.row0 + r;
      float acc = 0.0f;
      if (live) {
        const __nv_bfloat16* a = out + (row * hq + h) * D;
        const __nv_bfloat16* b = d_out + (row * hq + h) * D;
#pragma unroll
        for (int e = sub * 8; e < D; e += 64) {
          const uint4 x = *reinterpret_cast<const uint4*>(a + e);
          const uint4 y = *reinterpret_cast<const uint4*>(b + e);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc = fmaf(__uint_as_float(xs[i] << 16), __uint_as_float(ys[i] << 16), acc);
            acc = fmaf(__uint_as_float(xs[i] & 0xFFFF0000u), __uint_as_float(ys[i] & 0xFFFF0000u), acc);
          }
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      if (live && sub == 0) dvec[static_cast<int64_t>(h) * total_q + row] = acc;
    }
  }
}

// ---------------------------------------------------------------------------------
// 2. dQ
// ---------------------------------------------------------------------------------
template <int D, typename TOut>
__global__ void __launch_bounds__(kBwdThreads, 1)
    gva_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                      const BwdParams p) {
  using C = BCfg<D>;
  constexpr uint32_t NS = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtrl ctrl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = sQ + C::kTileBytes;
  uint8_t* sKV = sDO + C::kTileBytes;  // NS slots: K_0, V_0, K_1, V_1, ...
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctrl.abort;
  if (threadIdx.x == 0) init_ctrl(ctrl, NS);
  if (warp == 1) {
    tmem_alloc(&ctrl.tmem_base, kBwdTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  const int T = p.tokens_per_tile;
  const int G = p.group;
  // TMEM: S [0,128) (dS as bf16 pairs overwrites [0,64)), dP [128,256), dQ [256,256+D)
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

  if (warp == 0) {
    // The whole warp walks the work list; lane 0 issues the copies, and all lanes
    // clear the rows of partial K/V blocks past the used keys (they would meet P = 0 or
    // dS = 0 in an MMA, and 0 * NaN is NaN) before the slot is marked full.
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_do);
    }
    uint32_t q_it = 0, ld = 0, zph = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_items) break;
      const WorkItem it = load_item(p.items, idx);
      if (it.nblk == 0) continue;
      if (leader) ok = wait_bar(&ctrl.a_empty, (q_it & 1) ^ 1, abort_flag, p.error_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (leader) {
        mbar_arrive_expect_tx(&ctrl.a_full, 2 * C::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < C::kChunks; ++ch) {
          tma_load_3d(sQ + ch * kChunkBytes, &map_q, &ctrl.a_full, ch * 64, it.q_row0, it.head_kv * G);
          tma_load_3d(sDO + ch * kChunkBytes, &map_do, &ctrl.a_full, ch * 64, it.q_row0, it.head_kv * G);
        }
      }
      ++q_it;
      for (int j = 0; j < it.nblk && ok; ++j) {
        const KeyBlock blk = load_block(p.blocks, it.blk0 + j);
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t sl = ld % NS;
          if (leader) ok = wait_bar(&ctrl.r_empty[sl], ((ld / NS) & 1) ^ 1, abort_flag, p.error_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          uint8_t* dst = sKV + sl * C::kTileBytes;
          const CUtensorMap* map = kv == 0 ? &map_k : &map_v;
          uint64_t* bar = blk.valid == kBlockKeys ? &ctrl.r_full[sl] : &ctrl.zero_bar;
          if (leader) {
            mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_3d(dst + ch * kChunkBytes, map, bar, ch * 64, blk.row0, it.head_kv);
          }
          if (blk.valid < kBlockKeys) {
            ok = __all_sync(0xffffffffu, wait_bar(&ctrl.zero_bar, zph & 1, abort_flag, p.error_flag));
            if (!ok && leader) drain_bar(&ctrl.zero_bar, zph & 1, p.error_flag);
            ++zph;
            if (!ok) break;
            for (int r = blk.valid + lane; r < kBlockKeys; r += 32) zero_tile_row<D>(dst, r);
            fence_proxy_async_smem();
            __syncwarp();
            if (leader) mbar_arrive(&ctrl.r_full[sl]);
          }
          ++ld;
        }
      }
    }
    if (leader) {
      if (q_it > 0) drain_bar(&ctrl.a_full, (q_it - 1) & 1, p.error_flag);
      for (uint32_t i = (ld > NS ? ld - NS : 0); i < ld; ++i) drain_bar(&ctrl.r_full[i % NS], (i / NS) & 1, p.error_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t q_desc = make_smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t do_desc = make_smem_desc_sw128(smem_addr(sDO), 16, 1024);
      const uint64_t kv_desc0 = make_smem_desc_sw128(smem_addr(sKV), 16, 1024);            // K-major (K, V)
      const uint64_t kmn_desc0 = make_smem_desc_sw128(smem_addr(sKV), kChunkBytes, 1024);  // K as MN-major B
      auto slot_off = [](uint32_t sl) { return static_cast<uint64_t>(sl) * (C::kTileBytes >> 4); };
      uint32_t q_it = 0, blk = 0, pc = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_items) break;
        const WorkItem it = load_item(p.items, idx);
        if (it.nblk == 0) continue;
        ok = wait_bar(&ctrl.a_full, q_it & 1, abort_flag, p.error_flag);
        if (!ok) break;
        ++q_it;
        for (int j = 0; j < it.nblk; ++j) {
          const uint32_t kseq = 2 * (blk + j), vseq = kseq + 1;
          ok = wait_bar(&ctrl.r_full[kseq % NS], (kseq / NS) & 1, abort_flag, p.error_flag);
          if (ok) ok = wait_bar(&ctrl.r_full[vseq % NS], (vseq / NS) & 1, abort_flag, p.error_flag);
          if (!ok) break;
          tcgen05_fence_after();
          issue_qk<D>(tmem + kColS, q_desc, kv_desc0 + slot_off(kseq % NS));    // S = Q K^T
          issue_qk<D>(tmem + kColDP, do_desc, kv_desc0 + slot_off(vseq % NS));  // dP = dO V^T
          umma_commit(&ctrl.s_full);
          umma_commit(&ctrl.r_empty[vseq % NS]);
          if (j + 1 == it.nblk) umma_commit(&ctrl.a_empty);
          ok = wait_bar(&ctrl.p_full, pc & 1, abort_flag, p.error_flag);
          if (!ok) break;
          ++pc;
          tcgen05_fence_after();
          issue_pv<D>(tmem + kColDQ, tmem + kColS, kmn_desc0 + slot_off(kseq % NS), j > 0);  // dQ += dS K
          umma_commit(&ctrl.r_empty[kseq % NS]);
          if (j + 1 == it.nblk) umma_commit(&ctrl.acc_full);
        }
        blk += it.nblk;
      }
      umma_commit(&ctrl.mma_done);
      drain_bar(&ctrl.mma_done, 0, p.error_flag);
    }
    __syncwarp();
  } else {
    const int lane_base = (warp & 3) * 32;
    const int row = lane_base + lane;
    const int hl = row / T;
    const int tok = row - hl * T;
    const uint32_t s_addr = tmem_addr(tmem, lane_base, kColS);
    const uint32_t dp_addr = tmem_addr(tmem, lane_base, kColDP);
    const uint32_t dq_addr = tmem_addr(tmem, lane_base, kColDQ);
    const float c = p.scale_log2;
    const uint64_t c2 = f32x2(c, c);
    TOut* dq = reinterpret_cast<TOut*>(p.dq);
    uint32_t sc = 0, ac = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_items) break;
      const WorkItem it = load_item(p.items, idx);
      const bool valid = tok < it.q_rows;
      const int64_t token = static_cast<int64_t>(it.q_row0) + tok;
      const int head = it.head_kv * G + hl;
      TOut* qrow = dq + (token * p.num_heads_q + head) * D;
      if (it.nblk == 0) {  // keyless segment: O = 0 does not depend on Q
        if (valid) {
          float z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) store_row32<TOut>(qrow + ch * 32, z);
        }
        continue;
      }
      const int64_t li = static_cast<int64_t>(head) * p.total_q + token;
      const float lse2 = valid ? p.lse[li] * kLog2e : 0.0f;
      const float drow = valid ? p.dvec[li] : 0.0f;
      const uint64_t neg_l2 = f32x2(-lse2, -lse2);
      for (int j = 0; j < it.nblk; ++j) {
        ok = __all_sync(0xffffffffu, wait_bar(&ctrl.s_full, sc & 1, abort_flag, p.error_flag));
        if (!ok) break;
        ++sc;
        tcgen05_fence_after();
        const int rem = load_block(p.blocks, it.blk0 + j).valid;
        if (rem < kBlockKeys) {  // keys past the used length: P = 0 (range uniform over the warp)
          for (int col = rem; col < kBlockKeys; ++col) tmem_st1(s_addr + col, 0xff800000u);
          tmem_wait_st();
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sraw[64], draw[64];
          tmem_ld64_sync(s_addr + half * 64, sraw);
          tmem_ld64_sync(dp_addr + half * 64, draw);
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a, b;
            f32x2_split(ffma2(f32x2(__uint_as_float(sraw[2 * i]), __uint_as_float(sraw[2 * i + 1])), c2, neg_l2),
                        a, b);
            a = ex2_approx(a);
            b = ex2_approx(b);
            const float da = a * (__uint_as_float(draw[2 * i]) - drow);
            const float db = b * (__uint_as_float(draw[2 * i + 1]) - drow);
            pk[i] = pack_bf16x2(da, db);
          }
          tmem_st32(s_addr + half * 32, pk);  // dS pairs: columns [32 half, 32 half + 32)
        }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.p_full);
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_bar(&ctrl.acc_full, ac & 1, abort_flag, p.error_flag));
      if (!ok) break;
      ++ac;
      tcgen05_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32_sync(dq_addr + ch * 32, o);
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * p.scale;
        if (valid) store_row32<TOut>(qrow + ch * 32, x);
      }
    }
    tmem_wait_st();
  }
  tcgen05_fence_before();
  __syncthreads();
  if (warp == 1) {
    tcgen05_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// ---------------------------------------------------------------------------------
// 3. dK, dV
// ---------------------------------------------------------------------------------
template <int D, typename TOut>
__global__ void __launch_bounds__(kBwdThreads, 1)
    gva_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                        const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtrl ctrl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::kTileBytes;
  uint8_t* sSlots = sV + C::kTileBytes;  // 2 slots of {Q tile, dO tile}
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctrl.abort;
  if (threadIdx.x == 0) init_ctrl(ctrl, 2);
  if (warp == 1) {
    tmem_alloc(&ctrl.tmem_base, kBwdTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  const int T = p.tokens_per_tile;
  const int G = p.group;
  // TMEM: S^T [0,128) (P^T pairs overwrite [0,64)), dP^T [128,256) (dS^T pairs overwrite
  // [128,192)), dV [256,256+D), dK [384,384+D)
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
  auto n_tiles = [&](const KvUnit& u) { return (u.q_used + T - 1) / T; };

  if (warp == 0) {
    // As in the dQ kernel: lane 0 copies, the warp clears rows past the used keys of a
    // partial K/V block and the rows of unused tokens of a partial Q / dO tile.
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_do);
    }
    uint32_t kv_it = 0, ld = 0, zph = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_kv_units) break;
      const KvUnit u = load_unit(p.kv_units, idx);
      const int nqt = n_tiles(u);
      if (nqt == 0) continue;
      if (leader) ok = wait_bar(&ctrl.a_empty, (kv_it & 1) ^ 1, abort_flag, p.error_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      {
        uint64_t* bar = u.keys == kBlockKeys ? &ctrl.a_full : &ctrl.zero_bar;
        if (leader) {
          mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch) {
            tma_load_3d(sK + ch * kChunkBytes, &map_k, bar, ch * 64, u.key_row0, u.head_kv);
            tma_load_3d(sV + ch * kChunkBytes, &map_v, bar, ch * 64, u.key_row0, u.head_kv);
          }
        }
        if (u.keys < kBlockKeys) {
          ok = __all_sync(0xffffffffu, wait_bar(&ctrl.zero_bar, zph & 1, abort_flag, p.error_flag));
          if (!ok && leader) drain_bar(&ctrl.zero_bar, zph & 1, p.error_flag);
          ++zph;
          if (!ok) break;
          for (int r = u.keys + lane; r < kBlockKeys; r += 32) {
            zero_tile_row<D>(sK, r);
            zero_tile_row<D>(sV, r);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (leader) mbar_arrive(&ctrl.a_full);
        }
      }
      ++kv_it;
      for (int i = 0; i < nqt && ok; ++i) {
        const uint32_t sl = ld & 1;
        if (leader) ok = wait_bar(&ctrl.r_empty[sl], ((ld >> 1) & 1) ^ 1, abort_flag, p.error_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* tq = sSlots + sl * 2 * C::kTileBytes;
        uint8_t* tdo = tq + C::kTileBytes;
        const int t0 = u.q_row0 + i * T;
        const int vt = min(T, u.q_used - i * T);  // used tokens of this tile
        uint64_t* bar = vt == T ? &ctrl.r_full[sl] : &ctrl.zero_bar;
        if (leader) {
          mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch) {
            tma_load_3d(tq + ch * kChunkBytes, &map_q, bar, ch * 64, t0, u.head_kv * G);
            tma_load_3d(tdo + ch * kChunkBytes, &map_do, bar, ch * 64, t0, u.head_kv * G);
          }
        }
        if (vt < T) {
          ok = __all_sync(0xffffffffu, wait_bar(&ctrl.zero_bar, zph & 1, abort_flag, p.error_flag));
          if (!ok && leader) drain_bar(&ctrl.zero_bar, zph & 1, p.error_flag);
          ++zph;
          if (!ok) break;
          const int dead = T - vt;  // rows h * T + t, t >= vt, of every head h
          for (int x = lane; x < G * dead; x += 32) {
            const int h = x / dead, r = h * T + vt + (x - h * dead);
            zero_tile_row<D>(tq, r);
            zero_tile_row<D>(tdo, r);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (leader) mbar_arrive(&ctrl.r_full[sl]);
        }
        ++ld;
      }
    }
    if (leader) {
      if (kv_it > 0) drain_bar(&ctrl.a_full, (kv_it - 1) & 1, p.error_flag);
      for (uint32_t i = (ld > 2 ? ld - 2 : 0); i < ld; ++i) drain_bar(&ctrl.r_full[i & 1], (i >> 1) & 1, p.error_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t k_desc = make_smem_desc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t v_desc = make_smem_desc_sw128(smem_addr(sV), 16, 1024);
      const uint64_t slot_k0 = make_smem_desc_sw128(smem_addr(sSlots), 16, 1024);            // K-major
      const uint64_t slot_mn0 = make_smem_desc_sw128(smem_addr(sSlots), kChunkBytes, 1024);  // MN-major B
      constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
      uint32_t kv_it = 0, qi = 0, pc = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_kv_units) break;
        const KvUnit u = load_unit(p.kv_units, idx);
        const int nqt = n_tiles(u);
        if (nqt == 0) continue;
        ok = wait_bar(&ctrl.a_full, kv_it & 1, abort_flag, p.error_flag);
        if (!ok) break;
        ++kv_it;
        for (int i = 0; i < nqt; ++i) {
          const uint32_t sl = qi & 1;
          ok = wait_bar(&ctrl.r_full[sl], (qi >> 1) & 1, abort_flag, p.error_flag);
          if (!ok) break;
          tcgen05_fence_after();
          const uint64_t qk = slot_k0 + sl * 2 * kTileUnits, dok = qk + kTileUnits;
          const uint64_t qmn = slot_mn0 + sl * 2 * kTileUnits, domn = qmn + kTileUnits;
          issue_qk<D>(tmem + kColS, k_desc, qk);    // S^T = K Q^T
          issue_qk<D>(tmem + kColDP, v_desc, dok);  // dP^T = V dO^T
          umma_commit(&ctrl.s_full);
          ok = wait_bar(&ctrl.p_full, pc & 1, abort_flag, p.error_flag);
          if (!ok) break;
          ++pc;
          tcgen05_fence_after();
          issue_pv<D>(tmem + kColDV, tmem + kColS, domn, i > 0);  // dV += P^T dO
          issue_pv<D>(tmem + kColDK, tmem + kColDP, qmn, i > 0);  // dK += dS^T Q
          umma_commit(&ctrl.r_empty[sl]);
          ++qi;
        }
        if (!ok) break;
        umma_commit(&ctrl.a_empty);
        umma_commit(&ctrl.acc_full);
      }
      umma_commit(&ctrl.mma_done);
      drain_bar(&ctrl.mma_done, 0, p.error_flag);
    }
    __syncwarp();
  } else {
    const int lane_base = (warp & 3) * 32;
    const int key = lane_base + lane;  // S^T row = TMEM lane = key within the block
    const int rhl = key / T;           // as a loader: the Q-tile row this thread fetches
    const int rtok = key - rhl * T;
    const uint32_t s_addr = tmem_addr(tmem, lane_base, kColS);
    const uint32_t dp_addr = tmem_addr(tmem, lane_base, kColDP);
    const float c = p.scale_log2;
    TOut* dk = reinterpret_cast<TOut*>(p.dk);
    TOut* dv = reinterpret_cast<TOut*>(p.dv);
    uint32_t sc = 0, ac = 0, tiles = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_kv_units) break;
      const KvUnit u = load_unit(p.kv_units, idx);
      const int nqt = n_tiles(u);
      const bool key_valid = key < u.keys;
      const int64_t krow = static_cast<int64_t>(u.key_row0) + key;
      TOut* dkrow = dk + (krow * p.num_heads_kv + u.head_kv) * D;
      TOut* dvrow = dv + (krow * p.num_heads_kv + u.head_kv) * D;
      if (nqt == 0) {  // no query attends these keys
        if (key_valid) {
          float z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            store_row32<TOut>(dkrow + ch * 32, z);
            store_row32<TOut>(dvrow + ch * 32, z);
          }
        }
        continue;
      }
      for (int i = 0; i < nqt; ++i) {
        const int par = tiles & 1;
        ++tiles;
        // this thread fetches the log2-LSE and D of Q-tile row `key`; +inf LSE (P = 0)
        // for rows past the used queries
        const bool rvalid = i * T + rtok < u.q_used;
        const int64_t li = static_cast<int64_t>(u.head_kv * G + rhl) * p.total_q + u.q_row0 + i * T + rtok;
        ctrl.xl[par][key] = rvalid ? p.lse[li] * kLog2e : CUDART_INF_F;
        ctrl.xd[par][key] = rvalid ? p.dvec[li] : 0.0f;
        bool fine = __all_sync(0xffffffffu, wait_bar(&ctrl.s_full, sc & 1, abort_flag, p.error_flag));
        ++sc;
        if (named_barrier_or(1, 128, !fine)) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sraw[64], draw[64];
          tmem_ld64_sync(s_addr + half * 64, sraw);
          tmem_ld64_sync(dp_addr + half * 64, draw);
          uint32_t pp[32], pd[32];
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) {
            const int col = half * 64 + 2 * i2;
            float a = ex2_approx(fmaf(__uint_as_float(sraw[2 * i2]), c, -ctrl.xl[par][col]));
            float b = ex2_approx(fmaf(__uint_as_float(sraw[2 * i2 + 1]), c, -ctrl.xl[par][col + 1]));
            float da = a * (__uint_as_float(draw[2 * i2]) - ctrl.xd[par][col]);
            float db = b * (__uint_as_float(draw[2 * i2 + 1]) - ctrl.xd[par][col + 1]);
            if (!key_valid) a = b = da = db = 0.0f;
            pp[i2] = pack_bf16x2(a, b);
            pd[i2] = pack_bf16x2(da, db);
          }
          tmem_st32(s_addr + half * 32, pp);   // P^T pairs
          tmem_st32(dp_addr + half * 32, pd);  // dS^T pairs
        }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.p_full);
      }
      if (!ok) break;
      {  // all four warps take the same decision (the next unit's barrier needs all 128)
        const bool fine = __all_sync(0xffffffffu, wait_bar(&ctrl.acc_full, ac & 1, abort_flag, p.error_flag));
        if (named_barrier_or(1, 128, !fine)) break;
      }
      ++ac;
      tcgen05_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        float x[32];
        tmem_ld32_sync(tmem_addr(tmem, lane_base, kColDV + ch * 32), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]);
        if (key_valid) store_row32<TOut>(dvrow + ch * 32, x);
        tmem_ld32_sync(tmem_addr(tmem, lane_base, kColDK + ch * 32), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * p.scale;
        if (key_valid) store_row32<TOut>(dkrow + ch * 32, x);
      }
    }
    tmem_wait_st();
  }
  tcgen05_fence_before();
  __syncthreads();
  if (warp == 1) {
    tcgen05_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

template <int D, typename TQ, typename TKV>
cudaError_t launch_bwd_impl(const BwdParams& p, const MergeUnit* units, int32_t num_units, const void* out,
                            const void* d_out, float* dvec, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdo, int dq_grid, int sms,
                            cudaStream_t stream) {
  if (num_units > 0) {
    gva_bwd_dvec_kernel<D><<<min(num_units, sms * 8), 256, 0, stream>>>(
        units, num_units, static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(d_out), dvec,
        p.total_q, p.num_heads_q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.num_items > 0) {
    auto kq = gva_bwd_dq_kernel<D, TQ>;
    cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<D>::kSmemDq);
    if (e != cudaSuccess) return e;
    kq<<<dq_grid, kBwdThreads, BCfg<D>::kSmemDq, stream>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.num_kv_units > 0) {
    auto kkv = gva_bwd_dkdv_kernel<D, TKV>;
    cudaError_t e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<D>::kSmemDkv);
    if (e != cudaSuccess) return e;
    kkv<<<min(p.num_kv_units, sms), kBwdThreads, BCfg<D>::kSmemDkv, stream>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_bwd_d(bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units, int32_t num_units,
                         const void* out, const void* d_out, float* dvec, const CUtensorMap& mq,
                         const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo, int dq_grid,
                         cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dq_f32) {
    return dkv_f32 ? launch_bwd_impl<D, float, float>(p, units, num_units, out, d_out, dvec, mq, mk, mv, mdo, dq_grid,
                                                      sms, stream)
                   : launch_bwd_impl<D, float, __nv_bfloat16>(p, units, num_units, out, d_out, dvec, mq, mk, mv,
                                                              mdo, dq_grid, sms, stream);
  }
  return dkv_f32 ? launch_bwd_impl<D, __nv_bfloat16, float>(p, units, num_units, out, d_out, dvec, mq, mk, mv, mdo,
                                                            dq_grid, sms, stream)
                 : launch_bwd_impl<D, __nv_bfloat16, __nv_bfloat16>(p, units, num_units, out, d_out, dvec, mq, mk,
                                                                    mv, mdo, dq_grid, sms, stream);
}

}  // namespace

cudaError_t launch_backward(int head_dim, bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units,
                            int32_t num_units, const void* out, const void* d_out, float* dvec,
                            const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, int dq_grid, cudaStream_t stream) {
  if (head_dim == 128)
    return launch_bwd_d<128>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, map_q, map_k, map_v, map_do,
                             dq_grid, stream);
  return launch_bwd_d<64>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, map_q, map_k, map_v, map_do,
                          dq_grid, stream);
}

}  // namespace gva
