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
//      TMEM, P and dS by the compute threads, dQ += dS K with dS read from TMEM.
//   3. gva_bwd_dkdv_kernel: one key block of one KV head per unit, streaming the
//      segment's Q / dO tiles: S^T = K Q^T and dP^T = V dO^T into TMEM, P^T and dS^T by
//      the compute threads, dV += P^T dO and dK += dS^T Q accumulated in TMEM, then
//      written once. No atomics anywhere.
// Both kernels run two warpgroups of compute threads (one TMEM lane each), each on one
// 64-column half of a block's scores, and keep the tensor core busy while they work:
// the dQ kernel double-buffers S in TMEM and hands dP back as soon as it sits in
// registers, so block m+1's products run during block m's exponentials; the dK/dV
// kernel, whose TMEM is full (S^T, dP^T and both accumulators), issues the products per
// half and runs one half ahead. Operand rows past the used lengths (gaps, padding,
// possibly NaN) are zeroed in shared memory before an MMA could multiply them by a zero
// weight. Block-causal plans take separate kCausal instantiations.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "gva_device_common.cuh"
#include "gva_internal.h"
#include "sm103_ptx.cuh"

namespace gva {
namespace {

constexpr int kBwdThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 compute (two warpgroups)
constexpr uint32_t kBwdTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTileRows * D * 2;  // a Q, dO, K or V tile of 128 rows
  // dQ kernel: K lives from S(m) to dQ(m), which comes two products later, V only
  // until dP(m); three K slots and two V slots keep the next block's loads ahead.
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kSmemDq = (2 + kKSlots + kVSlots) * kTileBytes + 1024;
  static constexpr int kSmemDkv = 2 * kTileBytes + 2 * 2 * kTileBytes + 1024;
  static_assert(kSmemDq <= 227 * 1024 && kSmemDkv <= 227 * 1024, "shared memory budget");
};

// Zero row `row` of a 128-row tile (its 128-byte piece in every column chunk); the
// swizzle only permutes 16-byte pieces within a row, so a whole row clears in place.
template <int D>
__device__ __forceinline__ void zero_tile_row(uint8_t* tile, int row) {
#pragma unroll
  for (int ch = 0; ch < D / 64; ++ch) {
    uint4* r = reinterpret_cast<uint4*>(tile + ch * kChunkBytes + row * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = make_uint4(0, 0, 0, 0);
  }
}

// Zero rows [filled, 128) of `n` 128-row tiles spaced `stride` bytes apart, with all
// `nthreads` threads of the block. A folded Q / dO tile fills T * G rows (T =
// floor(128 / G) tokens of G heads); when G does not divide 128 the copies never write
// the remaining rows, which would otherwise meet zero weights (0 * NaN) in the MMAs.
template <int D>
__device__ __forceinline__ void zero_tile_tails(uint8_t* tile0, int stride, int n, int filled, int nthreads) {
  const int pad = kTileRows - filled;
  for (int x = threadIdx.x; x < n * pad * (D / 64) * 8; x += nthreads) {
    const int piece = x % 8, rest = x / 8;
    const int ch = rest % (D / 64), rest2 = rest / (D / 64);
    const int r = filled + rest2 % pad, t = rest2 / pad;
    *reinterpret_cast<uint4*>(tile0 + t * stride + ch * kChunkBytes + r * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ KvUnit load_unit(const KvUnit* units, int idx) {
  const int4* p = reinterpret_cast<const int4*>(units + idx);
  const int4 a = __ldg(p), b = __ldg(p + 1);
  KvUnit u;
  u.key_row0 = a.x; u.keys = a.y; u.seg0 = a.z; u.n_tiles = a.w;
  u.head_kv = b.x; u.tile0 = b.y; u.key_pos0 = b.z; u.pos_shift = b.w;
  return u;
}

// The Q tiles of a dK / dV unit, in order: tiles tile0 .. of its first segment, then
// every tile of each further segment. `next` must only be called while tiles remain.
struct TileWalk {
  const int2* segs;
  int s, k;   // current SegRef and tile within its segment
  int2 seg;   // (first token row, used rows) of that segment
  __device__ __forceinline__ void start(const SegRef* list, const KvUnit& u) {
    segs = reinterpret_cast<const int2*>(list);
    s = u.seg0;
    k = u.tile0;
    seg = __ldg(segs + s);
  }
  __device__ __forceinline__ void next(int T) {
    if (++k * T >= seg.y) {
      k = 0;
      seg = __ldg(segs + (++s));
    }
  }
};

// dK / dV kernel control block.
struct BwdCtrl {
  float xl[2][kTileRows];  // per-column log2-LSE of the current Q tile (two tiles in flight)
  float xd[2][kTileRows];  // per-column D
  int xlim[2][kTileRows];  // block-causal: per-column key limit
  uint64_t a_full, a_empty;            // K + V blocks
  uint64_t r_full[2], r_empty[2];      // Q / dO slots
  uint64_t zero_bar;                   // partial tiles: the producer's own copy wait
  uint64_t s_full, dp_full;            // S^T ready; dP^T ready
  uint64_t p_full[2], ds_full[2];      // per column half: P^T in TMEM; dS^T in TMEM
  uint64_t acc_full, mma_done;
  uint32_t tmem_base;
  int abort;
};

// dQ kernel control block (no per-column staging; K and V in separate rings).
struct DqCtrl {
  uint64_t a_full, a_empty;  // Q + dO tiles
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t zero_bar;         // partial blocks: the producer's own copy wait
  uint64_t p_full[2];        // per S buffer: dS in TMEM (256 compute threads)
  uint64_t dp_full, dp_consumed;
  uint64_t acc_full, mma_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void init_dq_ctrl(DqCtrl& c) {
  mbar_init(&c.a_full, 1);
  mbar_init(&c.a_empty, 1);
  for (int i = 0; i < 3; ++i) {
    mbar_init(&c.k_full[i], 1);
    mbar_init(&c.k_empty[i], 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&c.v_full[i], 1);
    mbar_init(&c.v_empty[i], 1);
    mbar_init(&c.p_full[i], 2 * kTileRows);
  }
  mbar_init(&c.zero_bar, 1);
  mbar_init(&c.dp_full, 1);
  mbar_init(&c.dp_consumed, 2 * kTileRows);
  mbar_init(&c.acc_full, 1);
  mbar_init(&c.mma_done, 1);
  c.abort = 0;
  fence_barrier_init();
}

__device__ __forceinline__ void init_ctrl(BwdCtrl& c) {
  mbar_init(&c.a_full, 1);
  mbar_init(&c.a_empty, 1);
  for (int i = 0; i < 2; ++i) {
    mbar_init(&c.r_full[i], 1);
    mbar_init(&c.r_empty[i], 1);
    mbar_init(&c.p_full[i], kTileRows);
    mbar_init(&c.ds_full[i], kTileRows);
  }
  mbar_init(&c.s_full, 1);
  mbar_init(&c.dp_full, 1);
  mbar_init(&c.zero_bar, 1);
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

// D[128 x D] (+)= A[128 x 64] B[rows 64h .. 64h + 63] with A (bf16 pairs, 32 columns)
// in TMEM and B MN-major in shared memory.
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc, int h,
                                              uint32_t accumulate) {
  constexpr uint32_t idesc = make_idesc_bf16(kTileRows, D, true);
  const uint64_t b = b_desc + static_cast<uint64_t>(h) * ((64 * 128) >> 4);
  umma_bf16_ts(tmem_d, tmem_a, b, idesc, accumulate);
#pragma unroll
  for (int kk = 1; kk < 4; ++kk) umma_bf16_ts(tmem_d, tmem_a + kk * 8, b + ((kk * 16 * 128) >> 4), idesc, 1u);
}

template <typename TOut, int N>
__device__ __forceinline__ void store_zero_cols(TOut* row) {
  float z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
  for (int c = 0; c < N / 32; ++c) store_row32<TOut>(row + c * 32, z);
}

// ---------------------------------------------------------------------------------
// 2. dQ
// ---------------------------------------------------------------------------------
template <int D, typename TOut, bool kCausal>
__global__ void __launch_bounds__(kBwdThreads, 1)
    gva_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                      const BwdParams p) {
  using C = BCfg<D>;
  constexpr uint32_t NK = C::kKSlots, NV = C::kVSlots;
  extern __shared__ uint8_t smem_raw[];
  __shared__ DqCtrl ctrl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = sQ + C::kTileBytes;
  uint8_t* sK = sDO + C::kTileBytes;      // NK slots; block m in slot m % NK
  uint8_t* sV = sK + NK * C::kTileBytes;  // NV slots; block m in slot m % NV
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctrl.abort;
  if (threadIdx.x == 0) init_dq_ctrl(ctrl);
  if (warp == 1) {
    tmem_alloc(&ctrl.tmem_base, kBwdTmemCols);
    tmem_relinquish_alloc_permit();
  }
  const int T = p.tokens_per_tile;
  const int G = p.group;
  zero_tile_tails<D>(sQ, C::kTileBytes, 2, T * G, kBwdThreads);  // the Q and dO tiles
  fence_proxy_async_smem();
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  const uint32_t q_tile_bytes = static_cast<uint32_t>(T * G) * D * 2;  // bytes one folded tile's copies bring
  // TMEM: two S buffers [0,128) and [128,256) (block m uses buffer m & 1), dP
  // [256,384), dQ [384,384+D). The dS of key half h (bf16 pairs) overwrites columns
  // [64h, 64h+32) of its block's S buffer. With S double-buffered, the products of
  // block m+1 run on the tensor core while the compute threads turn block m into dS;
  // dP has one buffer, released as soon as the compute threads hold it in registers.
  constexpr uint32_t kColS = 0, kColDP = 256, kColDQ = 384;

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
    uint32_t q_it = 0, m = 0, zph = 0;  // m: blocks of this CTA so far
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_items) break;
      const WorkItem it = load_item(p.items, idx);
      if (it.nblk == 0) continue;
      if (leader) ok = wait_bar(&ctrl.a_empty, (q_it & 1) ^ 1, abort_flag, p.error_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (leader) {
        mbar_arrive_expect_tx(&ctrl.a_full, 2 * q_tile_bytes);
#pragma unroll
        for (int ch = 0; ch < C::kChunks; ++ch) {
          tma_load_3d(sQ + ch * kChunkBytes, &map_q, &ctrl.a_full, ch * 64, it.q_row0, it.head_kv * G);
          tma_load_3d(sDO + ch * kChunkBytes, &map_do, &ctrl.a_full, ch * 64, it.q_row0, it.head_kv * G);
        }
      }
      ++q_it;
      for (int j = 0; j < it.nblk && ok; ++j, ++m) {
        const KeyBlock blk = load_block(p.blocks, it.blk0 + j);
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t nslots = kv == 0 ? NK : NV;
          const uint32_t sl = m % nslots;
          uint64_t* empty = kv == 0 ? &ctrl.k_empty[sl] : &ctrl.v_empty[sl];
          uint64_t* full = kv == 0 ? &ctrl.k_full[sl] : &ctrl.v_full[sl];
          if (leader) ok = wait_bar(empty, ((m / nslots) & 1) ^ 1, abort_flag, p.error_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          uint8_t* dst = (kv == 0 ? sK : sV) + sl * C::kTileBytes;
          const CUtensorMap* map = kv == 0 ? &map_k : &map_v;
          uint64_t* bar = blk.valid == kBlockKeys ? full : &ctrl.zero_bar;
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
            if (leader) mbar_arrive(full);
          }
        }
      }
    }
    if (leader) {
      // after an abort the drains below may wait on a load that was never issued;
      // each wait is bounded and the error is already recorded
      if (q_it > 0) drain_bar(&ctrl.a_full, (q_it - 1) & 1, p.error_flag);
      for (uint32_t i = (m > NK ? m - NK : 0); i < m; ++i) drain_bar(&ctrl.k_full[i % NK], (i / NK) & 1, p.error_flag);
      for (uint32_t i = (m > NV ? m - NV : 0); i < m; ++i) drain_bar(&ctrl.v_full[i % NV], (i / NV) & 1, p.error_flag);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // Per block m: S(m+1) into the other S buffer, dP(m+1) once the compute threads
      // hold dP(m), then dQ += dS(m) K(m) once dS(m) is in TMEM.
      const uint64_t q_desc = make_smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t do_desc = make_smem_desc_sw128(smem_addr(sDO), 16, 1024);
      const uint64_t k_desc0 = make_smem_desc_sw128(smem_addr(sK), 16, 1024);             // K-major
      const uint64_t v_desc0 = make_smem_desc_sw128(smem_addr(sV), 16, 1024);             // K-major
      const uint64_t kmn_desc0 = make_smem_desc_sw128(smem_addr(sK), kChunkBytes, 1024);  // K as MN-major B
      constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
      uint32_t q_it = 0, n = 0;  // n: blocks of this CTA so far (global block counter)
      bool ok = true;
      auto wait_kv = [&](uint32_t m) {
        bool r = wait_bar(&ctrl.k_full[m % NK], (m / NK) & 1, abort_flag, p.error_flag);
        if (r) r = wait_bar(&ctrl.v_full[m % NV], (m / NV) & 1, abort_flag, p.error_flag);
        if (r) tcgen05_fence_after();
        return r;
      };
      auto issue_s = [&](uint32_t m) {  // complete before dP(m), which is issued after it
        issue_qk<D>(tmem + kColS + 128 * (m & 1), q_desc, k_desc0 + (m % NK) * kTileUnits);
      };
      auto issue_dp = [&](uint32_t m) {  // after the compute threads released dP(m - 1)
        if (m > 0) {
          if (!wait_bar(&ctrl.dp_consumed, (m - 1) & 1, abort_flag, p.error_flag)) return false;
          tcgen05_fence_after();
        }
        issue_qk<D>(tmem + kColDP, do_desc, v_desc0 + (m % NV) * kTileUnits);
        umma_commit(&ctrl.dp_full);
        umma_commit(&ctrl.v_empty[m % NV]);  // V(m) read
        return true;
      };
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_items) break;
        const WorkItem it = load_item(p.items, idx);
        if (it.nblk == 0) continue;
        ok = wait_bar(&ctrl.a_full, q_it & 1, abort_flag, p.error_flag);
        if (ok) ok = wait_kv(n);
        if (!ok) break;
        ++q_it;
        issue_s(n);
        ok = issue_dp(n);
        if (!ok) break;
        if (it.nblk == 1) umma_commit(&ctrl.a_empty);  // Q, dO read
        for (int j = 0; j < it.nblk; ++j) {
          const uint32_t m = n + j;
          if (j + 1 < it.nblk) {
            ok = wait_kv(m + 1);
            if (!ok) break;
            issue_s(m + 1);
            ok = issue_dp(m + 1);
            if (!ok) break;
            if (j + 2 == it.nblk) umma_commit(&ctrl.a_empty);
          }
          // dS(m) is in TMEM (both warpgroups; for the first block of an item they
          // arrive only after reading out the previous item's dQ)
          ok = wait_bar(&ctrl.p_full[m & 1], (m >> 1) & 1, abort_flag, p.error_flag);
          if (!ok) break;
          tcgen05_fence_after();
          const uint32_t sb = tmem + kColS + 128 * (m & 1);
          issue_pv_half<D>(tmem + kColDQ, sb, kmn_desc0 + (m % NK) * kTileUnits, 0, j > 0);
          issue_pv_half<D>(tmem + kColDQ, sb + 64, kmn_desc0 + (m % NK) * kTileUnits, 1, 1u);
          umma_commit(&ctrl.k_empty[m % NK]);  // K(m) read
        }
        if (!ok) break;
        umma_commit(&ctrl.acc_full);
        n += it.nblk;
      }
      umma_commit(&ctrl.mma_done);
      drain_bar(&ctrl.mma_done, 0, p.error_flag);
    }
    __syncwarp();
  } else {
    const int wg = (warp - 2) >> 2;  // key half of each block this thread turns into dS
    const int lane_base = (warp & 3) * 32;
    const int row = lane_base + lane;
    const int hl = row / T;
    const int tok = row - hl * T;
    const uint32_t dp_addr = tmem_addr(tmem, lane_base, kColDP + 64 * wg);
    const uint32_t dq_addr = tmem_addr(tmem, lane_base, kColDQ + (D / 2) * wg);
    const float c = p.scale_log2;
    const uint64_t c2 = f32x2(c, c);
    TOut* dq = reinterpret_cast<TOut*>(p.dq);
    uint32_t n = 0, ac = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_items) break;
      const WorkItem it = load_item(p.items, idx);
      const bool valid = hl < G && tok < it.q_rows;
      const int64_t token = static_cast<int64_t>(it.q_row0) + tok;
      const int head = it.head_kv * G + hl;
      TOut* qrow = dq + (token * p.num_heads_q + head) * D + (D / 2) * wg;
      if (it.nblk == 0) {  // keyless segment: O = 0 does not depend on Q
        if (valid) store_zero_cols<TOut, D / 2>(qrow);
        continue;
      }
      const int64_t li = static_cast<int64_t>(head) * p.total_q + token;
      // block-causal: keys of the segment this row sees (one prefix range, so block j
      // holds keys 128 j ..); otherwise every used key of every block
      int row_limit = 1;
      if constexpr (kCausal) {
        const int pos = it.q_pos0 + tok;
        row_limit = pos < 0 ? 0 : min(it.k_len, (pos / p.causal_block + 1) * p.causal_block);
      }
      // a row that sees no key (its LSE is -inf) takes +inf here, so its P is 0
      const float lse2 = valid && row_limit > 0 ? p.lse[li] * kLog2e : CUDART_INF_F;
      const float drow = valid ? p.dvec[li] : 0.0f;
      const uint64_t neg_l2 = f32x2(-lse2, -lse2);
      // used keys of each block, fetched one block ahead (any block of a key range can
      // be partial)
      int valid_next = load_block(p.blocks, it.blk0).valid;
      for (int j = 0; j < it.nblk; ++j, ++n) {
        const int valid_keys = valid_next;
        if (j + 1 < it.nblk) valid_next = load_block(p.blocks, it.blk0 + j + 1).valid;
        // dP(n) complete implies S(n) complete (issued before it by the same thread)
        ok = __all_sync(0xffffffffu, wait_bar(&ctrl.dp_full, n & 1, abort_flag, p.error_flag));
        if (!ok) break;
        tcgen05_fence_after();
        const uint32_t s_addr = tmem_addr(tmem, lane_base, kColS + 128 * (n & 1) + 64 * wg);
        uint32_t sraw[64], dpr[64];
        tmem_ld64x2_sync(s_addr, sraw, dp_addr, dpr);
        tcgen05_fence_before();
        mbar_arrive(&ctrl.dp_consumed);  // the tensor core may overwrite dP now
        // keys of this half the row sees: the block's used keys, capped by the row's
        // block-causal limit (block-causal plans have one prefix range)
        const int rem = (kCausal ? min(valid_keys, row_limit - j * kBlockKeys) : valid_keys) - 64 * wg;
        if (rem < 64) {  // keys past the used length: P = 0 (uniform over the warp)
#pragma unroll
          for (int i = 0; i < 64; ++i) sraw[i] = i < rem ? sraw[i] : 0xff800000u;
        }
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a, b;
            f32x2_split(ffma2(f32x2(__uint_as_float(sraw[32 * part + 2 * i]), __uint_as_float(sraw[32 * part + 2 * i + 1])),
                              c2, neg_l2),
                        a, b);
            a = ex2_approx(a);
            b = ex2_approx(b);
            pk[i] = pack_bf16x2(a * (__uint_as_float(dpr[32 * part + 2 * i]) - drow),
                                b * (__uint_as_float(dpr[32 * part + 2 * i + 1]) - drow));
          }
          tmem_st16(s_addr + part * 16, pk);  // dS pairs: columns [16 part, 16 part + 16) of the half
        }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.p_full[n & 1]);
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_bar(&ctrl.acc_full, ac & 1, abort_flag, p.error_flag));
      if (!ok) break;
      ++ac;
      tcgen05_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t o[32];
        tmem_ld32_sync(dq_addr + ch * 32, o);
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * p.scale;
        if (valid) store_row32<TOut>(qrow + ch * 32, x);
      }
    }
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
template <int D, typename TOut, bool kCausal>
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
  if (threadIdx.x == 0) init_ctrl(ctrl);
  if (warp == 1) {
    tmem_alloc(&ctrl.tmem_base, kBwdTmemCols);
    tmem_relinquish_alloc_permit();
  }
  const int T = p.tokens_per_tile;
  const int G = p.group;
  zero_tile_tails<D>(sSlots, C::kTileBytes, 4, T * G, kBwdThreads);  // both slots' Q and dO tiles
  fence_proxy_async_smem();
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  const uint32_t q_tile_bytes = static_cast<uint32_t>(T * G) * D * 2;  // bytes one folded tile's copies bring
  // TMEM: S^T [0,128), dP^T [128,256), dV [256,256+D), dK [384,384+D). Column half h
  // (Q-tile rows 64h .. 64h+63) of S^T / dP^T is [64h, +64) / [128+64h, +64); its P^T
  // (bf16 pairs) overwrites [64h, +32) and its dS^T [128+64h, +32). P^T is ready before
  // dS^T, so dV += P^T dO runs while the compute threads still form dS^T; the next S^T
  // follows the dV products and the next dP^T the dK products.
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

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
      const int nqt = u.n_tiles;
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
      TileWalk tw;
      tw.start(p.kv_segs, u);
      for (int i = 0; i < nqt && ok; ++i) {
        if (i > 0) tw.next(T);
        const uint32_t sl = ld & 1;
        if (leader) ok = wait_bar(&ctrl.r_empty[sl], ((ld >> 1) & 1) ^ 1, abort_flag, p.error_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* tq = sSlots + sl * 2 * C::kTileBytes;
        uint8_t* tdo = tq + C::kTileBytes;
        const int t0 = tw.seg.x + tw.k * T;
        const int vt = min(T, tw.seg.y - tw.k * T);  // used tokens of this tile
        uint64_t* bar = vt == T ? &ctrl.r_full[sl] : &ctrl.zero_bar;
        if (leader) {
          mbar_arrive_expect_tx(bar, 2 * q_tile_bytes);
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
      // Pipe order per tile t: dV(t) per half as its P^T lands, S^T(t+1), dK(t) per half
      // as its dS^T lands, dP^T(t+1); the exponentials of tile t+1 and the dS^T of tile t
      // overlap these products.
      const uint64_t k_desc = make_smem_desc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t v_desc = make_smem_desc_sw128(smem_addr(sV), 16, 1024);
      const uint64_t slot_k0 = make_smem_desc_sw128(smem_addr(sSlots), 16, 1024);            // K-major
      const uint64_t slot_mn0 = make_smem_desc_sw128(smem_addr(sSlots), kChunkBytes, 1024);  // MN-major B
      constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
      uint32_t kv_it = 0, qi = 0;  // qi: Q tiles so far (global tile counter t)
      uint32_t pc[2] = {0, 0}, dc[2] = {0, 0};
      bool ok = true;
      auto wait_tile = [&](uint32_t t) {
        const bool r = wait_bar(&ctrl.r_full[t & 1], (t >> 1) & 1, abort_flag, p.error_flag);
        if (r) tcgen05_fence_after();
        return r;
      };
      auto issue_s = [&](uint32_t t) {  // S^T(t) = K Q_t^T (after tile t-1's dV read P^T)
        issue_qk<D>(tmem + kColS, k_desc, slot_k0 + (t & 1) * 2 * kTileUnits);
        umma_commit(&ctrl.s_full);
      };
      auto issue_dp = [&](uint32_t t) {  // dP^T(t) = V dO_t^T (after tile t-1's dK read dS^T)
        issue_qk<D>(tmem + kColDP, v_desc, slot_k0 + (t & 1) * 2 * kTileUnits + kTileUnits);
        umma_commit(&ctrl.dp_full);
      };
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_kv_units) break;
        const KvUnit u = load_unit(p.kv_units, idx);
        const int nqt = u.n_tiles;
        if (nqt == 0) continue;
        ok = wait_bar(&ctrl.a_full, kv_it & 1, abort_flag, p.error_flag);
        if (ok) ok = wait_tile(qi);
        if (!ok) break;
        ++kv_it;
        issue_s(qi);
        issue_dp(qi);
        if (nqt == 1) umma_commit(&ctrl.a_empty);  // K, V read
        for (int i = 0; i < nqt; ++i) {
          const uint32_t t = qi + i;
          const bool more = i + 1 < nqt;
          const uint64_t qmn = slot_mn0 + (t & 1) * 2 * kTileUnits, domn = qmn + kTileUnits;
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // dV += P^T dO
            // the unit's first products overwrite dV / dK: both warpgroups must be done
            // reading the previous unit's accumulators (they arrive after their epilogue)
            ok = wait_bar(&ctrl.p_full[h], pc[h] & 1, abort_flag, p.error_flag);
            if (ok && i == 0 && h == 0) ok = wait_bar(&ctrl.p_full[1], pc[1] & 1, abort_flag, p.error_flag);
            if (!ok) break;
            ++pc[h];
            tcgen05_fence_after();
            issue_pv_half<D>(tmem + kColDV, tmem + kColS + 64 * h, domn, h, (i > 0 || h > 0) ? 1u : 0u);
          }
          if (ok && more) {
            ok = wait_tile(t + 1);
            if (ok) issue_s(t + 1);
          }
          if (!ok) break;
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // dK += dS^T Q
            ok = wait_bar(&ctrl.ds_full[h], dc[h] & 1, abort_flag, p.error_flag);
            if (!ok) break;
            ++dc[h];
            tcgen05_fence_after();
            issue_pv_half<D>(tmem + kColDK, tmem + kColDP + 64 * h, qmn, h, (i > 0 || h > 0) ? 1u : 0u);
          }
          if (!ok) break;
          umma_commit(&ctrl.r_empty[t & 1]);
          if (more) {
            issue_dp(t + 1);
            if (i + 2 == nqt) umma_commit(&ctrl.a_empty);
          }
        }
        if (!ok) break;
        qi += nqt;
        umma_commit(&ctrl.acc_full);
      }
      umma_commit(&ctrl.mma_done);
      drain_bar(&ctrl.mma_done, 0, p.error_flag);
    }
    __syncwarp();
  } else {
    const int wg = (warp - 2) >> 2;        // column half: Q-tile rows 64 wg .. 64 wg + 63
    const int tid = threadIdx.x - 64 - 128 * wg;  // 0 .. 127 within the warpgroup
    const int lane_base = (warp & 3) * 32;
    const int key = lane_base + lane;  // epilogue: S^T row = TMEM lane = key within the block
    const int g = lane >> 2, c4 = lane & 3;  // 16-lane shapes: lane offset and column pair of this thread
    const int lrow = 64 * wg + (tid & 63);  // as a loader (tid < 64): the Q-tile row it fetches
    const int rhl = lrow / T;
    const int rtok = lrow - rhl * T;
    const float c = p.scale_log2;
    TOut* dk = reinterpret_cast<TOut*>(p.dk);
    TOut* dv = reinterpret_cast<TOut*>(p.dv);
    uint32_t sc = 0, ac = 0, tiles = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_kv_units) break;
      const KvUnit u = load_unit(p.kv_units, idx);
      const int nqt = u.n_tiles;
      const bool key_valid = key < u.keys;
      const int64_t krow = static_cast<int64_t>(u.key_row0) + key;
      TOut* dkrow = dk + (krow * p.num_heads_kv + u.head_kv) * D + (D / 2) * wg;
      TOut* dvrow = dv + (krow * p.num_heads_kv + u.head_kv) * D + (D / 2) * wg;
      if (nqt == 0) {  // no query attends these keys
        if (key_valid) {
          store_zero_cols<TOut, D / 2>(dkrow);
          store_zero_cols<TOut, D / 2>(dvrow);
        }
        continue;
      }
      // log2-LSE and D of this half's Q-tile rows (loader threads tid < 64), fetched one
      // tile ahead; +inf LSE (P = 0) and D = 0 past the used rows
      const int64_t lhead = static_cast<int64_t>(u.head_kv * G + rhl) * p.total_q;
      TileWalk fw;  // the tile the next fetch reads
      if (tid < 64 && nqt > 0) fw.start(p.kv_segs, u);
      auto fetch = [&](float& xl_v, float& xd_v, int& lim_v) {
        const int r = fw.k * T + rtok;  // row within the segment
        const bool rvalid = rhl < G && r < fw.seg.y;  // (rows past T * G fold no head)
        lim_v = 0x7fffffff;
        if constexpr (kCausal) {
          const int pos = r + u.pos_shift;
          lim_v = pos < 0 ? 0 : (pos / p.causal_block + 1) * p.causal_block;
        }
        const int64_t li = lhead + fw.seg.x + r;
        const float l = rvalid && lim_v > 0 ? __ldg(p.lse + li) : -CUDART_INF_F;
        xl_v = l > -CUDART_INF_F ? l * kLog2e : CUDART_INF_F;  // +inf: P = 0
        xd_v = rvalid ? __ldg(p.dvec + li) : 0.0f;
      };
      float nxl = 0.0f, nxd = 0.0f;
      int nlim = 0;
      if (tid < 64 && nqt > 0) fetch(nxl, nxd, nlim);
      for (int i = 0; i < nqt; ++i) {
        const int par = tiles & 1;
        ++tiles;
        if (tid < 64) {
          ctrl.xl[par][lrow] = nxl;
          ctrl.xd[par][lrow] = nxd;
          if constexpr (kCausal) ctrl.xlim[par][lrow] = nlim;
          if (i + 1 < nqt) {
            fw.next(T);
            fetch(nxl, nxd, nlim);
          }
        }
        const bool fine = __all_sync(0xffffffffu, wait_bar(&ctrl.s_full, sc & 1, abort_flag, p.error_flag));
        if (named_barrier_or(1 + wg, 128, !fine)) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
        // 16-lane TMEM shapes: each thread handles 4 keys (lanes) x 16 columns of its
        // half (8 per part), so it needs the LSE / D / limit of only 16 Q rows.
        const float* xl = &ctrl.xl[par][64 * wg];
        const float* xd = &ctrl.xd[par][64 * wg];
        const uint64_t c2 = f32x2(c, c);
        uint32_t sr[2][2][16];  // [part][lane half][register]
        {
          const uint32_t col = kColS + 64 * wg;
          tmem_ld16x256b_x4_quad_sync(tmem_addr(tmem, lane_base, col), sr[0][0], tmem_addr(tmem, lane_base + 16, col),
                                      sr[0][1], tmem_addr(tmem, lane_base, col + 32), sr[1][0],
                                      tmem_addr(tmem, lane_base + 16, col + 32), sr[1][1]);
        }
        // P^T = 2^(S^T c - lse2), kept as fp32 pairs in the same registers
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 l2 = *reinterpret_cast<const float2*>(xl + 32 * part + 8 * k + 2 * c4);
          const uint64_t nl2 = f32x2(-l2.x, -l2.y);
          int2 m2 = make_int2(0x7fffffff, 0x7fffffff);
          if constexpr (kCausal)
            m2 = *reinterpret_cast<const int2*>(&ctrl.xlim[par][64 * wg + 32 * part + 8 * k + 2 * c4]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ka = lane_base + 16 * h + g, kb = ka + 8;  // keys of registers 4k,4k+1 / 4k+2,4k+3
            const bool va = ka < u.keys, vb = kb < u.keys;
            const int pa = kCausal ? u.key_pos0 + ka : 0, pb = kCausal ? u.key_pos0 + kb : 0;
            uint32_t* sv = &sr[part][h][4 * k];
            float x0, x1, x2, x3;
            f32x2_split(ffma2(f32x2(__uint_as_float(sv[0]), __uint_as_float(sv[1])), c2, nl2), x0, x1);
            f32x2_split(ffma2(f32x2(__uint_as_float(sv[2]), __uint_as_float(sv[3])), c2, nl2), x2, x3);
            sv[0] = __float_as_uint(va && pa < m2.x ? ex2_approx(x0) : 0.0f);
            sv[1] = __float_as_uint(va && pa < m2.y ? ex2_approx(x1) : 0.0f);
            sv[2] = __float_as_uint(vb && pb < m2.x ? ex2_approx(x2) : 0.0f);
            sv[3] = __float_as_uint(vb && pb < m2.y ? ex2_approx(x3) : 0.0f);
          }
        }
        // P^T pairs over this half's first 32 columns of S^T (already read)
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pp[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t* pv = &sr[part][h][4 * k];
              pp[2 * k] = pack_bf16x2(__uint_as_float(pv[0]), __uint_as_float(pv[1]));
              pp[2 * k + 1] = pack_bf16x2(__uint_as_float(pv[2]), __uint_as_float(pv[3]));
            }
            tmem_st16x128b_x4(tmem_addr(tmem, lane_base + 16 * h, kColS + 64 * wg + 16 * part), pp);
          }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.p_full[wg]);  // dV += P^T dO may start
        ok = __all_sync(0xffffffffu, wait_bar(&ctrl.dp_full, sc & 1, abort_flag, p.error_flag));
        ++sc;
        if (named_barrier_or(1 + wg, 128, !ok)) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
        // dS^T = P^T (dP^T - D), as bf16 pairs over this half's first 32 columns of dP^T:
        // part p's pairs land on columns part 0 covers, each after part 0 is read
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          uint32_t dr[2][16];  // [lane half][register] of this part
          const uint32_t col = kColDP + 64 * wg + 32 * part;
          tmem_ld16x256b_x4_pair_sync(tmem_addr(tmem, lane_base, col), dr[0], tmem_addr(tmem, lane_base + 16, col),
                                      dr[1]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pd[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 d2 = *reinterpret_cast<const float2*>(xd + 32 * part + 8 * k + 2 * c4);
              const uint64_t nd2 = f32x2(-d2.x, -d2.y);
              const uint32_t* pv = &sr[part][h][4 * k];
              const uint32_t* dv4 = &dr[h][4 * k];
              const uint64_t p01 = f32x2(__uint_as_float(pv[0]), __uint_as_float(pv[1]));
              const uint64_t p23 = f32x2(__uint_as_float(pv[2]), __uint_as_float(pv[3]));
              float s0, s1, s2, s3;
              f32x2_split(ffma2(p01, fadd2(f32x2(__uint_as_float(dv4[0]), __uint_as_float(dv4[1])), nd2), 0ull),
                          s0, s1);
              f32x2_split(ffma2(p23, fadd2(f32x2(__uint_as_float(dv4[2]), __uint_as_float(dv4[3])), nd2), 0ull),
                          s2, s3);
              pd[2 * k] = pack_bf16x2(s0, s1);
              pd[2 * k + 1] = pack_bf16x2(s2, s3);
            }
            tmem_st16x128b_x4(tmem_addr(tmem, lane_base + 16 * h, kColDP + 64 * wg + 16 * part), pd);  // dS^T
          }
        }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.ds_full[wg]);  // dK += dS^T Q may start
      }
      if (!ok) break;
      {  // the warpgroup takes one decision (its next barrier needs all 128 threads)
        const bool fine = __all_sync(0xffffffffu, wait_bar(&ctrl.acc_full, ac & 1, abort_flag, p.error_flag));
        if (named_barrier_or(1 + wg, 128, !fine)) break;
      }
      ++ac;
      tcgen05_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t o[32];
        float x[32];
        tmem_ld32_sync(tmem_addr(tmem, lane_base, kColDV + (D / 2) * wg + ch * 32), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]);
        if (key_valid) store_row32<TOut>(dvrow + ch * 32, x);
        tmem_ld32_sync(tmem_addr(tmem, lane_base, kColDK + (D / 2) * wg + ch * 32), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * p.scale;
        if (key_valid) store_row32<TOut>(dkrow + ch * 32, x);
      }
    }
  }
  tcgen05_fence_before();
  __syncthreads();
  if (warp == 1) {
    tcgen05_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

template <int D, typename TQ, typename TKV, bool kCausal>
cudaError_t launch_bwd_impl(const BwdParams& p, const MergeUnit* units, int32_t num_units, const void* out,
                            const void* d_out, float* dvec, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mdo, int dq_grid, int kv_grid, int sms,
                            cudaStream_t stream) {
  if (num_units > 0) {
    gva_bwd_dvec_kernel<D><<<min(num_units, sms * 8), 256, 0, stream>>>(
        units, num_units, static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(d_out), dvec,
        p.total_q, p.num_heads_q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.num_items > 0) {
    auto kq = gva_bwd_dq_kernel<D, TQ, kCausal>;
    cudaError_t e = ensure_smem_limit<gva_bwd_dq_kernel<D, TQ, kCausal>>(BCfg<D>::kSmemDq);
    if (e != cudaSuccess) return e;
    kq<<<dq_grid, kBwdThreads, BCfg<D>::kSmemDq, stream>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.num_kv_units > 0) {
    auto kkv = gva_bwd_dkdv_kernel<D, TKV, kCausal>;
    cudaError_t e = ensure_smem_limit<gva_bwd_dkdv_kernel<D, TKV, kCausal>>(BCfg<D>::kSmemDkv);
    if (e != cudaSuccess) return e;
    kkv<<<kv_grid, kBwdThreads, BCfg<D>::kSmemDkv, stream>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, bool kCausal>
cudaError_t launch_bwd_dc(bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units, int32_t num_units,
                          const void* out, const void* d_out, float* dvec, const CUtensorMap& mq,
                          const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo, int dq_grid,
                          int kv_grid, int sms, cudaStream_t stream) {
  if (dq_f32) {
    return dkv_f32 ? launch_bwd_impl<D, float, float, kCausal>(p, units, num_units, out, d_out, dvec, mq, mk, mv, mdo,
                                                               dq_grid, kv_grid, sms, stream)
                   : launch_bwd_impl<D, float, __nv_bfloat16, kCausal>(p, units, num_units, out, d_out, dvec, mq, mk,
                                                                       mv, mdo, dq_grid, kv_grid, sms, stream);
  }
  return dkv_f32 ? launch_bwd_impl<D, __nv_bfloat16, float, kCausal>(p, units, num_units, out, d_out, dvec, mq, mk,
                                                                     mv, mdo, dq_grid, kv_grid, sms, stream)
                 : launch_bwd_impl<D, __nv_bfloat16, __nv_bfloat16, kCausal>(p, units, num_units, out, d_out, dvec,
                                                                             mq, mk, mv, mdo, dq_grid, kv_grid, sms, stream);
}

template <int D>
cudaError_t launch_bwd_d(bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units, int32_t num_units,
                         const void* out, const void* d_out, float* dvec, const CUtensorMap& mq,
                         const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo, int dq_grid,
                         int kv_grid, int sms, cudaStream_t stream) {
  if (p.causal_block > 0)
    return launch_bwd_dc<D, true>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, mq, mk, mv, mdo, dq_grid,
                                  kv_grid, sms, stream);
  return launch_bwd_dc<D, false>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, mq, mk, mv, mdo, dq_grid,
                                 kv_grid, sms, stream);
}

}  // namespace

cudaError_t launch_backward(int head_dim, bool dq_f32, bool dkv_f32, const BwdParams& p, const MergeUnit* units,
                            int32_t num_units, const void* out, const void* d_out, float* dvec,
                            const CUtensorMap& map_q, const CUtensorMap& map_k, const CUtensorMap& map_v,
                            const CUtensorMap& map_do, int dq_grid, int kv_grid, int sm_count, cudaStream_t stream) {
  if (head_dim == 128)
    return launch_bwd_d<128>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, map_q, map_k, map_v, map_do,
                             dq_grid, kv_grid, sm_count, stream);
  return launch_bwd_d<64>(dq_f32, dkv_f32, p, units, num_units, out, d_out, dvec, map_q, map_k, map_v, map_do,
                          dq_grid, kv_grid, sm_count, stream);
}

}  // namespace gva
