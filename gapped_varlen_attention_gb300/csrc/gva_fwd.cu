// Gapped variable-length attention forward, sm_103a.
//
// Computes, for every used query row of every segment and every query head, softmax
// attention over the segment's used keys, writing O and the natural-log LSE; rows past
// a segment's used length are not touched, and keyless segments get O = 0, LSE = -inf
// (cosmos-framework PR #302, "What"). Keys past the used length never enter the
// softmax (TensorRT-LLM issue #18687, "actual behavior": each attended zero key would
// add exp(0) = 1 to the denominator).
//
// Design (one persistent CTA per SM, 10 warps):
//   warp 0      TMA producer: the item's two Q tiles, then K and V blocks of 128 keys
//               into a ring of shared-memory stages (128-byte swizzle).
//   warp 1      TMEM allocator and MMA issuer (one thread): S_t = Q_t K^T into TMEM,
//               O_t += P_t V with P_t read from TMEM (tcgen05 "A from TMEM" form).
//   warps 2-5   softmax + epilogue of Q tile 0; warps 6-9 of Q tile 1. One thread owns
//               one tile row (= one TMEM lane): the row max comes with the row's TMEM
//               load (its max-reducing form) and the row sum is a register reduction,
//               with no shuffles or shared memory.
// A work item is (segment, KV head, 2 x 128 folded rows): the g = Hq/Hkv query heads
// of one KV head are folded into the tile's rows (128/g tokens x g heads), so each K/V
// block feeds 256 rows. Two tiles ping-pong: while the softmax warps of one tile work,
// the tensor core runs the other tile's PV and next QK^T.
//
// The epilogue of a full tile stages O in shared memory (128 bytes of every row at a
// time: 64 bf16 or 32 fp32 columns, in the 128-byte-swizzled layout a Q tile arrives in)
// and writes it with one TMA store per pass; each thread storing its own row would touch
// 32 lines per store instruction. Partial tiles store rows directly.
//
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [384,384+d).
// P_t (bf16, two per 32-bit column) overwrites the first 64 columns of S_t once S_t is
// in registers.
//
// The running max is kept in log2 units of the scaled logits. O is rescaled only when
// a row's max grows by more than 2^8 over the max its P values were computed with;
// the final O / l and LSE use the same max, so the result is exact up to rounding.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "gva_device_common.cuh"
#include "gva_internal.h"
#include "sm103_ptx.cuh"

namespace gva {
namespace {

constexpr int kThreads = 320;
constexpr int kWarpTma = 0;
constexpr int kWarpMma = 1;
constexpr int kFirstSoftmaxWarp = 2;
constexpr uint32_t kTmemCols = 512;
// TMEM column of S_t (and P_t) and of O_t.
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;                 // 128-byte rows per operand row
  static constexpr int kQBytes = kTileRows * D * 2;      // one Q tile
  static constexpr int kKVBytes = kBlockKeys * D * 2;    // one K or V block
  static constexpr int kQChunkBytes = kTileRows * 128;   // one 64-column chunk of a Q tile
  static constexpr int kKVChunkBytes = kBlockKeys * 128;
  // One ring of K/V slots, loaded in the order K_0, V_0, K_1, V_1, ... so the producer
  // runs two key blocks (five at d = 64) ahead of the tensor core.
  static constexpr int kSlots = D == 64 ? 10 : 4;
  static constexpr int kStageBytes = kTileRows * 128;   // 128 bytes of each row of a tile's O
  static constexpr int kSmem = kTilesPerItem * kQBytes + kSlots * kKVBytes + kTilesPerItem * kStageBytes;
  static constexpr int kSmemAlloc = kSmem + 1024;        // slack for 1024-byte alignment
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");
};

// Named barrier over the 128 threads of softmax warpgroup t (ids 1 and 2).
__device__ __forceinline__ void warpgroup_sync(int t) {
  if (t == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 2, 128;" ::: "memory");
}

// TMA store of a 3-D box from shared memory, and the bulk-group waits around it.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

struct Ctrl {
  uint64_t q_full, q_empty;
  uint64_t kv_full[10], kv_empty[10];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// kCausal: block-causal masking within each segment. Row token i of a segment sits at
// key position pos = i + used_k - used_q and sees keys j < (floor(pos / B) + 1) * B
// (B = p.causal_block); the plan gives each item only the key blocks its last row sees.
template <int D, typename TOut, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    gva_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                   const FwdParams p) {
  using C = Cfg<D>;
  constexpr uint32_t NS = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctrl ctrl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                          // 2 tiles
  uint8_t* sKV = sQ + kTilesPerItem * C::kQBytes;              // NS slots
  uint8_t* sStage = sKV + NS * C::kKVBytes;                    // O staging, one per tile

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctrl.abort;

  if (threadIdx.x == 0) {
    mbar_init(&ctrl.q_full, 1);
    mbar_init(&ctrl.q_empty, 1);
    for (uint32_t i = 0; i < NS; ++i) {
      mbar_init(&ctrl.kv_full[i], 1);
      mbar_init(&ctrl.kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctrl.s_full[t], 1);
      mbar_init(&ctrl.p_full[t], 128);
      mbar_init(&ctrl.o_full[t], 1);
    }
    mbar_init(&ctrl.mma_done, 1);
    ctrl.abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&ctrl.tmem_base, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  const int T = p.tokens_per_tile;
  const int G = p.group;
  // A folded Q tile fills T * G rows (T = floor(128 / G) tokens of G heads). When G does
  // not divide 128, the copies never write the last 128 - T * G rows: they are zeroed
  // once here, so those (never stored) rows compute on zeros.
  const int q_rows_filled = T * G;
  for (int x = threadIdx.x; x < kTilesPerItem * (kTileRows - q_rows_filled) * C::kChunks * 8; x += kThreads) {
    const int piece = x % 8, rest = x / 8;
    const int ch = rest % C::kChunks, rest2 = rest / C::kChunks;
    const int r = q_rows_filled + rest2 % (kTileRows - q_rows_filled), t = rest2 / (kTileRows - q_rows_filled);
    *reinterpret_cast<uint4*>(sQ + t * C::kQBytes + ch * C::kQChunkBytes + r * 128 + piece * 16) =
        make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  const uint32_t q_tile_bytes = static_cast<uint32_t>(q_rows_filled) * D * 2;  // bytes one tile's copies bring

  if (warp == kWarpTma) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      uint32_t q_it = 0, ld = 0;  // ld: loads issued into the K/V ring so far
      for (int round = 0;; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_items) break;
        const WorkItem it = load_item(p.items, idx);
        if (it.nblk == 0) continue;
        const int nblk = it.nblk;
        if (!wait_bar(&ctrl.q_empty, (q_it & 1) ^ 1, abort_flag, p.error_flag)) break;
        mbar_arrive_expect_tx(&ctrl.q_full, it.n_tiles * q_tile_bytes);
        for (int t = 0; t < it.n_tiles; ++t)
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_3d(sQ + t * C::kQBytes + ch * C::kQChunkBytes, &map_q, &ctrl.q_full, ch * 64,
                        it.q_row0 + t * T, it.head_kv * G);
        ++q_it;
        bool ok = true;
        for (int j = 0; j < nblk && ok; ++j) {
          const int key0 = load_block(p.blocks, it.blk0 + j).row0;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {  // K_j, then V_j
            const uint32_t sl = ld % NS;
            ok = wait_bar(&ctrl.kv_empty[sl], ((ld / NS) & 1) ^ 1, abort_flag, p.error_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&ctrl.kv_full[sl], C::kKVBytes);
            const CUtensorMap* map = kv == 0 ? &map_k : &map_v;
#pragma unroll
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_3d(sKV + sl * C::kKVBytes + ch * C::kKVChunkBytes, map, &ctrl.kv_full[sl], ch * 64, key0,
                          it.head_kv);
            ++ld;
          }
        }
        if (!ok) break;
      }
      // Drain: every copy this thread issued has landed before the CTA may exit.
      if (q_it > 0) drain_bar(&ctrl.q_full, (q_it - 1) & 1, p.error_flag);
      for (uint32_t i = (ld > NS ? ld - NS : 0); i < ld; ++i) drain_bar(&ctrl.kv_full[i % NS], (i / NS) & 1, p.error_flag);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors of the first buffer of each kind; the others are whole-buffer offsets
      // of the start-address field. A slot holds K (K-major operand) or V (MN-major).
      const uint64_t q_desc0 = make_smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t k_desc0 = make_smem_desc_sw128(smem_addr(sKV), 16, 1024);
      const uint64_t v_desc0 = make_smem_desc_sw128(smem_addr(sKV), C::kKVChunkBytes, 1024);
      const uint64_t q_desc[2] = {q_desc0, q_desc0 + (C::kQBytes >> 4)};
      auto k_desc = [&](uint32_t sl) { return k_desc0 + sl * (C::kKVBytes >> 4); };
      auto v_desc = [&](uint32_t sl) { return v_desc0 + sl * (C::kKVBytes >> 4); };
      uint32_t q_it = 0, blk = 0, pc0 = 0, pc1 = 0;  // blk: key blocks consumed so far
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round, blockIdx.x, gridDim.x);
        if (idx >= p.num_items) break;
        const WorkItem it = load_item(p.items, idx);
        if (it.nblk == 0) continue;
        const int nblk = it.nblk;
        const bool two = it.n_tiles == 2;
        ok = wait_bar(&ctrl.q_full, q_it & 1, abort_flag, p.error_flag);
        if (!ok) break;
        ++q_it;
        // K_j has ring sequence number 2 * (blk + j), V_j the next one.
        uint32_t kseq = 2 * blk;
        ok = wait_bar(&ctrl.kv_full[kseq % NS], (kseq / NS) & 1, abort_flag, p.error_flag);
        if (!ok) break;
        tcgen05_fence_after();
        issue_qk<D>(tmem + col_s(0), q_desc[0], k_desc(kseq % NS));
        umma_commit(&ctrl.s_full[0]);
        if (two) {
          issue_qk<D>(tmem + col_s(1), q_desc[1], k_desc(kseq % NS));
          umma_commit(&ctrl.s_full[1]);
        }
        umma_commit(&ctrl.kv_empty[kseq % NS]);
        if (nblk == 1) umma_commit(&ctrl.q_empty);
        for (int j = 0; j < nblk; ++j) {
          const bool more = j + 1 < nblk;
          const uint32_t vseq = 2 * (blk + j) + 1;
          kseq = vseq + 1;  // K_{j+1}
          ok = wait_bar(&ctrl.kv_full[vseq % NS], (vseq / NS) & 1, abort_flag, p.error_flag);
          if (ok) ok = wait_bar(&ctrl.p_full[0], pc0 & 1, abort_flag, p.error_flag);
          if (!ok) break;
          ++pc0;
          tcgen05_fence_after();
          issue_pv<D>(tmem + col_o(0), tmem + col_s(0), v_desc(vseq % NS), j > 0);
          if (!more) umma_commit(&ctrl.o_full[0]);
          if (more) {
            ok = wait_bar(&ctrl.kv_full[kseq % NS], (kseq / NS) & 1, abort_flag, p.error_flag);
            if (!ok) break;
            tcgen05_fence_after();
            issue_qk<D>(tmem + col_s(0), q_desc[0], k_desc(kseq % NS));
            umma_commit(&ctrl.s_full[0]);
          }
          if (two) {
            ok = wait_bar(&ctrl.p_full[1], pc1 & 1, abort_flag, p.error_flag);
            if (!ok) break;
            ++pc1;
            tcgen05_fence_after();
            issue_pv<D>(tmem + col_o(1), tmem + col_s(1), v_desc(vseq % NS), j > 0);
            if (!more) umma_commit(&ctrl.o_full[1]);
            if (more) {
              issue_qk<D>(tmem + col_s(1), q_desc[1], k_desc(kseq % NS));
              umma_commit(&ctrl.s_full[1]);
            }
          }
          umma_commit(&ctrl.kv_empty[vseq % NS]);
          if (more) {
            umma_commit(&ctrl.kv_empty[kseq % NS]);
            if (j + 2 == nblk) umma_commit(&ctrl.q_empty);
          }
        }
        blk += nblk;
      }
      // Every MMA issued so far completes before TMEM is released.
      umma_commit(&ctrl.mma_done);
      drain_bar(&ctrl.mma_done, 0, p.error_flag);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int t = (warp - kFirstSoftmaxWarp) >> 2;      // Q tile of this warpgroup
    const int lane_base = (warp & 3) * 32;              // TMEM lane quarter of this warp
    const int row = lane_base + lane;                   // tile row = TMEM lane
    const int hl = row / T;                             // folded head within the KV group
    const int tok = row - hl * T;                       // token within the tile
    const uint32_t s_addr = tmem_addr(tmem, lane_base, col_s(t));
    const uint32_t o_addr = tmem_addr(tmem, lane_base, col_o(t));
    const float c = p.scale_log2;
    TOut* out = reinterpret_cast<TOut*>(p.out);
    constexpr bool kBf16Out = sizeof(TOut) == 2;
    const bool store_issuer = warp == kFirstSoftmaxWarp + 4 * t && lane == 0;  // TMA stores of tile t
    uint32_t sc = 0, oc = 0, vb = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round, blockIdx.x, gridDim.x);
      if (idx >= p.num_items) break;
      const WorkItem it = load_item(p.items, idx);
      // the next round's item is pulled into L1 now, so its load does not sit between
      // this item's epilogue and the next item's softmax
      const int idx_next = item_index(round + 1, blockIdx.x, gridDim.x);
      if (idx_next < p.num_items) prefetch_l1(p.items + idx_next);
      if (it.n_tiles <= t) continue;
      const bool valid = hl < G && tok < it.q_rows - t * T;
      const int64_t token = static_cast<int64_t>(it.q_row0) + t * T + tok;
      const int head = it.head_kv * G + hl;
      TOut* orow = out + (token * p.num_heads_q + head) * D;
      float* lrow = p.lse + static_cast<int64_t>(head) * p.total_q + token;
      if (it.nblk == 0) {
        if (valid) {
          float z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            if (p.out_wide) store_row32_wide<TOut>(orow + ch * 32, z);
            else store_row32<TOut>(orow + ch * 32, z);
          }
          *lrow = -CUDART_INF_F;
        }
        continue;
      }
      const int nblk = it.nblk;
      int row_limit = 0;  // block-causal: keys of the segment this row sees
      if constexpr (kCausal) {
        const int pos = it.q_pos0 + t * T + tok;
        const int bc = p.causal_block;
        row_limit = pos < 0 ? 0 : min(it.k_len, (pos / bc + 1) * bc);
      }
      const int row_keys = kCausal ? row_limit : it.k_len;
      float m_used = -CUDART_INF_F;
      // Row sums of the unrounded P (for the LSE) and of the bf16-rounded P that the PV
      // product multiplies (for O). When a row's weight sits on a handful of keys, each
      // key's rounding stays in O unless O is divided by the rounded sum (then its
      // weights sum to one). A warp with a row that sees at most one block of keys sums
      // both (uniform over the warp); other warps divide by l, which adds at most 2^-9
      // |O| and averages over their keys.
      float l = 0.0f, lp = 0.0f;
      const bool few_keys = __any_sync(0xffffffffu, row_keys <= kBlockKeys);
      // used keys of each block (>= 1), fetched one block ahead so the load's latency
      // hides behind the wait for the scores
      int rem_next = load_block(p.blocks, it.blk0).valid;
      for (int j = 0; j < nblk; ++j) {
        const int rem = rem_next;
        if (j + 1 < nblk) rem_next = load_block(p.blocks, it.blk0 + j + 1).valid;
        ok = __all_sync(0xffffffffu, wait_bar(&ctrl.s_full[t], sc & 1, abort_flag, p.error_flag));
        if (!ok) break;
        ++sc;
        tcgen05_fence_after();
        if (rem < kBlockKeys) {
          // Last, partial block: keys past the used length (gap, padding or another
          // segment, possibly NaN) leave the softmax. Their score columns are set to
          // -inf in TMEM before the row is read (the range is uniform over the warp).
          for (int col = rem; col < kBlockKeys; ++col) tmem_st1(s_addr + col, 0xff800000u);
          tmem_wait_st();
        }
        float s[128];
        float mx;  // the row's largest score in this block: the load returns it
        {
          uint32_t raw[128];
          mx = tmem_ld128_max_sync(s_addr, raw);
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(raw[i]);
        }
        if constexpr (kCausal) {
          // Diagonal blocks: keys at or past the row's limit leave the softmax (the
          // limit differs per row, so this is done on the registers, and the max taken
          // again over what is left).
          const int lim = row_limit - j * kBlockKeys;
          if (__any_sync(0xffffffffu, lim < kBlockKeys)) {
#pragma unroll
            for (int i = 0; i < 128; ++i) s[i] = (i < lim) ? s[i] : -CUDART_INF_F;
            float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
            float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
            for (int i = 12; i < 124; i += 8) {
              mx0 = fmax3(mx0, s[i], s[i + 1]);
              mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
              mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
              mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
            }
            mx = fmax3(fmax3(mx0, mx1, s[124]), fmax3(mx2, mx3, s[125]), fmaxf(s[126], s[127]));
          }
        }
        const float m_new = fmaxf(m_used, mx * c);
        // O is rescaled when the row max grows by more than the threshold; the O update
        // itself comes after P is stored, when fewer registers are live.
        float f_resc = 1.0f;
        bool resc = false;
        if (j == 0) {
          m_used = m_new;
        } else if (__any_sync(0xffffffffu, m_new > m_used + kRescaleThreshold)) {
          resc = true;
          f_resc = ex2_approx(m_used - m_new);
          l *= f_resc;
          lp *= f_resc;
          m_used = m_new;
        }
        // P = 2^(s*c - m) as bf16 pairs (column i holds keys 2i, 2i+1), stored to the
        // first 64 columns of S_t in 16-column pieces as they are ready.
        const uint64_t c2 = f32x2(c, c);
        // A row that has seen no key yet (block-causal only) has m = -inf and all P = 0.
        const float m_ref = (kCausal && m_used == -CUDART_INF_F) ? 0.0f : m_used;
        const uint64_t neg_m2 = f32x2(-m_ref, -m_ref);
        uint64_t acc0 = f32x2(0.0f, 0.0f), acc1 = acc0;
        if (!few_keys) {
#pragma unroll
          for (int q16 = 0; q16 < 4; ++q16) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k2 = q16 * 32 + 2 * i;
              float a, b;
              f32x2_split(ffma2(f32x2(s[k2], s[k2 + 1]), c2, neg_m2), a, b);
              a = ex2_approx(a);
              b = ex2_approx(b);
              pk[i] = pack_bf16x2(a, b);
              if (i & 1) acc1 = fadd2(acc1, f32x2(a, b));
              else acc0 = fadd2(acc0, f32x2(a, b));
            }
            tmem_st16(s_addr + q16 * 16, pk);
          }
        } else {
          float r0 = 0.0f, r1 = 0.0f;
#pragma unroll
          for (int q16 = 0; q16 < 4; ++q16) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k2 = q16 * 32 + 2 * i;
              float a, b;
              f32x2_split(ffma2(f32x2(s[k2], s[k2 + 1]), c2, neg_m2), a, b);
              a = ex2_approx(a);
              b = ex2_approx(b);
              pk[i] = pack_bf16x2(a, b);
              // the two rounded values as fp32: the low one moves up 16 bits, the high
              // one is already in place
              r0 += __uint_as_float(pk[i] << 16);
              r1 += __uint_as_float(pk[i] & 0xFFFF0000u);
              if (i & 1) acc1 = fadd2(acc1, f32x2(a, b));
              else acc0 = fadd2(acc0, f32x2(a, b));
            }
            tmem_st16(s_addr + q16 * 16, pk);
          }
          lp += r0 + r1;
        }
        {
          float la, lb;
          f32x2_split(fadd2(acc0, acc1), la, lb);
          l += la + lb;
        }
        if (resc) {
          // Complete: the S MMA just waited for was issued after this tile's previous PV.
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32_sync(o_addr + ch * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f_resc);
            tmem_st32(o_addr + ch * 32, o);
          }
        }
        if (t == 0 && rem < kBlockKeys) {
          // Keys past the used length in this V block (gap, padding or another
          // segment) get P = 0, but 0 * NaN would still poison O: zero those rows of
          // the staged V block before the PV MMA reads it.
          const uint32_t vseq = 2 * (vb + j) + 1;  // ring sequence number of V_j
          ok = __all_sync(0xffffffffu,
                          wait_bar(&ctrl.kv_full[vseq % NS], (vseq / NS) & 1, abort_flag, p.error_flag));
          if (!ok) break;
          uint8_t* vbase = sKV + (vseq % NS) * C::kKVBytes;
          const int n16 = (kBlockKeys - rem) * C::kChunks * 8;  // 16-byte pieces to clear
          for (int i = row; i < n16; i += 128) {
            const int r = rem + i / (C::kChunks * 8);
            const int rest = i % (C::kChunks * 8);
            *reinterpret_cast<uint4*>(vbase + (rest / 8) * C::kKVChunkBytes + r * 128 + (rest % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tcgen05_fence_before();
        mbar_arrive(&ctrl.p_full[t]);
      }
      if (!ok) break;
      if (t == 0) vb += nblk;
      ok = __all_sync(0xffffffffu, wait_bar(&ctrl.o_full[t], oc & 1, abort_flag, p.error_flag));
      if (!ok) break;
      ++oc;
      tcgen05_fence_after();
      // l > 0 for every row with a key; a block-causal row that sees none gets 0 / -inf.
      const float inv_l = l > 0.0f ? 1.0f / (few_keys ? lp : l) : 0.0f;
      const float lse_val = l > 0.0f ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
      if (p.out_tma && it.q_rows - t * T >= T) {
        // a full tile: every one of its T * G rows is a used row of the segment. Each
        // pass stages 128 bytes of every row: 64 bf16 or 32 fp32 columns.
        constexpr int kCols = kBf16Out ? 64 : 32;
        uint8_t* stage = sStage + t * C::kStageBytes;
#pragma unroll
        for (int ch = 0; ch < D / kCols; ++ch) {
          warpgroup_sync(t);  // the previous store has finished reading the staging buffer
#pragma unroll
          for (int h = 0; h < kCols / 32; ++h) {  // 32 columns per TMEM load
            uint32_t o[32];
            tmem_ld32_sync(o_addr + ch * kCols + h * 32, o);
            constexpr int kPieces = kBf16Out ? 4 : 8;  // 16-byte pieces these columns fill
#pragma unroll
            for (int i = 0; i < kPieces; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if constexpr (kBf16Out)
                  w[k] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * k]) * inv_l,
                                     __uint_as_float(o[8 * i + 2 * k + 1]) * inv_l);
                else
                  w[k] = __float_as_uint(__uint_as_float(o[4 * i + k]) * inv_l);
              }
              *reinterpret_cast<uint4*>(stage + row * 128 + (((h * kPieces + i) ^ (row & 7)) << 4)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          fence_proxy_async_smem();
          warpgroup_sync(t);
          if (store_issuer) {
            tma_store_3d(&map_o, stage, ch * kCols, it.q_row0 + t * T, it.head_kv * G);
            bulk_wait_read();
          }
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32_sync(o_addr + ch * 32, o);
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * inv_l;
          if (valid) {
            if (p.out_wide) store_row32_wide<TOut>(orow + ch * 32, x);
            else store_row32<TOut>(orow + ch * 32, x);
          }
        }
      }
      if (valid) *lrow = lse_val;
    }
    tmem_wait_st();
    if (store_issuer) bulk_wait_all();  // this CTA's TMA stores are complete before it exits
  }

  tcgen05_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tcgen05_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, typename TOut, bool kCausal>
cudaError_t launch_impl(const FwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mo, int grid, cudaStream_t stream) {
  auto kern = gva_fwd_kernel<D, TOut, kCausal>;
  cudaError_t e = ensure_smem_limit<gva_fwd_kernel<D, TOut, kCausal>>(Cfg<D>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Cfg<D>::kSmemAlloc, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

int forward_smem_bytes(int head_dim) {
  return head_dim == 64 ? Cfg<64>::kSmemAlloc : Cfg<128>::kSmemAlloc;
}

cudaError_t launch_forward(int head_dim, bool out_f32, const FwdParams& p, const CUtensorMap& map_q,
                           const CUtensorMap& map_k, const CUtensorMap& map_v, const CUtensorMap& map_o, int grid,
                           cudaStream_t stream) {
  const bool causal = p.causal_block > 0;
  if (head_dim == 128) {
    if (causal)
      return out_f32 ? launch_impl<128, float, true>(p, map_q, map_k, map_v, map_o, grid, stream)
                     : launch_impl<128, __nv_bfloat16, true>(p, map_q, map_k, map_v, map_o, grid, stream);
    return out_f32 ? launch_impl<128, float, false>(p, map_q, map_k, map_v, map_o, grid, stream)
                   : launch_impl<128, __nv_bfloat16, false>(p, map_q, map_k, map_v, map_o, grid, stream);
  }
  if (causal)
    return out_f32 ? launch_impl<64, float, true>(p, map_q, map_k, map_v, map_o, grid, stream)
                   : launch_impl<64, __nv_bfloat16, true>(p, map_q, map_k, map_v, map_o, grid, stream);
  return out_f32 ? launch_impl<64, float, false>(p, map_q, map_k, map_v, map_o, grid, stream)
                 : launch_impl<64, __nv_bfloat16, false>(p, map_q, map_k, map_v, map_o, grid, stream);
}

}  // namespace gva
