// C ABI of the gapped varlen attention library: plan construction on the host, tensor
// maps, launches, status reporting. See include/gva.h for the contract.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <string>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "gva.h"
#include "gva_internal.h"

// The tensor maps of the last call, keyed by the tensors' addresses: a plan is normally
// called again and again on the same buffers, and encoding three or four maps costs
// host time on every call of a short launch.
struct MapCache {
  const void* ptr[4] = {nullptr, nullptr, nullptr, nullptr};
  int out_dtype = -1;  // the forward's output map (ptr[3]) depends on its dtype too
  CUtensorMap map[4];
  bool valid = false;
};

struct gva_plan {
  int device = -1;
  int sm_count = 0;
  int32_t num_segments = 0, num_heads_q = 0, num_heads_kv = 0, head_dim = 0, group = 0, causal_block = 0;
  int64_t total_q = 0, total_k = 0;
  int32_t num_items = 0, num_units = 0, grid = 0;
  int32_t num_item_slots = 0;  // entries of d_items: each CTA's items in the kernels' walk, padded
  double used_flops = 0.0;
  gva::WorkItem* d_items = nullptr;
  gva::KeyBlock* d_blocks = nullptr;
  gva::MergeUnit* d_units = nullptr;
  int* d_error = nullptr;
  // backward work: one Q tile per dQ item; one piece of at most 128 K/V rows of one KV
  // head per dK / dV unit, with the segments that attend it
  int32_t num_bwd_items = 0, num_kv_units = 0, bwd_grid = 0, kv_grid = 0;
  gva::WorkItem* d_bwd_items = nullptr;
  gva::KvUnit* d_kv_units = nullptr;
  gva::SegRef* d_kv_segs = nullptr;
  std::mutex map_mutex;  // calls on one plan may come from several host threads
  MapCache fwd_maps, bwd_maps;
};

namespace {

thread_local std::string g_last_error;

gva_status fail(gva_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gva_status ok() {
  g_last_error.clear();
  return GVA_OK;
}

gva_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GVA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
  }
  return fn;
}

// A 3-D tensor map over a packed [rows, heads, d] tensor (bf16, or fp32 with `f32`),
// viewed as (d, rows, heads) so that a box of (128 bytes of d, box_rows, box_heads)
// lands in shared memory head-major: smem row = head_in_box * box_rows + row_in_box, 128
// bytes per row.
gva_status make_map(CUtensorMap* map, const void* base, int64_t rows, int32_t heads, int32_t d, uint32_t box_rows,
                    uint32_t box_heads, const char* name, bool f32 = false) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return fail(GVA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(heads) * d * es, static_cast<cuuint64_t>(d) * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), box_rows, box_heads};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, elem,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GVA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return GVA_OK;
}

gva_status validate_offsets(const int32_t* cu, const int32_t* used, int32_t n, const char* name) {
  if (cu[0] < 0) return fail(GVA_ERR_INVALID_ARG, "cu_seqlens_%s[0] = %d is negative", name, cu[0]);
  for (int32_t b = 0; b < n; ++b) {
    if (cu[b + 1] < cu[b])
      return fail(GVA_ERR_INVALID_ARG, "cu_seqlens_%s decreases at segment %d (%d -> %d)", name, b, cu[b], cu[b + 1]);
    const int32_t cap = cu[b + 1] - cu[b];
    if (used[b] < 0 || used[b] > cap)
      return fail(GVA_ERR_INVALID_ARG, "seqused_%s[%d] = %d outside [0, capacity %d]", name, b, used[b], cap);
  }
  return GVA_OK;
}

void free_plan(struct gva_plan* p) {
  if (p == nullptr) return;
  if (p->d_items) cudaFree(p->d_items);
  if (p->d_blocks) cudaFree(p->d_blocks);
  if (p->d_units) cudaFree(p->d_units);
  if (p->d_error) cudaFree(p->d_error);
  if (p->d_bwd_items) cudaFree(p->d_bwd_items);
  if (p->d_kv_units) cudaFree(p->d_kv_units);
  if (p->d_kv_segs) cudaFree(p->d_kv_segs);
  delete p;
}

// Estimated run time of a forward item, in key blocks of a two-tile item. Measured per
// item: 1.6 us per key block with two Q tiles, 1.38 us with one (its serial chain of
// scores, softmax and PV is not hidden behind another tile's), and about 3 us for its
// first copies and its epilogue.
double item_cost(const gva::WorkItem& it) {
  return 1.9 + (it.n_tiles == 2 ? 1.0 : 0.86) * it.nblk;
}

// Backward work: a dQ item is one Q tile over its key blocks (three products per
// block), a dK / dV unit one key block over its Q tiles (four per tile); each also pays
// a fixed cost of about two blocks or tiles.
double dq_item_cost(const gva::WorkItem& it) { return 2.0 + it.nblk; }
double kv_unit_cost(const gva::KvUnit& u) { return 2.0 + u.n_tiles; }

// A work list as the kernels walk it: CTA c reads entry item_index(r, c, grid) in round r.
// Work (sorted longest first, with estimated costs `cost`) is assigned to CTAs longest
// first, each to the CTA with the least estimated work, and then single moves or swaps
// between the most and the least loaded CTA are applied while they lower the larger of
// the two. Returns, per entry, the index of its work in the sorted list, or -1 for
// padding past the end of a CTA's list.
std::vector<int32_t> balanced_walk(const std::vector<double>& cost, int grid) {
  std::vector<int32_t> walk;
  if (cost.empty() || grid <= 0) return walk;
  std::vector<std::vector<int32_t>> lists(grid);
  std::vector<double> load(grid, 0.0);
  using Load = std::pair<double, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0.0, c});
  for (size_t i = 0; i < cost.size(); ++i) {
    const Load top = heap.top();
    heap.pop();
    lists[top.second].push_back(static_cast<int32_t>(i));
    load[top.second] = top.first + cost[i];
    heap.push({load[top.second], top.second});
  }
  // Each pass costs O(n log n) in the two lists' lengths: the best swap partner of an
  // item of the most loaded CTA is found by binary search in the least loaded CTA's
  // costs (the best exchange moves half the load gap).
  std::vector<std::pair<double, int32_t>> lo_costs;
  for (int iter = 0; iter < 4 * grid + 1000; ++iter) {
    const int hi = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    const int lo = static_cast<int>(std::min_element(load.begin(), load.end()) - load.begin());
    const double gap = load[hi] - load[lo];
    double best = load[hi] - 1e-9;
    int bi = -1, bj = -1;  // bj < 0: move item bi of hi to lo; else swap it with item bj of lo
    lo_costs.clear();
    for (size_t b = 0; b < lists[lo].size(); ++b) lo_costs.push_back({cost[lists[lo][b]], static_cast<int32_t>(b)});
    std::sort(lo_costs.begin(), lo_costs.end());
    for (size_t a = 0; a < lists[hi].size(); ++a) {
      const double ca = cost[lists[hi][a]];
      if (std::max(load[hi] - ca, load[lo] + ca) < best) {
        best = std::max(load[hi] - ca, load[lo] + ca);
        bi = static_cast<int>(a);
        bj = -1;
      }
      // swap partners: costs just below and just above ca - gap / 2
      const auto it = std::lower_bound(lo_costs.begin(), lo_costs.end(), std::make_pair(ca - 0.5 * gap, -1));
      for (auto c = (it == lo_costs.begin() ? it : it - 1); c != lo_costs.end() && c <= it; ++c) {
        const double d = ca - c->first;
        if (d > 0.0 && std::max(load[hi] - d, load[lo] + d) < best) {
          best = std::max(load[hi] - d, load[lo] + d);
          bi = static_cast<int>(a);
          bj = c->second;
        }
      }
    }
    // stop when no exchange helps, or when the best one gains under 0.01 % of the
    // largest load (long lists balance within that long before the pass limit)
    if (bi < 0 || load[hi] - best < 1e-4 * load[hi]) break;
    const int32_t a = lists[hi][bi];
    lists[hi].erase(lists[hi].begin() + bi);
    double d = cost[a];
    if (bj >= 0) {
      const int32_t b = lists[lo][bj];
      lists[lo].erase(lists[lo].begin() + bj);
      lists[hi].push_back(b);
      d -= cost[b];
    }
    lists[lo].push_back(a);
    load[hi] -= d;
    load[lo] += d;
  }
  size_t rounds = 0;
  for (auto& l : lists) {
    std::sort(l.begin(), l.end());  // the sorted list's order: longest first
    rounds = std::max(rounds, l.size());
  }
  walk.assign(rounds * grid, -1);
  for (int c = 0; c < grid; ++c)
    for (size_t r = 0; r < lists[c].size(); ++r) walk[gva::item_index(static_cast<int>(r), c, grid)] = lists[c][r];
  return walk;
}

// The work laid out along balanced_walk; padding entries are value-initialised (no
// tiles, no key blocks, no keys), which every role of the forward, dQ and dK / dV
// kernels skips.
template <typename T, typename Cost>
std::vector<T> balanced_layout(const std::vector<T>& sorted, int grid, Cost cost_of) {
  std::vector<double> cost(sorted.size());
  for (size_t i = 0; i < sorted.size(); ++i) cost[i] = cost_of(sorted[i]);
  const std::vector<int32_t> walk = balanced_walk(cost, grid);
  std::vector<T> laid(walk.size(), T{});
  for (size_t e = 0; e < walk.size(); ++e)
    if (walk[e] >= 0) laid[e] = sorted[walk[e]];
  return laid;
}

// Units of the LSE merge (and of the backward's D = rowsum(dO * O) kernel): runs of at
// most kMergeRows used rows of one segment. When 16-row units overflow one wave of the
// merge's resident CTAs (about four per SM), the last wave can hold only a few units,
// which then run on an otherwise idle GPU; the rows per unit are then chosen so that the
// units fill the waves they need (each segment's last unit may be shorter: one unit of
// slack per segment). Units that fit one wave keep 16 rows: smaller ones only add
// per-unit work.
void build_merge_units(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                       int32_t resident, std::vector<gva::MergeUnit>& units) {
  int64_t total = 0, n16 = 0;
  for (int32_t b = 0; b < num_segments; ++b) {
    total += seqused_q[b];
    n16 += (seqused_q[b] + gva::kMergeRows - 1) / gva::kMergeRows;
  }
  int32_t rows = gva::kMergeRows;
  if (resident > 0 && n16 > resident) {
    const int64_t waves = (n16 + resident - 1) / resident;
    const int64_t slots = waves * resident - num_segments;
    if (slots >= resident / 2)
      rows = static_cast<int32_t>(std::min<int64_t>(gva::kMergeRows, std::max<int64_t>(1, (total + slots - 1) / slots)));
  }
  units.clear();
  for (int32_t b = 0; b < num_segments; ++b)
    for (int32_t r0 = 0; r0 < seqused_q[b]; r0 += rows)
      units.push_back({cu_seqlens_q[b] + r0, std::min(rows, seqused_q[b] - r0)});
}

// Merge CTAs resident at once per SM, as the merge launches them for its usual shapes.
constexpr int32_t kMergeCtasPerSm = 4;

// Shared by gva_plan and gva_plan_ranges once the arguments are validated: segment b's
// keys are the ranges range_off[b] .. range_off[b+1] of (range_start, range_len).
// causal_block > 0 (block-causal, one prefix range per segment): each item only gets the
// key blocks its last row sees, and FLOPs count the visible keys of every row.
// backward: also build the dQ items and the dK / dV units (every plan kind).
struct HostWork {
  std::vector<gva::KeyBlock> blocks;
  std::vector<gva::WorkItem> items;  // forward, sorted longest first
  std::vector<gva::MergeUnit> units;
  std::vector<gva::WorkItem> bwd_items;
  std::vector<gva::KvUnit> kv_units;
  std::vector<gva::SegRef> kv_segs;
  double flops = 0.0;
};

gva_status build_work(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                      const int32_t* range_off, const int32_t* range_start, const int32_t* range_len,
                      int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t causal_block,
                      bool backward, HostWork& w) {
  const int32_t group = num_heads_q / num_heads_kv;
  // ---- key blocks: each range cut into blocks of at most kBlockKeys keys
  std::vector<gva::KeyBlock>& blocks = w.blocks;
  std::vector<int32_t> seg_blk0(num_segments), seg_nblk(num_segments), seg_keys(num_segments);
  for (int32_t b = 0; b < num_segments; ++b) {
    seg_blk0[b] = static_cast<int32_t>(blocks.size());
    int64_t keys = 0;
    for (int32_t r = range_off[b]; r < range_off[b + 1]; ++r) {
      for (int32_t o = 0; o < range_len[r]; o += gva::kBlockKeys)
        blocks.push_back({range_start[r] + o, std::min(gva::kBlockKeys, range_len[r] - o)});
      keys += range_len[r];
    }
    if (keys > INT32_MAX) return fail(GVA_ERR_INVALID_ARG, "segment %d has more than 2^31 keys", b);
    seg_nblk[b] = static_cast<int32_t>(blocks.size()) - seg_blk0[b];
    seg_keys[b] = static_cast<int32_t>(keys);
  }
  // ---- work list: (segment, KV head, 2 x 128 folded rows), keyless items epilogue-only
  const int32_t tokens_per_tile = gva::kTileRows / group;
  const int32_t tokens_per_item = tokens_per_tile * gva::kTilesPerItem;
  std::vector<gva::WorkItem> items;
  std::vector<double> cost;
  double& flops = w.flops;
  // keys visible to the row at key position pos (block-causal)
  auto limit_at = [&](int64_t pos, int32_t keys) -> int32_t {
    if (pos < 0) return 0;
    return static_cast<int32_t>(std::min<int64_t>(keys, (pos / causal_block + 1) * causal_block));
  };
  for (int32_t b = 0; b < num_segments; ++b) {
    const int32_t uq = seqused_q[b];
    const int32_t pos_shift = seg_keys[b] - uq;  // key position of row token 0
    if (causal_block > 0) {
      double pairs = 0.0;
      for (int32_t i = 0; i < uq; ++i) pairs += limit_at(static_cast<int64_t>(i) + pos_shift, seg_keys[b]);
      flops += 4.0 * head_dim * num_heads_q * pairs;
    } else {
      flops += 4.0 * head_dim * num_heads_q * static_cast<double>(uq) * static_cast<double>(seg_keys[b]);
    }
    for (int32_t hk = 0; hk < num_heads_kv; ++hk) {
      for (int32_t t0 = 0; t0 < uq; t0 += tokens_per_item) {
        gva::WorkItem it{};
        it.q_row0 = cu_seqlens_q[b] + t0;
        it.q_rows = std::min(tokens_per_item, uq - t0);
        it.blk0 = seg_blk0[b];
        it.nblk = seg_nblk[b];
        it.head_kv = hk;
        it.n_tiles = it.q_rows > tokens_per_tile ? 2 : 1;
        it.k_len = seg_keys[b];
        if (causal_block > 0) {
          it.q_pos0 = t0 + pos_shift;
          const int32_t last = limit_at(static_cast<int64_t>(it.q_pos0) + it.q_rows - 1, seg_keys[b]);
          it.nblk = (last + gva::kBlockKeys - 1) / gva::kBlockKeys;
        }
        items.push_back(it);
        cost.push_back(item_cost(it));
      }
    }
  }
  std::vector<int32_t> order(items.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = static_cast<int32_t>(i);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t c) { return cost[a] > cost[c]; });
  std::vector<gva::WorkItem>& sorted = w.items;
  sorted.resize(items.size());
  for (size_t i = 0; i < order.size(); ++i) sorted[i] = items[order[i]];

  // ---- backward work lists, longest first
  std::vector<gva::WorkItem>& bwd_items = w.bwd_items;
  std::vector<gva::KvUnit>& kv_units = w.kv_units;
  if (backward) {
    for (int32_t b = 0; b < num_segments; ++b) {
      const int32_t uq = seqused_q[b];
      const int32_t pos_shift = seg_keys[b] - uq;  // block-causal: key position of row 0
      for (int32_t hk = 0; hk < num_heads_kv; ++hk) {
        for (int32_t t0 = 0; t0 < uq; t0 += tokens_per_tile) {
          gva::WorkItem it{};
          it.q_row0 = cu_seqlens_q[b] + t0;
          it.q_rows = std::min(tokens_per_tile, uq - t0);
          it.blk0 = seg_blk0[b];
          it.nblk = seg_nblk[b];
          it.head_kv = hk;
          it.n_tiles = 1;
          it.k_len = seg_keys[b];
          if (causal_block > 0) {  // the key blocks the tile's last row sees
            it.q_pos0 = t0 + pos_shift;
            const int32_t last = limit_at(static_cast<int64_t>(it.q_pos0) + it.q_rows - 1, seg_keys[b]);
            it.nblk = (last + gva::kBlockKeys - 1) / gva::kBlockKeys;
          }
          bwd_items.push_back(it);
        }
      }
    }
    std::stable_sort(bwd_items.begin(), bwd_items.end(),
                     [](const gva::WorkItem& a, const gva::WorkItem& c) { return a.nblk > c.nblk; });

    // dK / dV units: pieces of at most kBlockKeys K/V rows, each with the segments that
    // attend them (SegRef runs shared by every KV head), so every K/V row has one unit
    // per KV head and a single writer.
    std::vector<gva::SegRef>& segs = w.kv_segs;
    struct Piece {
      int32_t row0, keys, seg0, n_tiles, tile0, key_pos0, pos_shift;
    };
    std::vector<Piece> pieces;
    auto tiles_of = [&](int32_t rows) { return (rows + tokens_per_tile - 1) / tokens_per_tile; };
    if (causal_block > 0) {
      // one prefix range per segment: its key blocks, each attended by that segment only,
      // from the first Q tile whose rows see the block's first key
      for (int32_t b = 0; b < num_segments; ++b) {
        const int32_t uq = seqused_q[b];
        const int32_t pos_shift = seg_keys[b] - uq;
        const int32_t seg0 = static_cast<int32_t>(segs.size());
        if (uq > 0) segs.push_back({cu_seqlens_q[b], uq});
        for (int32_t j = 0; j < seg_nblk[b]; ++j) {
          const gva::KeyBlock& kb = blocks[seg_blk0[b] + j];
          Piece pc{kb.row0, kb.valid, seg0, 0, 0, j * gva::kBlockKeys, pos_shift};
          if (uq > 0) {
            // rows at key positions >= the start of the frame holding the block's first
            // key see it; tiles before the first such row never do
            const int64_t pos_min = (static_cast<int64_t>(pc.key_pos0) / causal_block) * causal_block;
            const int64_t row_min = std::max<int64_t>(0, pos_min - pos_shift);
            pc.tile0 = static_cast<int32_t>(std::min<int64_t>(row_min / tokens_per_tile, tiles_of(uq)));
            pc.n_tiles = tiles_of(uq) - pc.tile0;
          }
          pieces.push_back(pc);
        }
      }
    } else {
      // The union of every segment's key ranges, cut wherever a range starts or ends:
      // within a piece the attending segments do not change. A segment with several
      // ranges over the same rows attends them that many times and is listed so.
      struct Edge {
        int64_t x;
        int32_t seg, delta;
      };
      std::vector<Edge> edges;
      for (int32_t b = 0; b < num_segments; ++b)
        for (int32_t r = range_off[b]; r < range_off[b + 1]; ++r)
          if (range_len[r] > 0) {
            edges.push_back({range_start[r], b, +1});
            edges.push_back({static_cast<int64_t>(range_start[r]) + range_len[r], b, -1});
          }
      std::sort(edges.begin(), edges.end(), [](const Edge& a, const Edge& c) { return a.x < c.x; });
      std::map<int32_t, int32_t> active;  // segment -> ranges of it covering the piece
      for (size_t e = 0; e < edges.size();) {
        const int64_t x = edges[e].x;
        for (; e < edges.size() && edges[e].x == x; ++e) {
          const int32_t m = (active[edges[e].seg] += edges[e].delta);
          if (m == 0) active.erase(edges[e].seg);
        }
        if (active.empty() || e == edges.size()) continue;
        const int64_t x1 = edges[e].x;  // the piece is rows [x, x1)
        const int32_t seg0 = static_cast<int32_t>(segs.size());
        int32_t n_tiles = 0;
        for (const auto& am : active) {
          const int32_t uq = seqused_q[am.first];
          if (uq == 0) continue;  // no rows: contributes nothing
          for (int32_t c = 0; c < am.second; ++c) {
            segs.push_back({cu_seqlens_q[am.first], uq});
            n_tiles += tiles_of(uq);
          }
        }
        for (int64_t o = x; o < x1; o += gva::kBlockKeys)
          pieces.push_back({static_cast<int32_t>(o), static_cast<int32_t>(std::min<int64_t>(gva::kBlockKeys, x1 - o)),
                            seg0, n_tiles, 0, 0, 0});
      }
    }
    for (int32_t hk = 0; hk < num_heads_kv; ++hk)
      for (const Piece& pc : pieces)
        kv_units.push_back({pc.row0, pc.keys, pc.seg0, pc.n_tiles, hk, pc.tile0, pc.key_pos0, pc.pos_shift});
    std::stable_sort(kv_units.begin(), kv_units.end(),
                     [](const gva::KvUnit& a, const gva::KvUnit& c) { return a.n_tiles > c.n_tiles; });
  }
  return GVA_OK;
}

gva_status build_plan(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                      const int32_t* range_off, const int32_t* range_start, const int32_t* range_len,
                      int64_t total_k, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                      int32_t causal_block, bool backward, gva_plan_t* out_plan) {
  HostWork w;
  gva_status st = build_work(cu_seqlens_q, seqused_q, num_segments, range_off, range_start, range_len,
                             num_heads_q, num_heads_kv, head_dim, causal_block, backward, w);
  if (st != GVA_OK) return st;
  const int32_t group = num_heads_q / num_heads_kv;
  const std::vector<gva::KeyBlock>& blocks = w.blocks;
  const std::vector<gva::WorkItem>& sorted = w.items;
  const std::vector<gva::WorkItem>& bwd_items = w.bwd_items;
  const std::vector<gva::KvUnit>& kv_units = w.kv_units;
  const std::vector<gva::SegRef>& kv_segs = w.kv_segs;
  const double flops = w.flops;

  // ---- device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GVA_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(GVA_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300); device %d is sm_%d%d", dev, major,
                minor);

  build_merge_units(cu_seqlens_q, seqused_q, num_segments, kMergeCtasPerSm * sms, w.units);
  const std::vector<gva::MergeUnit>& units = w.units;

  struct gva_plan* p = new struct gva_plan();
  p->device = dev;
  p->sm_count = sms;
  p->num_segments = num_segments;
  p->num_heads_q = num_heads_q;
  p->num_heads_kv = num_heads_kv;
  p->head_dim = head_dim;
  p->group = group;
  p->causal_block = causal_block;
  p->total_q = cu_seqlens_q[num_segments];
  p->total_k = total_k;
  p->num_items = static_cast<int32_t>(sorted.size());
  p->num_units = static_cast<int32_t>(units.size());
  p->grid = std::min(p->num_items, sms);
  p->used_flops = flops;
  const std::vector<gva::WorkItem> laid = balanced_layout(sorted, p->grid, item_cost);
  p->num_item_slots = static_cast<int32_t>(laid.size());
  if ((e = cudaMalloc(&p->d_error, sizeof(int))) != cudaSuccess || (e = cudaMemset(p->d_error, 0, sizeof(int))) != cudaSuccess) {
    free_plan(p);
    return cuda_fail(e, "allocating the plan's error word");
  }
  if (!laid.empty()) {
    if ((e = cudaMalloc(&p->d_items, laid.size() * sizeof(gva::WorkItem))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_items, laid.data(), laid.size() * sizeof(gva::WorkItem), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the work list");
    }
  }
  if (!blocks.empty()) {
    if ((e = cudaMalloc(&p->d_blocks, blocks.size() * sizeof(gva::KeyBlock))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_blocks, blocks.data(), blocks.size() * sizeof(gva::KeyBlock), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the key blocks");
    }
  }
  if (!units.empty()) {
    if ((e = cudaMalloc(&p->d_units, units.size() * sizeof(gva::MergeUnit))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_units, units.data(), units.size() * sizeof(gva::MergeUnit), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the merge units");
    }
  }
  // Both backward lists balanced like the forward's, each for the grid its launch takes.
  p->bwd_grid = std::min(static_cast<int32_t>(bwd_items.size()), sms);
  p->kv_grid = std::min(static_cast<int32_t>(kv_units.size()), sms);
  const std::vector<gva::WorkItem> bwd_laid = balanced_layout(bwd_items, p->bwd_grid, dq_item_cost);
  const std::vector<gva::KvUnit> kv_laid = balanced_layout(kv_units, p->kv_grid, kv_unit_cost);
  p->num_bwd_items = static_cast<int32_t>(bwd_laid.size());
  p->num_kv_units = static_cast<int32_t>(kv_laid.size());
  if (!bwd_laid.empty()) {
    if ((e = cudaMalloc(&p->d_bwd_items, bwd_laid.size() * sizeof(gva::WorkItem))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_bwd_items, bwd_laid.data(), bwd_laid.size() * sizeof(gva::WorkItem),
                        cudaMemcpyHostToDevice)) != cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the backward work list");
    }
  }
  if (!kv_laid.empty()) {
    if ((e = cudaMalloc(&p->d_kv_units, kv_laid.size() * sizeof(gva::KvUnit))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_kv_units, kv_laid.data(), kv_laid.size() * sizeof(gva::KvUnit),
                        cudaMemcpyHostToDevice)) != cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the dK / dV units");
    }
  }
  if (!kv_segs.empty()) {
    if ((e = cudaMalloc(&p->d_kv_segs, kv_segs.size() * sizeof(gva::SegRef))) != cudaSuccess ||
        (e = cudaMemcpy(p->d_kv_segs, kv_segs.data(), kv_segs.size() * sizeof(gva::SegRef),
                        cudaMemcpyHostToDevice)) != cudaSuccess) {
      free_plan(p);
      return cuda_fail(e, "uploading the dK / dV units' segments");
    }
  }
  *out_plan = p;
  return ok();
}

// Checks shared by both plan builders (before any CUDA call).
gva_status validate_common(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                           int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim) {
  if (num_segments < 0) return fail(GVA_ERR_INVALID_ARG, "num_segments = %d < 0", num_segments);
  if (cu_seqlens_q == nullptr || (num_segments > 0 && seqused_q == nullptr))
    return fail(GVA_ERR_INVALID_ARG, "a geometry array is NULL");
  if (num_heads_q <= 0 || num_heads_kv <= 0)
    return fail(GVA_ERR_INVALID_ARG, "head counts must be positive (Hq=%d, Hkv=%d)", num_heads_q, num_heads_kv);
  if (num_heads_q % num_heads_kv != 0)
    return fail(GVA_ERR_INVALID_ARG, "num_heads_q=%d is not divisible by num_heads_kv=%d", num_heads_q, num_heads_kv);
  const int32_t group = num_heads_q / num_heads_kv;
  // A Q tile folds floor(128 / group) tokens of the group's heads into its 128 rows.
  if (group > gva::kTileRows)
    return fail(GVA_ERR_UNSUPPORTED, "query heads per KV head (%d) must be at most %d", group, gva::kTileRows);
  if (head_dim != 64 && head_dim != 128)
    return fail(GVA_ERR_UNSUPPORTED, "head_dim=%d is not supported (64 or 128)", head_dim);
  if (num_heads_q > 256) return fail(GVA_ERR_UNSUPPORTED, "num_heads_q=%d is too large (at most 256)", num_heads_q);
  return validate_offsets(cu_seqlens_q, seqused_q, num_segments, "q");
}

// Key ranges of gva_plan_ranges: offsets start at 0 and do not decrease, every range lies
// in [0, total_k). Ranges may overlap, within a segment or across segments.
gva_status validate_ranges(int32_t num_segments, const int32_t* key_range_offsets, const int32_t* key_range_starts,
                           const int32_t* key_range_lengths, int64_t total_k) {
  if (key_range_offsets == nullptr) return fail(GVA_ERR_INVALID_ARG, "key_range_offsets is NULL");
  if (total_k < 0 || total_k > INT32_MAX) return fail(GVA_ERR_INVALID_ARG, "total_k=%lld is out of range", (long long)total_k);
  if (key_range_offsets[0] != 0) return fail(GVA_ERR_INVALID_ARG, "key_range_offsets[0] must be 0");
  for (int32_t b = 0; b < num_segments; ++b)
    if (key_range_offsets[b + 1] < key_range_offsets[b])
      return fail(GVA_ERR_INVALID_ARG, "key_range_offsets decreases at segment %d", b);
  const int32_t num_ranges = key_range_offsets[num_segments];
  if (num_ranges > 0 && (key_range_starts == nullptr || key_range_lengths == nullptr))
    return fail(GVA_ERR_INVALID_ARG, "key range arrays are NULL");
  for (int32_t r = 0; r < num_ranges; ++r) {
    const int64_t st = key_range_starts[r], n = key_range_lengths[r];
    if (st < 0 || n < 0 || st + n > total_k)
      return fail(GVA_ERR_INVALID_ARG, "key range %d = [%lld, %lld) is outside [0, total_k=%lld)", r, (long long)st,
                  (long long)(st + n), (long long)total_k);
  }
  return GVA_OK;
}
}  // namespace

namespace gva {
void set_last_error(const char* message) { g_last_error = message; }
}  // namespace gva

extern "C" {

gva_status gva_plan(const int32_t* cu_seqlens_q, const int32_t* seqused_q, const int32_t* cu_seqlens_k,
                    const int32_t* seqused_k, int32_t num_segments, int32_t num_heads_q, int32_t num_heads_kv,
                    int32_t head_dim, gva_plan_t* out_plan) {
  if (out_plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  // ---- host-only validation (no CUDA call before it passes)
  gva_status s = validate_common(cu_seqlens_q, seqused_q, num_segments, num_heads_q, num_heads_kv, head_dim);
  if (s != GVA_OK) return s;
  if (cu_seqlens_k == nullptr || (num_segments > 0 && seqused_k == nullptr))
    return fail(GVA_ERR_INVALID_ARG, "a geometry array is NULL");
  s = validate_offsets(cu_seqlens_k, seqused_k, num_segments, "k");
  if (s != GVA_OK) return s;
  // one key range per segment: its used prefix
  std::vector<int32_t> off(num_segments + 1), start(num_segments), len(num_segments);
  for (int32_t b = 0; b <= num_segments; ++b) off[b] = b;
  for (int32_t b = 0; b < num_segments; ++b) {
    start[b] = cu_seqlens_k[b];
    len[b] = seqused_k[b];
  }
  return build_plan(cu_seqlens_q, seqused_q, num_segments, off.data(), start.data(), len.data(),
                    cu_seqlens_k[num_segments], num_heads_q, num_heads_kv, head_dim, 0, true, out_plan);
}

gva_status gva_plan_causal(const int32_t* cu_seqlens_q, const int32_t* seqused_q, const int32_t* cu_seqlens_k,
                           const int32_t* seqused_k, int32_t num_segments, int32_t causal_block,
                           int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, gva_plan_t* out_plan) {
  if (out_plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  if (causal_block < 1) return fail(GVA_ERR_INVALID_ARG, "causal_block=%d must be >= 1", causal_block);
  gva_status s = validate_common(cu_seqlens_q, seqused_q, num_segments, num_heads_q, num_heads_kv, head_dim);
  if (s != GVA_OK) return s;
  if (cu_seqlens_k == nullptr || (num_segments > 0 && seqused_k == nullptr))
    return fail(GVA_ERR_INVALID_ARG, "a geometry array is NULL");
  s = validate_offsets(cu_seqlens_k, seqused_k, num_segments, "k");
  if (s != GVA_OK) return s;
  std::vector<int32_t> off(num_segments + 1), start(num_segments), len(num_segments);
  for (int32_t b = 0; b <= num_segments; ++b) off[b] = b;
  for (int32_t b = 0; b < num_segments; ++b) {
    start[b] = cu_seqlens_k[b];
    len[b] = seqused_k[b];
  }
  return build_plan(cu_seqlens_q, seqused_q, num_segments, off.data(), start.data(), len.data(),
                    cu_seqlens_k[num_segments], num_heads_q, num_heads_kv, head_dim, causal_block, true,
                    out_plan);
}

gva_status gva_plan_ranges(const int32_t* cu_seqlens_q, const int32_t* seqused_q, int32_t num_segments,
                           const int32_t* key_range_offsets, const int32_t* key_range_starts,
                           const int32_t* key_range_lengths, int64_t total_k, int32_t num_heads_q,
                           int32_t num_heads_kv, int32_t head_dim, gva_plan_t* out_plan) {
  if (out_plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  gva_status s = validate_common(cu_seqlens_q, seqused_q, num_segments, num_heads_q, num_heads_kv, head_dim);
  if (s != GVA_OK) return s;
  s = validate_ranges(num_segments, key_range_offsets, key_range_starts, key_range_lengths, total_k);
  if (s != GVA_OK) return s;
  return build_plan(cu_seqlens_q, seqused_q, num_segments, key_range_offsets, key_range_starts, key_range_lengths,
                    total_k, num_heads_q, num_heads_kv, head_dim, 0, true, out_plan);
}

gva_status gva_plan_inspect(const int32_t* cu_seqlens_q, const int32_t* seqused_q, const int32_t* cu_seqlens_k,
                            const int32_t* seqused_k, int32_t num_segments, const int32_t* key_range_offsets,
                            const int32_t* key_range_starts, const int32_t* key_range_lengths, int64_t total_k,
                            int32_t causal_block, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                            int32_t grid, int32_t walk_list, gva_work_summary* summary, int32_t* items,
                            int32_t items_capacity, int32_t* walk, int32_t walk_capacity, int32_t* bwd_items,
                            int32_t bwd_items_capacity, int32_t* kv_units, int32_t kv_units_capacity,
                            int32_t* kv_segs, int32_t kv_segs_capacity) {
  if (summary == nullptr) return fail(GVA_ERR_INVALID_ARG, "summary is NULL");
  if (causal_block < 0) return fail(GVA_ERR_INVALID_ARG, "causal_block=%d must be >= 0", causal_block);
  if (grid < 1) return fail(GVA_ERR_INVALID_ARG, "grid=%d must be >= 1", grid);
  if (walk_list < 0 || walk_list > 2) return fail(GVA_ERR_INVALID_ARG, "walk_list=%d is not 0, 1 or 2", walk_list);
  gva_status s = validate_common(cu_seqlens_q, seqused_q, num_segments, num_heads_q, num_heads_kv, head_dim);
  if (s != GVA_OK) return s;
  std::vector<int32_t> off, start, len;
  if (key_range_offsets != nullptr) {  // as gva_plan_ranges
    if (causal_block > 0) return fail(GVA_ERR_INVALID_ARG, "block-causal plans take prefix keys, not ranges");
    s = validate_ranges(num_segments, key_range_offsets, key_range_starts, key_range_lengths, total_k);
    if (s != GVA_OK) return s;
    const int32_t n = key_range_offsets[num_segments];
    off.assign(key_range_offsets, key_range_offsets + num_segments + 1);
    start.assign(key_range_starts, key_range_starts + n);
    len.assign(key_range_lengths, key_range_lengths + n);
  } else {  // as gva_plan / gva_plan_causal
    if (cu_seqlens_k == nullptr || (num_segments > 0 && seqused_k == nullptr))
      return fail(GVA_ERR_INVALID_ARG, "a geometry array is NULL");
    s = validate_offsets(cu_seqlens_k, seqused_k, num_segments, "k");
    if (s != GVA_OK) return s;
    off.resize(num_segments + 1);
    start.resize(num_segments);
    len.resize(num_segments);
    for (int32_t b = 0; b <= num_segments; ++b) off[b] = b;
    for (int32_t b = 0; b < num_segments; ++b) {
      start[b] = cu_seqlens_k[b];
      len[b] = seqused_k[b];
    }
  }
  HostWork w;
  s = build_work(cu_seqlens_q, seqused_q, num_segments, off.data(), start.data(), len.data(), num_heads_q,
                 num_heads_kv, head_dim, causal_block, true, w);
  if (s != GVA_OK) return s;
  summary->backward_ok = 1;
  // the chosen list as a grid of min(grid, its length) CTAs walks it
  std::vector<double> cost;
  if (walk_list == 0) {
    for (const auto& it : w.items) cost.push_back(item_cost(it));
  } else if (walk_list == 1) {
    for (const auto& it : w.bwd_items) cost.push_back(dq_item_cost(it));
  } else {
    for (const auto& u : w.kv_units) cost.push_back(kv_unit_cost(u));
  }
  const std::vector<int32_t> laid = balanced_walk(cost, std::min<int32_t>(grid, static_cast<int32_t>(cost.size())));
  summary->num_walk_entries = static_cast<int32_t>(laid.size());
  if (walk != nullptr && walk_capacity > 0)
    std::memcpy(walk, laid.data(), std::min<size_t>(laid.size(), walk_capacity) * sizeof(int32_t));
  summary->num_work_items = static_cast<int32_t>(w.items.size());
  summary->num_key_blocks = static_cast<int32_t>(w.blocks.size());
  build_merge_units(cu_seqlens_q, seqused_q, num_segments, kMergeCtasPerSm * grid, w.units);
  summary->num_merge_units = static_cast<int32_t>(w.units.size());
  summary->num_bwd_items = static_cast<int32_t>(w.bwd_items.size());
  summary->num_kv_units = static_cast<int32_t>(w.kv_units.size());
  summary->num_kv_segs = static_cast<int32_t>(w.kv_segs.size());
  summary->used_flops = w.flops;
  static_assert(sizeof(gva::WorkItem) == 8 * sizeof(int32_t) && sizeof(gva::KvUnit) == 8 * sizeof(int32_t),
                "8 int32 per exported record");
  auto copy_out = [](int32_t* dst, int32_t cap, const void* src, size_t n) {
    if (dst != nullptr && cap > 0) std::memcpy(dst, src, std::min<size_t>(n, cap) * 8 * sizeof(int32_t));
  };
  copy_out(items, items_capacity, w.items.data(), w.items.size());
  copy_out(bwd_items, bwd_items_capacity, w.bwd_items.data(), w.bwd_items.size());
  copy_out(kv_units, kv_units_capacity, w.kv_units.data(), w.kv_units.size());
  static_assert(sizeof(gva::SegRef) == 2 * sizeof(int32_t), "2 int32 per exported segment");
  if (kv_segs != nullptr && kv_segs_capacity > 0)
    std::memcpy(kv_segs, w.kv_segs.data(), std::min<size_t>(w.kv_segs.size(), kv_segs_capacity) * sizeof(gva::SegRef));
  return ok();
}

gva_status gva_forward(gva_plan_t plan, const void* q, const void* k, const void* v, void* out, gva_dtype out_dtype,
                       float* lse, float softmax_scale, cudaStream_t stream) {
  if (plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "plan is NULL");
  if (out_dtype != GVA_BF16 && out_dtype != GVA_FP32) return fail(GVA_ERR_INVALID_ARG, "bad out_dtype %d", (int)out_dtype);
  if (plan->num_items == 0) return ok();  // no used rows: nothing to write
  // With no keys at all (every item keyless) K and V are never read and may be empty.
  const bool has_keys = plan->total_k > 0;
  if (!has_keys) k = v = q;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr)
    return fail(GVA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(GVA_ERR_INVALID_ARG, "q, k, v, out and lse must be 16-byte aligned");
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale))
    return fail(GVA_ERR_INVALID_ARG, "softmax_scale is not finite");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != plan->device)
    return fail(GVA_ERR_INVALID_ARG, "the plan was built on device %d, the current device is %d", plan->device, dev);
  const int32_t tokens_per_tile = gva::kTileRows / plan->group;
  // full tiles leave through TMA stores, over a map of out laid out like Q's
  CUtensorMap mq, mk, mv, mo;
  {
    std::lock_guard<std::mutex> lock(plan->map_mutex);
    MapCache& c = plan->fwd_maps;
    if (!(c.valid && c.ptr[0] == q && c.ptr[1] == k && c.ptr[2] == v && c.ptr[3] == out &&
          c.out_dtype == static_cast<int>(out_dtype))) {
      c.valid = false;
      gva_status s;
      const int64_t krows = has_keys ? plan->total_k : 1;
      if ((s = make_map(&c.map[0], q, plan->total_q, plan->num_heads_q, plan->head_dim, tokens_per_tile, plan->group,
                        "Q")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[1], k, krows, plan->num_heads_kv, plan->head_dim, gva::kBlockKeys, 1, "K")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[2], v, krows, plan->num_heads_kv, plan->head_dim, gva::kBlockKeys, 1, "V")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[3], out, plan->total_q, plan->num_heads_q, plan->head_dim, tokens_per_tile,
                        plan->group, "O", out_dtype == GVA_FP32)) != GVA_OK)
        return s;
      c.ptr[0] = q;
      c.ptr[1] = k;
      c.ptr[2] = v;
      c.ptr[3] = out;
      c.out_dtype = static_cast<int>(out_dtype);
      c.valid = true;
    }
    mq = c.map[0];
    mk = c.map[1];
    mv = c.map[2];
    mo = c.map[3];
  }
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(plan->head_dim));
  gva::FwdParams prm{};
  prm.items = plan->d_items;
  prm.blocks = plan->d_blocks;
  prm.num_items = plan->num_item_slots;
  prm.out = out;
  prm.out_wide = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  prm.out_tma = 1;
  prm.lse = lse;
  prm.total_q = plan->total_q;
  prm.num_heads_q = plan->num_heads_q;
  prm.group = plan->group;
  prm.tokens_per_tile = tokens_per_tile;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.causal_block = plan->causal_block;
  prm.error_flag = plan->d_error;
  e = gva::launch_forward(plan->head_dim, out_dtype == GVA_FP32, prm, mq, mk, mv, mo, plan->grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the forward kernel");
  return ok();
}

gva_status gva_lse_merge(gva_plan_t plan, int32_t num_parts, const void* const* outs, gva_dtype in_dtype,
                         const float* const* lses, void* out, gva_dtype out_dtype, float* lse, cudaStream_t stream) {
  if (plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "plan is NULL");
  if (num_parts < 1 || num_parts > gva::kMaxMergeParts)
    return fail(GVA_ERR_INVALID_ARG, "num_parts=%d outside [1, %d]", num_parts, gva::kMaxMergeParts);
  if ((in_dtype != GVA_BF16 && in_dtype != GVA_FP32) || (out_dtype != GVA_BF16 && out_dtype != GVA_FP32))
    return fail(GVA_ERR_INVALID_ARG, "bad dtype");
  if (outs == nullptr || lses == nullptr) return fail(GVA_ERR_INVALID_ARG, "outs / lses is NULL");
  if (plan->num_units == 0) return ok();
  gva::MergeParams prm{};
  for (int i = 0; i < num_parts; ++i) {
    if (outs[i] == nullptr || lses[i] == nullptr) return fail(GVA_ERR_INVALID_ARG, "partition %d has a NULL pointer", i);
    if (!aligned16(outs[i])) return fail(GVA_ERR_INVALID_ARG, "outs[%d] must be 16-byte aligned", i);
    if ((reinterpret_cast<uintptr_t>(lses[i]) & 3u) != 0) return fail(GVA_ERR_INVALID_ARG, "lses[%d] misaligned", i);
    prm.outs[i] = outs[i];
    prm.lses[i] = lses[i];
  }
  if (out == nullptr || lse == nullptr) return fail(GVA_ERR_INVALID_ARG, "out / lse is NULL");
  if (!aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(GVA_ERR_INVALID_ARG, "out must be 16-byte aligned and lse 4-byte aligned");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != plan->device)
    return fail(GVA_ERR_INVALID_ARG, "the plan was built on device %d, the current device is %d", plan->device, dev);
  prm.units = plan->d_units;
  prm.num_units = plan->num_units;
  prm.num_parts = num_parts;
  prm.out = out;
  prm.lse = lse;
  prm.total_q = plan->total_q;
  prm.num_heads_q = plan->num_heads_q;
  prm.head_dim = plan->head_dim;
  prm.error_flag = plan->d_error;
  int ring_slots = 0;
  if (gva::merge_smem_bytes(in_dtype == GVA_FP32, num_parts, plan->num_heads_q, &ring_slots) < 0)
    return fail(GVA_ERR_UNSUPPORTED, "%d partitions of %d query heads do not fit the merge's shared memory",
                num_parts, plan->num_heads_q);
  e = gva::launch_merge(in_dtype == GVA_FP32, out_dtype == GVA_FP32, prm, plan->sm_count, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the LSE merge kernel");
  return ok();
}

gva_status gva_backward_workspace_size(gva_plan_t plan, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return fail(GVA_ERR_INVALID_ARG, "plan or bytes is NULL");
  *bytes = static_cast<size_t>(plan->num_heads_q) * static_cast<size_t>(plan->total_q) * sizeof(float);
  return ok();
}

gva_status gva_backward(gva_plan_t plan, const void* q, const void* k, const void* v, const void* out,
                        const void* d_out, const float* lse, void* dq, gva_dtype dq_dtype, void* dk, void* dv,
                        gva_dtype dkv_dtype, void* workspace, size_t workspace_bytes, float softmax_scale,
                        cudaStream_t stream) {
  if (plan == nullptr) return fail(GVA_ERR_INVALID_ARG, "plan is NULL");
  if ((dq_dtype != GVA_BF16 && dq_dtype != GVA_FP32) || (dkv_dtype != GVA_BF16 && dkv_dtype != GVA_FP32))
    return fail(GVA_ERR_INVALID_ARG, "bad gradient dtype");
  if (plan->num_bwd_items == 0 && plan->num_kv_units == 0) return ok();  // no used row and no used key
  // With no keys (or no rows) at all, the K-side (or Q-side) tensors are never read or
  // written and may be empty; one of the two sides is non-empty here.
  const bool has_keys = plan->total_k > 0;
  const bool has_rows = plan->total_q > 0;
  if (!has_keys) k = v = dk = dv = const_cast<void*>(q);
  if (!has_rows) {
    q = out = d_out = dq = const_cast<void*>(k);
    lse = static_cast<const float*>(k);
  }
  if (q == nullptr || k == nullptr || v == nullptr || dk == nullptr || dv == nullptr || out == nullptr ||
      d_out == nullptr || lse == nullptr || dq == nullptr)
    return fail(GVA_ERR_INVALID_ARG, "a tensor pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(d_out) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return fail(GVA_ERR_INVALID_ARG, "every tensor and the workspace must be 16-byte aligned");
  const size_t need = static_cast<size_t>(plan->num_heads_q) * static_cast<size_t>(plan->total_q) * sizeof(float);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(GVA_ERR_INVALID_ARG, "the workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (!(softmax_scale == softmax_scale) || std::isinf(softmax_scale))
    return fail(GVA_ERR_INVALID_ARG, "softmax_scale is not finite");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != plan->device)
    return fail(GVA_ERR_INVALID_ARG, "the plan was built on device %d, the current device is %d", plan->device, dev);
  const int32_t tokens_per_tile = gva::kTileRows / plan->group;
  const int64_t qrows = has_rows ? plan->total_q : 1;  // the maps need one row
  const int64_t krows = has_keys ? plan->total_k : 1;
  CUtensorMap mq, mk, mv, mdo;
  {
    std::lock_guard<std::mutex> lock(plan->map_mutex);
    MapCache& c = plan->bwd_maps;
    if (!(c.valid && c.ptr[0] == q && c.ptr[1] == k && c.ptr[2] == v && c.ptr[3] == d_out)) {
      c.valid = false;
      gva_status s;
      if ((s = make_map(&c.map[0], q, qrows, plan->num_heads_q, plan->head_dim, tokens_per_tile, plan->group,
                        "Q")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[1], k, krows, plan->num_heads_kv, plan->head_dim, gva::kBlockKeys, 1, "K")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[2], v, krows, plan->num_heads_kv, plan->head_dim, gva::kBlockKeys, 1, "V")) != GVA_OK)
        return s;
      if ((s = make_map(&c.map[3], d_out, qrows, plan->num_heads_q, plan->head_dim, tokens_per_tile, plan->group,
                        "dO")) != GVA_OK)
        return s;
      c.ptr[0] = q;
      c.ptr[1] = k;
      c.ptr[2] = v;
      c.ptr[3] = d_out;
      c.valid = true;
    }
    mq = c.map[0];
    mk = c.map[1];
    mv = c.map[2];
    mdo = c.map[3];
  }
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(plan->head_dim));
  gva::BwdParams prm{};
  prm.items = plan->d_bwd_items;
  prm.blocks = plan->d_blocks;
  prm.num_items = plan->num_bwd_items;
  prm.kv_units = plan->d_kv_units;
  prm.kv_segs = plan->d_kv_segs;
  prm.num_kv_units = plan->num_kv_units;
  prm.lse = lse;
  prm.dvec = static_cast<float*>(workspace);
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.total_q = plan->total_q;
  prm.num_heads_q = plan->num_heads_q;
  prm.num_heads_kv = plan->num_heads_kv;
  prm.group = plan->group;
  prm.tokens_per_tile = tokens_per_tile;
  prm.scale = scale;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.causal_block = plan->causal_block;
  prm.error_flag = plan->d_error;
  e = gva::launch_backward(plan->head_dim, dq_dtype == GVA_FP32, dkv_dtype == GVA_FP32, prm, plan->d_units,
                           plan->num_units, out, d_out, static_cast<float*>(workspace), mq, mk, mv, mdo,
                           plan->bwd_grid, plan->kv_grid, plan->sm_count, stream);
  if (e != cudaSuccess) return cuda_fail(e, "launching the backward kernels");
  return ok();
}

gva_status gva_plan_destroy(gva_plan_t plan) {
  free_plan(plan);
  return ok();
}

gva_status gva_plan_get_info(gva_plan_t plan, gva_plan_info* info) {
  if (plan == nullptr || info == nullptr) return fail(GVA_ERR_INVALID_ARG, "plan or info is NULL");
  info->num_segments = plan->num_segments;
  info->num_heads_q = plan->num_heads_q;
  info->num_heads_kv = plan->num_heads_kv;
  info->head_dim = plan->head_dim;
  info->total_q = plan->total_q;
  info->total_k = plan->total_k;
  info->num_work_items = plan->num_items;
  info->num_merge_units = plan->num_units;
  info->grid_ctas = plan->grid;
  info->sm_count = plan->sm_count;
  info->used_flops = plan->used_flops;
  return ok();
}

gva_status gva_device_status(gva_plan_t plan) {
  if (plan == nullptr) return static_cast<gva_status>(gva::noalloc_device_status());
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int word = 0;
  if ((e = cudaMemcpy(&word, plan->d_error, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the device error word");
  if (word != 0) {
    cudaMemset(plan->d_error, 0, sizeof(int));
    return fail(GVA_ERR_DEVICE_CHECK, "a kernel recorded device error bits 0x%x (1 = bounded wait timed out)", word);
  }
  return ok();
}

const char* gva_status_string(gva_status status) {
  switch (status) {
    case GVA_OK: return "GVA_OK";
    case GVA_ERR_INVALID_ARG: return "GVA_ERR_INVALID_ARG";
    case GVA_ERR_UNSUPPORTED: return "GVA_ERR_UNSUPPORTED";
    case GVA_ERR_CUDA: return "GVA_ERR_CUDA";
    case GVA_ERR_DEVICE_CHECK: return "GVA_ERR_DEVICE_CHECK";
  }
  return "GVA_UNKNOWN_STATUS";
}

const char* gva_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
