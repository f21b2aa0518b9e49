// Training driver: level-wise growth of each tree ("Module Design: Training
// Core" s.6): for every level, build the histograms of the active nodes (the
// smaller child of each sibling pair directly, the larger by subtraction),
// select splits by the frozen rule, route rows to the children, then freeze
// the last level as leaves and update the training predictions.
//
// The host only queues work: every grid is sized from host-known bounds
// (at most 2^d slots at level d), kernels read the actual level sizes from
// device memory and idle blocks exit, so no level needs a device-to-host
// round trip.  The only synchronisations are the input checks at the start
// and the single copy of the finished model at the end ("Module Design:
// Training Core" s.5: no partial model leaves a failed run).
#include <atomic>
#include <vector>

#include "rows.cuh"

namespace gbdt {

namespace {


struct LevelStats {
  int64_t n_act;         // rows in the level's nodes
  int64_t n_built_rows;  // rows of the nodes whose histograms are built directly
  int64_t n_split_rows;  // rows of the nodes that split
  int64_t n_scan_rows;   // rows the histogram pass reads (at odd levels a built node's whole pair)
  int32_t n_slots;
  int32_t n_built;
};

std::atomic<int32_t> g_fail_after_levels{-1};

// The next level's histogram work (written by the level above, so that the histogram launch needs no
// setup launch of its own): the work list in that level's scratch view, the plan's CTA bound and least
// cost per CTA, and at a filtered (odd) level each slot's scan range and filter.  st null: no next
// histogram level.
struct NextWork {
  SegWorkView wv;
  int32_t max_ctas;
  int64_t min_rows;
  gbdt_segment* scan;    // non-null when the next level is filtered
  gbdt_filter* filters;
};

__device__ __forceinline__ int32_t work_ctas(long long cost, const NextWork& nw) {
  const long long by_size = (cost + nw.min_rows - 1) / nw.min_rows;
  return static_cast<int32_t>(by_size < nw.max_ctas ? by_size : nw.max_ctas);
}

// budget[0]: leaves of the tree's earlier levels; budget[1]: 1 once the leaf budget has bound;
// budget[2]: index of the tree being grown (-1 before the first), advanced here at each tree's start so
// that the per-tree launch sequence is the same for every tree (it can be replayed as one graph).
__global__ void reset_root_kernel(gbdt_level* level, uint8_t* build_flag, gbdt_segment* seg, int64_t N,
                                  int32_t* budget, NextWork nw) {
  level->node_begin = 0;
  level->n_slots = 1;
  build_flag[0] = 1;
  seg[0] = gbdt_segment{0, N};
  budget[0] = 0;
  budget[1] = 0;
  budget[2] += 1;
  if (nw.wv.st) {  // the root's work list: one slot of N rows
    nw.wv.build_slot[0] = 0;
    nw.wv.row_start[0] = 0;
    nw.wv.row_start[1] = N;
    const long long cost = N + kSlotCost;
    *nw.wv.st = SegWork{N, cost, 1, work_ctas(cost, nw)};
  }
}

__global__ void iota_kernel(uint32_t* __restrict__ v, int64_t N) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x)
    v[i] = static_cast<uint32_t>(i);
}

// Root totals when the root is also the last level (max_depth 0): count and
// fixed-point sum of g (and, logistic, of h) over all rows; integer adds, so
// the order is irrelevant.
__global__ void root_totals_kernel(const double* __restrict__ g, int64_t N, const int32_t* __restrict__ fixed_exp,
                                   int logistic, SlotTotals* __restrict__ tot) {
  const double scale = ldexp(1.0, fixed_exp[0]);
  const double scale_h = logistic ? ldexp(1.0, fixed_exp[1]) : 0.0;
  long long acc = 0, acc_h = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    acc += to_fixed(g[i], scale);
    if (logistic) acc_h += to_fixed(logistic_hess(g[i]), scale_h);
  }
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, o);
    acc_h += __shfl_xor_sync(0xffffffffu, acc_h, o);
  }
  if ((threadIdx.x & 31) == 0 && acc != 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(&tot->q), static_cast<unsigned long long>(acc));
  if ((threadIdx.x & 31) == 0 && acc_h != 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(&tot->qh), static_cast<unsigned long long>(acc_h));
  if (blockIdx.x == 0 && threadIdx.x == 0) tot->cnt = static_cast<uint32_t>(N);
}

// One CTA of 1024 threads: child numbering by an in-order scan of the split
// flags, node records of this level, and the next level's bookkeeping.
__global__ void __launch_bounds__(1024)
    apply_level_kernel(int d, int D, const gbdt_level* __restrict__ level, int32_t max_slots,
                       const gbdt_split* __restrict__ splits, const SlotTotals* __restrict__ totals,
                       const uint8_t* __restrict__ build_flag, const int32_t* __restrict__ fixed_exp, double lambda,
                       const gbdt_segment* __restrict__ seg, gbdt_node* __restrict__ trees,
                       int32_t* __restrict__ n_nodes, gbdt_level* __restrict__ next_level,
                       SlotTotals* __restrict__ next_totals, gbdt_segment* __restrict__ next_seg,
                       int32_t* __restrict__ pair_parent, uint8_t* __restrict__ next_build, Route* __restrict__ route,
                       LevelStats* __restrict__ level_stats, int32_t num_leaves, int32_t* __restrict__ budget,
                       int logistic, int32_t* __restrict__ err, NextWork nw, RowsSetup rs) {
  // this tree's node array, node count and level statistics (trees, n_nodes: per tree; level_stats:
  // level d of tree 0, D + 1 records per tree)
  const int t = budget[2];
  gbdt_node* __restrict__ tree = trees + static_cast<int64_t>(t) * ((2 << D) - 1);
  int32_t* __restrict__ n_nodes_out = n_nodes + t;
  LevelStats* __restrict__ stats = level_stats + static_cast<int64_t>(t) * (D + 1);
  __shared__ int s_w[33];
  __shared__ long long s_wl[33];
  long long s_rows_pre = 0;  // block-uniform: rows of the next level's work list before the current chunk
  __shared__ double s_gain[kMaxSlots];                  // leaf budget: the level's candidate gains
  __shared__ uint32_t s_cand[kMaxSlots / 32], s_keep[kMaxSlots / 32];
  __shared__ int s_ncand, s_bind;
  __shared__ unsigned long long s_act, s_built_rows, s_split_rows, s_scan_rows;
  __shared__ int s_built;
  int s_pre = 0;  // block-uniform: splitting slots before the current chunk
  if (threadIdx.x == 0) {
    s_act = s_built_rows = s_split_rows = s_scan_rows = 0;
    s_built = 0;
  }
  __syncthreads();
  const int node_begin = level->node_begin;
  int n_slots = level->n_slots;
  if (n_slots > max_slots) {
    if (threadIdx.x == 0) raise_error(err, kErrLevelSize);
    n_slots = max_slots;
  }
  const int next_begin = node_begin + n_slots;
  const int S = fixed_exp[0];
  const int S_h = logistic ? fixed_exp[1] : 0;
  // After the leaf budget has bound, the level below it is the last: every node is a leaf.
  const bool stopped = budget[1] != 0;
  const bool leaf_level = d >= D || stopped;
  // Leaf budget: if every candidate of the level splitting would leave more than num_leaves leaves,
  // only the first K = num_leaves - (leaves so far + the level's nodes) in (gain desc, slot asc)
  // split (a total order: the slot is unique), and the budget has bound.
  if (threadIdx.x == 0) {
    s_ncand = 0;
    s_bind = 0;
  }
  for (int w = threadIdx.x; w < kMaxSlots / 32; w += blockDim.x) s_cand[w] = s_keep[w] = 0;
  __syncthreads();
  if (num_leaves > 0 && !leaf_level) {
    for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {  // one ballot per warp of 32 slots
      const int s = c0 + threadIdx.x;
      const bool cand = s < n_slots && splits[s].feature >= 0;
      if (cand) s_gain[s] = splits[s].gain;
      const uint32_t m = __ballot_sync(0xffffffffu, cand);
      if ((threadIdx.x & 31) == 0 && m) {
        s_cand[s >> 5] = m;  // s is a multiple of 32 here (blockDim.x is)
        atomicAdd(&s_ncand, __popc(m));
      }
    }
    __syncthreads();
    const int K = num_leaves - (budget[0] + n_slots);
    if (s_ncand > K) {
      for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
        if (!(s_cand[s >> 5] >> (s & 31) & 1u)) continue;
        const double gs = s_gain[s];
        int rank = 0;
        for (int o = 0; o < n_slots; ++o)
          if ((s_cand[o >> 5] >> (o & 31) & 1u) && (s_gain[o] > gs || (s_gain[o] == gs && o < s))) ++rank;
        if (rank < K) atomicOr(&s_keep[s >> 5], 1u << (s & 31));
      }
      if (threadIdx.x == 0) s_bind = 1;
    }
    __syncthreads();
  }
  const bool bind = s_bind != 0;
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool in = s < n_slots;
    int is_split = 0;
    gbdt_split sp{};
    SlotTotals tot{};
    if (in) {
      if (d < D) {
        sp = splits[s];
        is_split = !stopped && sp.feature >= 0 && (!bind || (s_keep[s >> 5] >> (s & 31) & 1u));
        if (d > 0 && (sp.q_total != totals[s].q || sp.cnt_total != totals[s].cnt || sp.h_total != totals[s].qh))
          raise_error(err, kErrHistTotals);
        tot.q = sp.q_total;
        tot.qh = sp.h_total;
        tot.cnt = sp.cnt_total;
      } else {
        tot = totals[s];
      }
      if (seg[s].count != static_cast<int64_t>(tot.cnt)) raise_error(err, kErrHistTotals);
    }
    {  // the level's statistics: warp sums, one shared atomic per warp and counter
      const bool built = in && d < D && build_flag[s];
      // at odd levels a node's rows still sit in its pair's (its parent's) segment
      const unsigned long long scan =
          built ? static_cast<unsigned long long>((d & 1) ? seg[s & ~1].count + seg[s | 1].count : seg[s].count) : 0;
      unsigned long long act = in ? tot.cnt : 0, brows = built ? tot.cnt : 0, srows = is_split ? tot.cnt : 0;
      unsigned long long sc = scan;
      int nb = built ? 1 : 0;
      for (int o = 16; o > 0; o >>= 1) {
        act += __shfl_xor_sync(0xffffffffu, act, o);
        brows += __shfl_xor_sync(0xffffffffu, brows, o);
        srows += __shfl_xor_sync(0xffffffffu, srows, o);
        sc += __shfl_xor_sync(0xffffffffu, sc, o);
        nb += __shfl_xor_sync(0xffffffffu, nb, o);
      }
      if ((threadIdx.x & 31) == 0) {
        if (act) atomicAdd(&s_act, act);
        if (nb) {
          atomicAdd(&s_built, nb);
          atomicAdd(&s_built_rows, brows);
          atomicAdd(&s_scan_rows, sc);
        }
        if (srows) atomicAdd(&s_split_rows, srows);
      }
    }
    int n_split;
    const int e_split = block_scan_excl(is_split, s_w, &n_split);
    // the next level's work list: the built child of the k-th split (its rows; at a filtered level the scan
    // covers the whole pair, the parent's rows)
    long long wrows = 0;
    if (is_split) wrows = nw.scan ? static_cast<long long>(tot.cnt)
                                  : static_cast<long long>(sp.cnt_left <= tot.cnt - sp.cnt_left ? sp.cnt_left
                                                                                                 : tot.cnt - sp.cnt_left);
    long long n_wrows;
    const long long e_rows = block_scan_excl(wrows, s_wl, &n_wrows);
    if (in) {
      const int k = s_pre + e_split;
      const double G = from_fixed(tot.q, S);
      const double H = logistic ? from_fixed(tot.qh, S_h) : static_cast<double>(tot.cnt);
      gbdt_node nd;
      nd.leaf_value = __ddiv_rn(-G, __dadd_rn(H, lambda));
      nd.reserved[0] = nd.reserved[1] = nd.reserved[2] = nd.reserved[3] = 0;
      nd.reserved[4] = nd.reserved[5] = nd.reserved[6] = 0;
      Route rt{-1, -1, -1, k};
      if (is_split) {
        nd.feature = sp.feature;
        nd.threshold_bin = sp.bin;
        nd.left = next_begin + 2 * k;
        nd.right = next_begin + 2 * k + 1;
        nd.gain = sp.gain;
        nd.is_leaf = 0;
        const uint32_t cl = sp.cnt_left, cr = sp.cnt_total - sp.cnt_left;
        next_totals[2 * k] = SlotTotals{sp.q_left, sp.h_left, cl, 0};
        next_totals[2 * k + 1] = SlotTotals{
            static_cast<int64_t>(static_cast<uint64_t>(sp.q_total) - static_cast<uint64_t>(sp.q_left)),
            static_cast<int64_t>(static_cast<uint64_t>(sp.h_total) - static_cast<uint64_t>(sp.h_left)), cr, 0};
        next_seg[2 * k] = gbdt_segment{seg[s].start, static_cast<int64_t>(cl)};
        next_seg[2 * k + 1] = gbdt_segment{seg[s].start + cl, static_cast<int64_t>(cr)};
        pair_parent[k] = s;
        const uint8_t left_small = cl <= cr ? 1 : 0;  // build the smaller child; ties build the left one
        next_build[2 * k] = left_small;
        next_build[2 * k + 1] = 1 - left_small;
        rt = Route{sp.feature, sp.bin, next_begin + 2 * k, k};
        if (nw.wv.st) {
          nw.wv.build_slot[k] = left_small ? 2 * k : 2 * k + 1;
          nw.wv.row_start[k] = s_rows_pre + e_rows;
        }
        if (nw.scan) {  // both children scan the pair's rows (the parent's segment), each keeps its side
          nw.scan[2 * k] = nw.scan[2 * k + 1] = gbdt_segment{seg[s].start, static_cast<int64_t>(tot.cnt)};
          nw.filters[2 * k] = gbdt_filter{sp.feature, sp.bin, 0, 0};
          nw.filters[2 * k + 1] = gbdt_filter{sp.feature, sp.bin, 1, 0};
        }
      } else {
        nd.feature = nd.threshold_bin = nd.left = nd.right = -1;
        nd.gain = 0.0;
        nd.is_leaf = 1;
      }
      tree[node_begin + s] = nd;
      route[s] = rt;
    }
    s_pre += n_split;
    s_rows_pre += n_wrows;
  }
  __syncthreads();  // the shared statistics are complete, and this level's routes and next segments
  if (threadIdx.x == 0) {
    budget[0] += n_slots - s_pre;  // this level's leaves
    if (bind) budget[1] = 1;
    next_level->node_begin = next_begin;
    next_level->n_slots = 2 * s_pre;
    *n_nodes_out = next_begin + 2 * s_pre;
    stats->n_act = static_cast<int64_t>(s_act);
    stats->n_built_rows = static_cast<int64_t>(s_built_rows);
    stats->n_split_rows = static_cast<int64_t>(s_split_rows);
    stats->n_scan_rows = static_cast<int64_t>(s_scan_rows);
    stats->n_slots = n_slots;
    stats->n_built = s_built;
    if (nw.wv.st) {
      nw.wv.row_start[s_pre] = s_rows_pre;
      const long long cost = s_rows_pre + kSlotCost * s_pre;
      *nw.wv.st = SegWork{s_rows_pre, cost, s_pre, work_ctas(cost, nw)};
    }
  }
  // the setup of the row launches that follow (the pair routes read the routes and next segments this
  // block wrote before the barrier above)
  if (rs.kind == kRowsSlotTiles) {
    rows_slot_tiles(level, max_slots, seg, rs.mv_tile_start, rs.mv_st);
  } else if (rs.kind == kRowsPairRoutes) {
    rows_pair_routes(level, max_slots, seg, route, rs.route_prev, rs.pair_parent, next_seg, rs.floc, rs.pairs,
                     rs.pair_tile_start, rs.pair_st, rs.tile_status, rs.n_status);
  }
}

struct TrainWs {
  double* g0;         // gradients in original row order (level 0 positions)
  uint32_t* orig0;    // identity: original row id of level-0 positions
  uint16_t* leaf;     // leaf of each original row in the current tree
  uint8_t* bins_rb0;    // the caller's bins in the row-block layout (levels 0 and 1)
  uint32_t* floc;       // [F] where each feature's bins sit in the row-block copies (slot, nibble)
  uint32_t* slot_src;   // [F] the features of each slot
  int32_t* fsched;      // [F] the split search's features: those with more than kSplitNarrowBins bins, then the rest
  uint8_t* bins_xy[2];  // row-block copies in later orders (alternating)
  double* g_xy[2];
  uint32_t* orig_xy[2];
  gbdt_segment* seg[2];
  gbdt_segment* scan;    // odd levels: each slot's scan range (its pair's rows)
  gbdt_filter* filters;  // odd levels: each slot's side of its parent's split
  void* seg_scratch;
  void* move_scratch;
  uint32_t* hist_cnt[2];
  int64_t* hist_q[2];
  int64_t* hist_h[2];  // logistic only (else null)
  uint32_t* root_cnt;  // the root's count histogram [F][256] (the same for every tree of a call)
  gbdt_split* splits;
  void* split_scratch;
  SlotTotals* totals[2];
  gbdt_level* level[2];
  uint8_t* build[2];
  int32_t* pair_parent[2];  // by level parity: sibling pair -> parent slot
  Route* route[2];          // by level parity: each slot's split routing
  gbdt_node* trees;
  int32_t* n_nodes;
  LevelStats* stats;
  unsigned long long* maxabs;
  int32_t* budget;  // leaf budget state of the current tree; [2]: the tree's index
  int32_t* fixed_exp;  // [2]: S of g, S_h of the logistic hessians
  double* init;
  double* label_partials;
  int32_t* err;
  int32_t* nonfinite;
};

int32_t max_nodes_of(int D) { return (1 << (D + 1)) - 1; }

// A captured sequence of launches (one tree) replayed with cudaGraphLaunch.  The capture runs on a
// stream of its own (the caller's stream may be the legacy default stream, which cannot capture);
// capturing only records the launches, and the launch counter is corrected for them.  Timing events
// recorded during the capture become event-record nodes; before each replay they are pointed at that
// tree's events (the graph is kept for their node handles).
struct TreeGraph {
  cudaStream_t cs = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int64_t launches = 0;                  // kernels in the graph
  std::vector<cudaGraphNode_t> marks;    // event-record nodes
  std::vector<cudaEvent_t> mark_events;  // the event each one recorded in the capture
  TreeGraph() = default;
  TreeGraph(const TreeGraph&) = delete;
  TreeGraph& operator=(const TreeGraph&) = delete;
  ~TreeGraph() {  // an executable graph still in flight is released when it completes
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    if (cs) cudaStreamDestroy(cs);
  }
  template <typename F>
  int capture(F&& record) {
    GBDT_CUDA(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    GBDT_CUDA(cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed));
    const int64_t l0 = launch_count();
    const int rc = record(cs);
    const cudaError_t e = cudaStreamEndCapture(cs, &graph);
    launches = launch_count() - l0;
    count_launches(static_cast<int>(-launches));
    if (rc != GBDT_OK) return rc;
    if (e != cudaSuccess) {
      set_error("gbdt_train: capturing a tree's launches failed: %s", cudaGetErrorString(e));
      return GBDT_ERR_CUDA;
    }
    size_t n = 0;
    GBDT_CUDA(cudaGraphGetNodes(graph, nullptr, &n));
    std::vector<cudaGraphNode_t> nodes(n);
    GBDT_CUDA(cudaGraphGetNodes(graph, nodes.data(), &n));
    for (cudaGraphNode_t node : nodes) {
      cudaGraphNodeType type;
      GBDT_CUDA(cudaGraphNodeGetType(node, &type));
      if (type != cudaGraphNodeTypeEventRecord) continue;
      cudaEvent_t ev = nullptr;
      GBDT_CUDA(cudaGraphEventRecordNodeGetEvent(node, &ev));
      marks.push_back(node);
      mark_events.push_back(ev);
    }
    const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
    if (ei != cudaSuccess) {
      exec = nullptr;
      set_error("gbdt_train: instantiating a tree's graph failed: %s", cudaGetErrorString(ei));
      return GBDT_ERR_CUDA;
    }
    return GBDT_OK;
  }
};
TrainWs carve_train(void* ws, size_t bytes, int64_t N, int32_t F, int64_t ldb, const gbdt_params& p,
                    size_t* need) {
  Carve c(ws, bytes);
  TrainWs w{};
  const int D = p.max_depth;
  const int64_t hist_slots = D >= 1 ? (int64_t(1) << (D - 1)) : 1;
  const int level_slots = 1 << D;
  const int64_t hist_entries = hist_slots * F * kBins;
  const int T = p.n_trees > 0 ? p.n_trees : 1;
  const int64_t n16 = (N + 15) / 16 * 16;
  w.g0 = c.take<double>(n16);
  w.orig0 = c.take<uint32_t>(n16);
  w.leaf = c.take<uint16_t>(n16);
  w.floc = c.take<uint32_t>(F);
  w.slot_src = c.take<uint32_t>(F);
  w.fsched = c.take<int32_t>(F);
  if (D >= 1) {
    w.bins_rb0 = c.take<uint8_t>(row_block_bytes(N, F));
    for (int i = 0; i < 2; ++i) {
      w.bins_xy[i] = c.take<uint8_t>(row_block_bytes(N, F));
      w.g_xy[i] = c.take<double>(n16);
      w.orig_xy[i] = c.take<uint32_t>(n16);
    }
  }
  for (int i = 0; i < 2; ++i) w.seg[i] = c.take<gbdt_segment>(level_slots);
  w.scan = c.take<gbdt_segment>(level_slots);
  w.filters = c.take<gbdt_filter>(level_slots);
  w.seg_scratch = c.take<unsigned char>(seg_hist_scratch_bytes(static_cast<int32_t>(hist_slots)));
  w.move_scratch = c.take<unsigned char>(move_scratch_bytes(N, level_slots));
  const bool logistic = p.objective == GBDT_OBJECTIVE_LOGISTIC;
  for (int i = 0; i < 2; ++i) {
    w.hist_cnt[i] = c.take<uint32_t>(hist_entries);
    w.hist_q[i] = c.take<int64_t>(hist_entries);
    w.hist_h[i] = logistic ? c.take<int64_t>(hist_entries) : nullptr;
  }
  w.root_cnt = c.take<uint32_t>(static_cast<size_t>(F) * kBins);
  w.splits = c.take<gbdt_split>(level_slots);
  w.split_scratch = c.take<unsigned char>(find_splits_scratch_bytes(F, static_cast<int32_t>(hist_slots)));
  for (int i = 0; i < 2; ++i) {
    w.totals[i] = c.take<SlotTotals>(level_slots);
    w.level[i] = c.take<gbdt_level>(1);
    w.build[i] = c.take<uint8_t>(level_slots);
  }
  for (int i = 0; i < 2; ++i) {
    w.pair_parent[i] = c.take<int32_t>(level_slots / 2 + 1);
    w.route[i] = c.take<Route>(level_slots);
  }
  w.trees = c.take<gbdt_node>(static_cast<size_t>(T) * max_nodes_of(D));
  w.n_nodes = c.take<int32_t>(T);
  w.stats = c.take<LevelStats>(static_cast<size_t>(T) * (D + 1));
  w.maxabs = c.take<unsigned long long>(2);
  w.budget = c.take<int32_t>(4);
  w.fixed_exp = c.take<int32_t>(2);
  w.init = c.take<double>(1);
  w.label_partials = c.take<double>(kSumBlocks);
  w.err = c.take<int32_t>(1);
  w.nonfinite = c.take<int32_t>(1);
  *need = c.used;
  return w;
}

// Timing events of the histogram launches, reused across calls.
struct EventPool {
  std::vector<cudaEvent_t> ev;
  cudaError_t ensure(size_t n) {
    while (ev.size() < n) {
      cudaEvent_t e;
      cudaError_t r = cudaEventCreate(&e);
      if (r != cudaSuccess) return r;
      ev.push_back(e);
    }
    return cudaSuccess;
  }
};
EventPool& event_pool() {
  static EventPool pool;
  return pool;
}

}  // namespace

}  // namespace gbdt

using namespace gbdt;

int validate_params(const gbdt_params* p);

extern "C" size_t gbdt_train_workspace_size(int64_t N, int32_t F, const gbdt_params* p) {
  if (!p || N < 1 || F < 1 || p->max_depth < 0 || p->max_depth > GBDT_MAX_DEPTH) return 0;
  size_t need = 0;
  carve_train(nullptr, 0, N, F, (N + 15) / 16 * 16, *p, &need);
  return need;
}

extern "C" void gbdt_debug_inject_failure(int32_t after_levels) { g_fail_after_levels.store(after_levels); }

extern "C" int gbdt_train(const uint8_t* bins, int64_t ldb, const int32_t* n_bins, int64_t N, int32_t F,
                          const float* label, const gbdt_params* p, double* pred_out, double* init_pred_out,
                          gbdt_node* nodes_out, int32_t* nodes_per_tree, gbdt_diagnostics* diag, void* ws,
                          size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && n_bins && label && p && pred_out && init_pred_out && nodes_out && nodes_per_tree,
                 "gbdt_train: null pointer");
  int rc = validate_params(p);
  if (rc != GBDT_OK) return rc;
  for (int t = 0; t < p->n_trees; ++t) nodes_per_tree[t] = 0;
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31), "gbdt_train: N out of range");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096, "gbdt_train: F out of range");
  GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins, 16), "gbdt_train: bins need ldb >= N, ldb %% 16 == 0 "
                 "and a 16-byte aligned base");
  size_t need = 0;
  TrainWs w = carve_train(ws, ws_bytes, N, F, ldb, *p, &need);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_train: workspace needs %zu bytes (got %zu)", need, ws_bytes);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = p->max_depth, T = p->n_trees, M = max_nodes_of(D);
  const bool logistic = p->objective == GBDT_OBJECTIVE_LOGISTIC;

  // ---- input checks (one synchronisation) ----
  std::vector<int32_t> hb(F);
  GBDT_CUDA(cudaMemcpyAsync(hb.data(), n_bins, sizeof(int32_t) * F, cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaMemsetAsync(w.err, 0, sizeof(int32_t), s));
  GBDT_CUDA(cudaMemsetAsync(w.nonfinite, 0, sizeof(int32_t), s));
  GBDT_CUDA(cudaMemsetAsync(split_counters(w.split_scratch, F, 1), 0, sizeof(int32_t) * kMaxSlots, s));
  launch_label_sum(label, N, w.label_partials, w.nonfinite, logistic, s);
  int32_t nonfinite = 0;
  GBDT_CUDA(cudaMemcpyAsync(&nonfinite, w.nonfinite, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  for (int j = 0; j < F; ++j)
    GBDT_CHECK_ARG(hb[j] >= 1 && hb[j] <= GBDT_MAX_BINS, "gbdt_train: n_bins[%d] = %d outside 1..256", j, hb[j]);
  if (nonfinite & 1) {
    set_error("gbdt_train: labels contain NaN or Inf");
    return GBDT_ERR_NONFINITE;
  }
  if (nonfinite & 2) {
    set_error("gbdt_train: the logistic objective needs labels 0 or 1");
    return GBDT_ERR_INVALID_ARG;
  }

  EventPool& pool = event_pool();
  const bool timing = diag != nullptr;
  // per tree and level: histogram start/end, partition start/end
  if (timing) GBDT_CUDA(pool.ensure(2 + 4 * static_cast<size_t>(T) * (D + 1)));
  auto ev_hist = [&](int t, int d, int k) { return pool.ev[2 + 4 * (static_cast<size_t>(t) * (D + 1) + d) + k]; };
  const int64_t launches0 = launch_count();
  if (timing) GBDT_CUDA(cudaEventRecord(pool.ev[0], s));

  launch_label_mean(w.label_partials, N, w.init, logistic, s);
  iota_kernel<<<sm_count() * 4, 256, 0, s>>>(w.orig0, N);
  count_launches();
  // the training levels read the bins in the row-block layout, features with at most 16 bins two per
  // byte (4-bit slots); the pair moves read them through tensor maps (one per buffer: the converted
  // input and the two alternating orders)
  std::vector<uint32_t> h_loc(F), h_src(F);
  // register slots (features of at most kRegMaxCodes codes accumulated in registers), squared error only
  int reg_begin = 0, reg_codes = 0;
  const bool regs = p->hist_registers == GBDT_HIST_REGISTERS_ON && !logistic;
  const int S = plan_row_block_slots_ex(hb.data(), F, p->bin_packing == GBDT_BIN_PACKING_4BIT, regs, h_loc.data(),
                                        h_src.data(), &reg_begin, &reg_codes);
  const int reg_arg = reg_begin < S ? reg_begin : -1;
  const int64_t pitch = rb_pitch(S);
  // the split search's feature schedule: a warp for each wide feature, a thread for each narrow one
  std::vector<int32_t> h_sched;
  h_sched.reserve(F);
  for (int j = 0; j < F; ++j)
    if (hb[j] > kSplitNarrowBins) h_sched.push_back(j);
  const int n_narrow = F - static_cast<int>(h_sched.size());
  for (int j = 0; j < F; ++j)
    if (hb[j] <= kSplitNarrowBins) h_sched.push_back(j);
  GBDT_CUDA(cudaMemcpyAsync(w.fsched, h_sched.data(), sizeof(int32_t) * F, cudaMemcpyHostToDevice, s));
  CUtensorMap maps[3];
  if (D >= 1) {
    GBDT_CUDA(cudaMemcpyAsync(w.floc, h_loc.data(), sizeof(uint32_t) * F, cudaMemcpyHostToDevice, s));
    GBDT_CUDA(cudaMemcpyAsync(w.slot_src, h_src.data(), sizeof(uint32_t) * S, cudaMemcpyHostToDevice, s));
    launch_cols_to_row_blocks(bins, ldb, N, S, w.slot_src, n_bins, w.bins_rb0, w.err, s);
    const uint8_t* bufs[3] = {w.bins_rb0, w.bins_xy[0], w.bins_xy[1]};
    for (int i = 0; i < 3; ++i) {
      rc = make_row_block_map(&maps[i], bufs[i], N, S);
      if (rc != GBDT_OK) return rc;
    }
  }
  // the work the histogram launch of level dn reads, prepared by the level above it (none past the last
  // histogram level)
  auto next_work = [&](int dn) {
    NextWork nw{};
    if (dn >= D) return nw;
    const int ms = 1 << dn;
    const SegHistPlan pl = plan_seg_histograms(N, S, ms, dn == 0 ? 1 : ms / 2, logistic, (dn & 1) != 0, reg_arg,
                                               reg_codes);
    nw.wv = seg_work_view(w.seg_scratch, ms);
    nw.max_ctas = pl.max_ctas;
    nw.min_rows = pl.min_rows;
    if (dn & 1) {
      nw.scan = w.scan;
      nw.filters = w.filters;
    }
    return nw;
  };
  const int fail_after = g_fail_after_levels.load();
  int levels_done = 0;
  // The launches of one tree on stream s.  Every kernel finds the tree it works on through the tree
  // index in device memory (budget[2], advanced by reset_root_kernel), so the sequence is the same for
  // every tree but the first (which counts the root's counts and keeps them) and the last (no next
  // gradients), and the trees between them replay it as one captured graph.
  // timing events recorded while a tree is captured become event-record nodes of its graph
  unsigned rec_flags = cudaEventRecordDefault;
  // The timing events hang off a stream of their own: at each mark it waits for the tree's stream and
  // records the event there, so in a replayed tree the event nodes are branches of the graph that no
  // kernel waits for; each tree ends by joining that stream back.
  struct Marks {
    cudaStream_t ts = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    Marks() = default;
    Marks(const Marks&) = delete;
    Marks& operator=(const Marks&) = delete;
    ~Marks() {
      if (fork) cudaEventDestroy(fork);
      if (join) cudaEventDestroy(join);
      if (ts) cudaStreamDestroy(ts);
    }
  } mk;
  if (timing) {
    GBDT_CUDA(cudaStreamCreateWithFlags(&mk.ts, cudaStreamNonBlocking));
    GBDT_CUDA(cudaEventCreateWithFlags(&mk.fork, cudaEventDisableTiming));
    GBDT_CUDA(cudaEventCreateWithFlags(&mk.join, cudaEventDisableTiming));
  }
  auto mark = [&](cudaEvent_t ev, cudaStream_t s) -> int {
    GBDT_CUDA(cudaEventRecord(mk.fork, s));
    GBDT_CUDA(cudaStreamWaitEvent(mk.ts, mk.fork, 0));
    GBDT_CUDA(cudaEventRecordWithFlags(ev, mk.ts, rec_flags));
    return GBDT_OK;
  };
  auto grow_tree = [&](int t, cudaStream_t s) -> int {
    launch_fixed_exp(w.maxabs, N, w.fixed_exp, logistic, s, /*clear=*/true);  // finish_tree raises them again
    reset_root_kernel<<<1, 1, 0, s>>>(w.level[0], w.build[0], w.seg[0], N, w.budget, next_work(0));
    count_launches();
    if (D == 0) {
      GBDT_CUDA(cudaMemsetAsync(w.totals[0], 0, sizeof(SlotTotals), s));
      root_totals_kernel<<<sm_count() * 4, 256, 0, s>>>(w.g0, N, w.fixed_exp, logistic ? 1 : 0, w.totals[0]);
      count_launches();
    }
    for (int d = 0; d <= D; ++d) {
      const int cur = d & 1, nxt = cur ^ 1;
      const bool odd = (d & 1) != 0;
      const int max_slots = 1 << d;
      LevelStats* st = w.stats + d;  // level d of tree 0: the kernel adds the tree's offset
      // Rows are partitioned every second level: levels 0 and 1 read the caller's order; after each
      // odd level the rows move straight into the order of the level below it.  At an odd level a
      // node's rows still sit in its pair's segment, and its histogram filters them by the parent's
      // split; its segment is where its rows will be once they move (a virtual segment).
      const int ph = d < 2 ? -1 : ((d >> 1) - 1) & 1;
      const uint8_t* lb = D == 0 ? bins : ph < 0 ? w.bins_rb0 : w.bins_xy[ph];
      const double* lg = ph < 0 ? w.g0 : w.g_xy[ph];
      const uint32_t* lo = ph < 0 ? w.orig0 : w.orig_xy[ph];
      if (d < D) {
        const int max_build = d == 0 ? 1 : max_slots / 2;
        const SegHistPlan plan = plan_seg_histograms(N, S, max_slots, max_build, logistic, odd, reg_arg, reg_codes);
        // a level's histograms start where the level above ended its partition (that event serves both)
        if (timing && d == 0 && (rc = mark(ev_hist(t, d, 0), s)) != GBDT_OK) return rc;
        const gbdt_segment* hseg = w.seg[cur];
        const gbdt_filter* hfil = nullptr;
        if (odd) {  // scan ranges and filters written by the level above (apply_level_kernel)
          hseg = w.scan;
          hfil = w.filters;
        }
        // the root's counts depend on the bins alone: the first tree counts them, the others copy them
        // and add only G (and H)
        rc = launch_seg_histograms(plan, lb, pitch, N, F, lg, GBDT_DTYPE_F64, w.fixed_exp, w.level[cur], max_slots,
                                   w.build[cur], hseg, hfil, w.seg_scratch, w.hist_cnt[cur], w.hist_q[cur],
                                   w.hist_h[cur], s, true, w.floc, w.slot_src,
                                   d == 0 && t > 0 ? w.root_cnt : nullptr, n_bins, /*work_ready=*/true);
        if (rc != GBDT_OK) return rc;
        if (timing && (rc = mark(ev_hist(t, d, 1), s)) != GBDT_OK) return rc;
        if (d == 0 && t == 0)
          GBDT_CUDA(cudaMemcpyAsync(w.root_cnt, w.hist_cnt[cur], sizeof(uint32_t) * F * kBins,
                                    cudaMemcpyDeviceToDevice, s));
        // past the root the larger child of each pair is its parent minus its built sibling, formed and
        // stored by the split search itself
        launch_find_splits(w.hist_cnt[cur], w.hist_q[cur], w.hist_h[cur], w.fixed_exp, F, n_bins, w.level[cur],
                           max_slots, *p, w.splits, w.split_scratch, w.err, s, w.fsched, n_narrow,
                           d > 0 ? w.totals[cur] : nullptr, d > 0 ? w.hist_cnt[nxt] : nullptr, w.hist_q[nxt],
                           w.hist_h[nxt], w.pair_parent[cur], w.build[cur]);
      }
      // the row launches after this level (below) find their tiles and pair records set up by the level
      // kernel itself
      RowsSetup rs{};
      if (d < D && d + 1 < D)
        rs = odd ? rows_setup_pairs(w.move_scratch, N, max_slots, true, w.route[nxt], w.pair_parent[cur], w.floc)
                 : rows_setup_slot_tiles(w.move_scratch, N, max_slots);
      else if (d + 1 == D && odd)
        rs = rows_setup_pairs(w.move_scratch, N, max_slots, false, w.route[nxt], w.pair_parent[cur], w.floc);
      else if (d + 1 == D || D == 0)
        rs = rows_setup_slot_tiles(w.move_scratch, N, max_slots);
      apply_level_kernel<<<1, 1024, 0, s>>>(d, D, w.level[cur], max_slots, d < D ? w.splits : nullptr, w.totals[cur],
                                            w.build[cur], w.fixed_exp, p->reg_lambda, w.seg[cur], w.trees,
                                            w.n_nodes, w.level[nxt], w.totals[nxt], w.seg[nxt],
                                            w.pair_parent[nxt], w.build[nxt], w.route[cur], st, p->num_leaves,
                                            w.budget, logistic ? 1 : 0, w.err, next_work(d + 1), rs);
      count_launches();
      // rows: after an odd level they move into the next order (four grandchild runs per pair); at
      // even levels nothing moves and the rows of nodes that do not split record their leaf; at the
      // last split level every row records its leaf.
      // the last level of a tree partitions nothing: no events around it
      const bool part_events = timing && (d < D || D == 0);
      if (part_events && (rc = mark(ev_hist(t, d, 2), s)) != GBDT_OK) return rc;
      if (d < D && d + 1 < D) {
        if (odd) {
          const int out = ((d + 1) >> 1) - 1 & 1;
          launch_move_pairs(maps[ph + 1], lb, w.bins_xy[out], pitch, w.floc, N, S, lg, w.g_xy[out], lo,
                            w.orig_xy[out],
                            w.level[cur], max_slots, w.seg[cur], w.route[cur], w.route[nxt], w.pair_parent[cur],
                            w.seg[nxt], w.leaf, w.move_scratch, w.err, s, /*setup_done=*/true);
        } else {
          launch_leaf_rows(lb, pitch, w.floc, N, lo, w.level[cur], max_slots, w.seg[cur], w.route[cur], true, w.leaf,
                           w.move_scratch, s, /*setup_done=*/true);
        }
      } else if (d + 1 == D && odd) {
        launch_leaf_pairs(lb, pitch, w.floc, N, lo, w.level[cur], max_slots, w.seg[cur], w.route[cur], w.route[nxt],
                          w.pair_parent[cur], w.seg[nxt], w.leaf, w.move_scratch, s, /*setup_done=*/true);
      } else if (d + 1 == D || D == 0) {
        launch_leaf_rows(lb, pitch, w.floc, N, lo, w.level[cur], max_slots, w.seg[cur], w.route[cur], false, w.leaf,
                         w.move_scratch, s, /*setup_done=*/true);
      }
      if (part_events && (rc = mark(ev_hist(t, d, 3), s)) != GBDT_OK) return rc;
      GBDT_LAUNCH_CHECK();
      ++levels_done;
      if (fail_after >= 0 && levels_done >= fail_after) {
        cudaStreamSynchronize(s);
        set_error("gbdt_train: failure injected after %d levels", levels_done);
        return GBDT_ERR_INTERNAL;
      }
    }
    const bool next = t + 1 < T;  // maxabs was cleared by this tree's fixed_exp launch
    launch_finish_tree(w.trees, w.n_nodes, w.budget + 2, M, p->learning_rate, label, N, p->objective, pred_out,
                       w.g0, w.leaf, w.maxabs, next, s);
    GBDT_LAUNCH_CHECK();
    if (timing) {  // the timing stream joins the tree's stream (a captured tree must end joined)
      GBDT_CUDA(cudaEventRecord(mk.join, mk.ts));
      GBDT_CUDA(cudaStreamWaitEvent(s, mk.join, 0));
    }
    return GBDT_OK;
  };

  GBDT_CUDA(cudaMemsetAsync(w.budget + 2, 0xff, sizeof(int32_t), s));  // tree index -1
  // Trees 1 .. T - 2 as one graph, captured once per call: a tree is a chain of dependent launches,
  // and a graph replay shortens the gap between each and the next.  With diagnostics the per-level
  // timing events are nodes of the graph, pointed at each tree's events before its replay.
  // Failure-injection runs launch tree by tree.
  const bool use_graph = fail_after < 0 && T >= 4;
  TreeGraph tg;
  for (int t = 0; t < T; ++t) {
    if (t == 0) {
      GBDT_CUDA(cudaMemsetAsync(w.maxabs, 0, 2 * sizeof(unsigned long long), s));
      launch_start_tree0(w.init, label, N, p->objective, pred_out, w.g0, w.leaf, w.maxabs, s);
    }
    if (use_graph && t >= 1 && t + 1 < T) {
      if (tg.exec == nullptr) {
        rec_flags = cudaEventRecordExternal;
        rc = tg.capture([&](cudaStream_t cs) { return grow_tree(t, cs); });
        rec_flags = cudaEventRecordDefault;
        if (rc != GBDT_OK) return rc;
      }
      for (size_t i = 0; i < tg.marks.size(); ++i) {  // this tree's timing events (captured as tree t0's)
        const int t0 = 1;
        int slot = -1;
        for (int d = 0; d <= D && slot < 0; ++d)
          for (int k = 0; k < 4; ++k)
            if (tg.mark_events[i] == ev_hist(t0, d, k)) slot = 4 * d + k;
        if (slot < 0) {
          set_error("gbdt_train: an event of the tree graph is not a timing event");
          return GBDT_ERR_INTERNAL;
        }
        GBDT_CUDA(cudaGraphExecEventRecordNodeSetEvent(tg.exec, tg.marks[i], ev_hist(t, slot / 4, slot % 4)));
      }
      GBDT_CUDA(cudaGraphLaunch(tg.exec, s));
      count_launches(static_cast<int>(tg.launches));
      continue;
    }
    rc = grow_tree(t, s);
    if (rc != GBDT_OK) return rc;
  }
  if (T == 0) {
    // no tree: predictions are the initial value
    GBDT_CUDA(cudaMemsetAsync(w.maxabs, 0, 2 * sizeof(unsigned long long), s));
    launch_start_tree0(w.init, label, N, p->objective, pred_out, w.g0, w.leaf, w.maxabs, s);
  }
  if (timing) GBDT_CUDA(cudaEventRecord(pool.ev[1], s));

  // ---- one copy of the finished model ----
  std::vector<gbdt_node> h_nodes(static_cast<size_t>(T) * M);
  std::vector<int32_t> h_n(T > 0 ? T : 1);
  std::vector<LevelStats> h_stats(static_cast<size_t>(T) * (D + 1) + 1);
  int32_t h_err = 0;
  double h_init = 0.0;
  if (T > 0) {
    GBDT_CUDA(cudaMemcpyAsync(h_nodes.data(), w.trees, sizeof(gbdt_node) * h_nodes.size(), cudaMemcpyDeviceToHost, s));
    GBDT_CUDA(cudaMemcpyAsync(h_n.data(), w.n_nodes, sizeof(int32_t) * T, cudaMemcpyDeviceToHost, s));
    GBDT_CUDA(cudaMemcpyAsync(h_stats.data(), w.stats, sizeof(LevelStats) * T * (D + 1), cudaMemcpyDeviceToHost, s));
  }
  GBDT_CUDA(cudaMemcpyAsync(&h_err, w.err, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaMemcpyAsync(&h_init, w.init, sizeof(double), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (h_err & kErrBinRange) {
    set_error("gbdt_train: a bin is not below its feature's n_bins");
    return GBDT_ERR_INVALID_ARG;
  }
  if (h_err != 0) {
    set_error("gbdt_train: device consistency check failed (error bits 0x%x)", h_err);
    return GBDT_ERR_INTERNAL;
  }
  for (int t = 0; t < T; ++t) {
    if (h_n[t] < 1 || h_n[t] > M) {
      set_error("gbdt_train: tree %d has an invalid node count %d", t, h_n[t]);
      return GBDT_ERR_INTERNAL;
    }
    const gbdt_node* tn = h_nodes.data() + static_cast<size_t>(t) * M;
    for (int i = 0; i < h_n[t]; ++i) {  // "Validate all indices on creation" (s.3)
      const gbdt_node& nd = tn[i];
      const bool ok = nd.is_leaf ? (nd.left == -1 && nd.right == -1 && nd.feature == -1)
                                 : (nd.left > i && nd.right == nd.left + 1 && nd.right < h_n[t] && nd.feature >= 0 &&
                                    nd.feature < F && nd.threshold_bin >= 0 && nd.threshold_bin < GBDT_MAX_BINS);
      if (!ok) {
        set_error("gbdt_train: tree %d node %d failed index validation", t, i);
        return GBDT_ERR_INTERNAL;
      }
    }
  }
  // success: publish the model
  for (int t = 0; t < T; ++t) {
    std::copy(h_nodes.begin() + static_cast<size_t>(t) * M, h_nodes.begin() + static_cast<size_t>(t) * M + h_n[t],
              nodes_out + static_cast<size_t>(t) * M);
    nodes_per_tree[t] = h_n[t];
  }
  *init_pred_out = h_init;
  if (timing) {
    gbdt_diagnostics dg{};
    float ms = 0.f;
    GBDT_CUDA(cudaEventElapsedTime(&ms, pool.ev[0], pool.ev[1]));
    dg.total_ms = ms;
    const double row_bytes = static_cast<double>(S) + 8.0;       // a scanned row: bins (slots) + fp64 g
    const double move_bytes = 2.0 * (S + 8.0 + 4.0);             // a moved row: read + write every slot
    for (int t = 0; t < T; ++t) {
      for (int d = 0; d <= D; ++d) {
        const LevelStats& ls = h_stats[static_cast<size_t>(t) * (D + 1) + d];
        const bool odd = (d & 1) != 0;
        if (d < D) {
          GBDT_CUDA(cudaEventElapsedTime(&ms, d == 0 ? ev_hist(t, 0, 0) : ev_hist(t, d - 1, 3), ev_hist(t, d, 1)));
          dg.hist_ms += ms;
          dg.hist_launches += 1;
          dg.hist_rows += ls.n_built_rows;
          const double out_bytes = static_cast<double>(ls.n_built) * F * kBins * (logistic ? 20.0 : 12.0);
          dg.hist_bytes += static_cast<double>(ls.n_scan_rows) * (row_bytes + (odd ? 1.0 : 0.0)) + out_bytes;
          dg.hist_level_bytes += static_cast<double>(ls.n_act) * (F + 8.0 + 2.0) + out_bytes;
        }
        if (d == D && D > 0) continue;  // nothing partitioned (no events recorded)
        GBDT_CUDA(cudaEventElapsedTime(&ms, ev_hist(t, d, 2), ev_hist(t, d, 3)));
        dg.part_ms += ms;
        // a moved row reads and writes every column and its two decision bytes are read; a row that
        // records its leaf reads its row id (and its decision bytes) and writes a 2-byte leaf id
        const double split = static_cast<double>(ls.n_split_rows), frozen = static_cast<double>(ls.n_act) - split;
        if (d + 1 < D) {
          dg.part_bytes += odd ? split * (move_bytes + 2.0) + frozen * 7.0 : frozen * 6.0;
        } else if (d + 1 == D) {
          dg.part_bytes += odd ? static_cast<double>(ls.n_act) * 8.0 : split * 7.0 + frozen * 6.0;
        } else if (D == 0) {
          dg.part_bytes += static_cast<double>(ls.n_act) * 6.0;
        }
      }
      if (h_n[t] == M) dg.trees_at_full_size += 1;
    }
    dg.kernel_launches = launch_count() - launches0;
    *diag = dg;
  }
  return GBDT_OK;
}
