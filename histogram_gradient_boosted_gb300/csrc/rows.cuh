// Bookkeeping of the row launches that follow a level's splits (recording leaves, moving sibling pairs),
// shared by the move kernels (segments.cu) and the level kernel (train.cu), which does this setup itself
// at its end so that no separate one-CTA launch sits between it and the row launches.
#pragma once

#include "kernels.cuh"

namespace gbdt {

constexpr int kMvTile = 4096;  // positions per tile

struct MvState {
  int32_t total_tiles;
  int32_t pad;
};

struct PairRoute {
  int64_t start, count;  // the pair's rows (both children) in the current order
  int64_t dst[4];        // first position of each grandchild in the next order
  int64_t want[4];       // its row count from the split records; -1: its child does not split
  int32_t f1, b1;        // the parent's split (f1: its feature's locator): which child a row belongs to
  int32_t f2[2], b2[2];  // the children's splits (locators); f2 < 0: the child is a leaf
  int32_t node[2];       // the children's node ids
  int32_t left[2];       // node id of each child's left child
};

struct PairState {
  int32_t n_pairs;
  int32_t total_tiles;
};

// Tiles per slot of the level, every slot (split slots are moved, the others have their rows recorded
// as leaves): tile_start[s] = the slot's first tile, st->total_tiles.  One CTA; every thread calls it.
__device__ __forceinline__ void rows_slot_tiles(const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                                                int32_t* tile_start, MvState* st) {
  __shared__ int s_w[33];
  int s_pre = 0;  // block-uniform running total
  const int n_slots = min(level->n_slots, max_slots);
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const int tiles = s < n_slots ? static_cast<int>((seg[s].count + kMvTile - 1) / kMvTile) : 0;
    int n;
    const int e = block_scan_excl(tiles, s_w, &n);
    if (s < n_slots) tile_start[s] = s_pre + e;
    s_pre += n;
  }
  if (threadIdx.x == 0) {
    tile_start[n_slots] = s_pre;
    st->total_tiles = s_pre;
  }
}

// Per sibling pair of an odd level (slots 2k and 2k + 1): its rows, both levels' splits and the
// grandchildren's places in the next order (pairs[k]), its first tile (tile_start[k]), and st.  level,
// seg, route_cur: this level; route_prev, pair_parent: the level above; seg_next: the next level.
// tile_status[0 .. n_status): the look-back status words of the move that follows, zeroed (null: no
// move follows).  One CTA; every thread calls it.  route_cur and seg_next may have been written by the
// calling kernel before a barrier, so they are read with ordinary loads.
__device__ __forceinline__ void rows_pair_routes(const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                                                 const Route* route_cur, const Route* route_prev,
                                                 const int32_t* pair_parent, const gbdt_segment* seg_next,
                                                 const uint32_t* floc, PairRoute* pairs, int32_t* tile_start,
                                                 PairState* st, unsigned long long* tile_status, int32_t n_status) {
  __shared__ int s_w[33];
  for (int i = threadIdx.x; i < n_status; i += blockDim.x) tile_status[i] = 0;
  int s_pre = 0;  // block-uniform running total
  const int n_pairs = min(level->n_slots, max_slots) / 2;
  for (int c0 = 0; c0 < n_pairs; c0 += blockDim.x) {
    const int k = c0 + threadIdx.x;
    int tiles = 0;
    if (k < n_pairs) {
      PairRoute pr;
      const Route up = route_prev[pair_parent[k]];
      pr.f1 = static_cast<int32_t>(floc ? floc[up.feature] : up.feature), pr.b1 = up.bin;
      pr.start = seg[2 * k].start;
      pr.count = seg[2 * k].count + seg[2 * k + 1].count;
      for (int c = 0; c < 2; ++c) {
        const Route rt = route_cur[2 * k + c];
        pr.node[c] = level->node_begin + 2 * k + c;
        pr.f2[c] = rt.feature < 0 ? -1 : static_cast<int32_t>(floc ? floc[rt.feature] : rt.feature);
        pr.b2[c] = rt.bin, pr.left[c] = rt.left_node;
        for (int j = 0; j < 2; ++j) {
          if (rt.feature >= 0) {
            const gbdt_segment g2 = seg_next[2 * rt.pad + j];
            pr.dst[2 * c + j] = g2.start, pr.want[2 * c + j] = g2.count;
          } else {
            pr.dst[2 * c + j] = 0, pr.want[2 * c + j] = -1;
          }
        }
      }
      pairs[k] = pr;
      tiles = static_cast<int>((pr.count + kMvTile - 1) / kMvTile);
    }
    int n;
    const int e = block_scan_excl(tiles, s_w, &n);
    if (k < n_pairs) tile_start[k] = s_pre + e;
    s_pre += n;
  }
  if (threadIdx.x == 0) {
    tile_start[n_pairs] = s_pre;
    st->n_pairs = n_pairs;
    st->total_tiles = s_pre;
  }
}

// The setup the level kernel does for the row launches that follow it (kind kRowsNone: none).
enum : int32_t { kRowsNone = 0, kRowsSlotTiles = 1, kRowsPairRoutes = 2 };
struct RowsSetup {
  int32_t kind;
  int32_t n_status;  // kRowsPairRoutes: status words to zero (0 when no move follows)
  MvState* mv_st;    // kRowsSlotTiles
  int32_t* mv_tile_start;
  PairRoute* pairs;  // kRowsPairRoutes
  int32_t* pair_tile_start;
  PairState* pair_st;
  unsigned long long* tile_status;
  const Route* route_prev;
  const int32_t* pair_parent;
  const uint32_t* floc;
};

// The setup for launch_leaf_rows over move scratch (move_scratch_bytes(N, max_slots)).
RowsSetup rows_setup_slot_tiles(void* scratch, int64_t N, int32_t max_slots);
// The setup for launch_move_pairs (move true) or launch_leaf_pairs over move scratch.
RowsSetup rows_setup_pairs(void* scratch, int64_t N, int32_t max_slots, bool move, const Route* route_prev,
                           const int32_t* pair_parent, const uint32_t* floc);

}  // namespace gbdt
