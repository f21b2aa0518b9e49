// Internal launchers shared between the entry points and the training driver.
#pragma once

#include "common.cuh"

namespace gbdt {

// ---- gradients.cu -------------------------------------------------------------------
// Deterministic mean of labels: fixed grid, fixed reduction order.
constexpr int kSumBlocks = 512;
constexpr int kSumThreads = 256;
// nonfinite: bit 1 for a NaN/Inf label; with binary, bit 2 for a label other than 0 or 1.
void launch_label_sum(const float* label, int64_t N, double* partials /*[kSumBlocks]*/, int32_t* nonfinite,
                      bool binary, cudaStream_t s);
// *init = mean(label), or 0 with zero (the logistic objective's initial margin).
void launch_label_mean(const double* partials, int64_t N, double* init /*device*/, bool zero, cudaStream_t s);
// pred = *init; g = gradient of the objective at pred; node = 0; maxabs[0] = max |g| and, for the
// logistic objective, maxabs[1] = max h (maxabs must be reset to 0 first).
void launch_start_tree0(const double* init, const float* label, int64_t N, int32_t objective, double* pred,
                        double* g, uint16_t* node, unsigned long long* maxabs /*[2]*/, cudaStream_t s);
// pred += lr * leaf_value(node); if next: g at the new pred, node = 0, maxabs as launch_start_tree0.
// trees / n_nodes: per-tree arrays (max_nodes nodes per tree); the tree is the one *tree_index names
// (device memory), so the launch is the same for every tree.
void launch_finish_tree(const gbdt_node* trees, const int32_t* n_nodes, const int32_t* tree_index,
                        int32_t max_nodes, double lr, const float* label, int64_t N, int32_t objective, double* pred,
                        double* g, uint16_t* node, unsigned long long* maxabs, bool next, cudaStream_t s);
void launch_gradients(const double* pred, const float* label, int64_t N, int32_t objective, double* g,
                      unsigned long long* maxabs, cudaStream_t s);
void launch_maxabs(const void* g, int32_t dtype, int64_t N, unsigned long long* maxabs, cudaStream_t s);
// fixed_exp[0] from maxabs[0]; with_h: fixed_exp[1] from maxabs[1]; clear: maxabs reset to 0 after it is read.
void launch_fixed_exp(unsigned long long* maxabs, int64_t N, int32_t* fixed_exp, bool with_h, cudaStream_t s,
                      bool clear = false);

// ---- histogram.cu ---------------------------------------------------------------------
struct HistPlan {
  int group_slots;  // built slots per CTA
  int group_feats;  // features per CTA
  int n_sgroups, n_fgroups, n_chunks;
  int64_t rows_per_chunk;
  size_t smem;
  int blocks() const { return n_sgroups * n_fgroups * n_chunks; }
};
HistPlan plan_histograms(int64_t N, int32_t F, int32_t max_slots, int32_t max_build);
// Zeroes the flagged slots of hist_cnt/hist_q (and hist_h when not null); cnt0 (not null): slot 0's
// counts are copied from cnt0 ([F][256]) instead.  n_bins (not null): only each feature's bins below
// its n_bins (the training's histograms, whose other bins no pass writes or reads).
void launch_hist_zero(const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag, int32_t F,
                      uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, cudaStream_t s,
                      const uint32_t* cnt0 = nullptr, const int32_t* n_bins = nullptr);
int launch_hist_build(const HistPlan& plan, const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g,
                      int32_t g_dtype, const int32_t* fixed_exp, const uint16_t* node_of_row,
                      const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag, uint32_t* hist_cnt,
                      int64_t* hist_q, int32_t* err, cudaStream_t s);
// prev_h/hist_h: both null, or the H histograms subtracted likewise.  n_bins (not null): only each
// feature's bins below its n_bins.
void launch_hist_subtract(const uint32_t* prev_cnt, const int64_t* prev_q, const int64_t* prev_h,
                          const int32_t* pair_parent, const uint8_t* build_flag, const gbdt_level* level,
                          int32_t max_slots, int32_t F, uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h,
                          int32_t* err, cudaStream_t s, const int32_t* n_bins = nullptr);

// ---- grouping.cu -----------------------------------------------------------------------
// Rows of a level's built slots copied, grouped by slot, into a row-block buffer rb (pitch
// rb_pitch(F)) and a gradient buffer g_out (g_size bytes per row): slot s's rows are positions
// seg[s].start .. + seg[s].count (start a multiple of 32; unbuilt slots get count 0), in no set order.
// count, cursor: [max_slots] scratch.  Buffers hold group_rows_capacity(N, max_slots) rows.
size_t group_rows_capacity(int64_t N, int32_t max_slots);
size_t group_rows_smem_bytes(int32_t max_slots);
void launch_group_rows(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g, int g_size,
                       const uint16_t* node, const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag,
                       uint32_t* count, uint32_t* cursor, gbdt_segment* seg, uint8_t* rb, void* g_out,
                       int32_t* err, cudaStream_t s);

// ---- split.cu -------------------------------------------------------------------------
// A slot's totals: fixed-point G, fixed-point H (logistic; else 0) and the row count.
struct SlotTotals {
  int64_t q;
  int64_t qh;  // logistic: fixed-point H (exponent fixed_exp[1]); else 0
  uint32_t cnt;
  uint32_t pad;
};
size_t find_splits_scratch_bytes(int32_t F, int32_t max_slots);
// The per-slot counters inside that scratch: zero them before the first launch_find_splits on it
// (every launch leaves them zero again).
int32_t* split_counters(void* scratch, int32_t F, int32_t max_slots);
// hist_h: null (H = count) or the H histograms with exponent fixed_exp[1].  fsched (device, may be null):
// the features whose n_bins is above kSplitNarrowBins first, then the n_narrow others, each of which one
// thread searches alone; null: a warp per feature, in order.  totals (device, may be null): each slot's
// expected totals (the parent split's sides), which every feature's histogram must sum to; null: the
// totals are summed from feature 0's histogram.  prev_cnt (device, may be null): the previous level's
// histograms (prev_q, prev_h), pair_parent and build_flag of this level: each slot not built is formed
// as its parent's histogram minus its built sibling's, searched and stored (the sibling subtraction
// fused into the search); null: every slot's histogram is in place.
constexpr int kSplitNarrowBins = 8;
void launch_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int64_t* hist_h,
                        const int32_t* fixed_exp, int32_t F, const int32_t* n_bins, const gbdt_level* level,
                        int32_t max_slots, const gbdt_params& p, gbdt_split* out, void* scratch, int32_t* err,
                        cudaStream_t s, const int32_t* fsched = nullptr, int32_t n_narrow = 0,
                        const SlotTotals* totals = nullptr, const uint32_t* prev_cnt = nullptr,
                        const int64_t* prev_q = nullptr, const int64_t* prev_h = nullptr,
                        const int32_t* pair_parent = nullptr, const uint8_t* build_flag = nullptr);

// ---- partition.cu ---------------------------------------------------------------------
// Routing entry of a slot: split feature (-1: none), threshold bin, left child node id.
struct Route {
  int32_t feature;
  int32_t bin;
  int32_t left_node;
  int32_t pad;
};
// ---- segments.cu ----------------------------------------------------------------------
// Register groups of a histogram launch: the slots from reg_begin on hold features of at most
// kRegMaxCodes codes (one with at most 8 bins, or a 4-bit pair whose bin counts multiply to at most 8);
// they form groups of 32 after the n_norm_groups ordinary ones, and accumulate in registers.
constexpr int kRegMaxCodes = 8;
struct RegGroups {
  int32_t reg_begin;      // S when there are none
  int32_t n_norm_groups;  // ordinary groups (they come first in grid.y)
  int32_t weight;         // a register group's share weight
  int32_t codes;          // codes a register lane keeps: 4 or 8
  const int32_t* n_bins;  // device [F]
};
// Histograms of the flagged slots of a level whose rows are contiguous segments.
struct SegHistPlan {
  int n_cols;        // columns the lanes read: slots of the row blocks (features in the column layout)
  int n_fgroups, group_feats;  // groups of columns (full groups of group_feats and the remainder)
  int row_weight;    // a group's weight is its 32-lane halves + row_weight (see seg_hist_kernel)
  int total_weight;  // sum over groups of (32-lane halves + row_weight)
  int sm_budget;     // CTAs of one wave, shared by the groups in proportion to their weights
  int max_ctas;      // CTAs of a full group
  int64_t min_rows;  // least work (rows + a fixed cost per slot) a CTA takes when the level is small
  bool with_h;       // logistic: H histograms too (h = logistic_hess(g), exponent fixed_exp[1])
  size_t smem;
  int reg_begin;     // first register slot (S: none)
  int n_norm_groups; // ordinary groups
  int reg_weight;    // share weight of a register group
  int reg_codes;     // codes per register lane (4 or 8)
};
// The histogram work of a level is cut by cost: every built slot costs its rows plus kSlotCost, the
// fixed work of taking up a slot (the dependent loads of its first rows, two barriers and the flush of
// the CTA's shared histograms, about what 128 rows of updates take).  Cutting by rows alone put a run
// of many tiny slots (deep levels) on one CTA, which then took them one by one.
constexpr int64_t kSlotCost = 128;
// The work list a level's histogram launch reads: the built slots with their rows in slot order.
struct SegWork {
  int64_t total_rows;  // rows over all built slots
  int64_t total_cost;  // total_rows + kSlotCost x n_built
  int32_t n_built;     // built slots
  int32_t ctas;        // CTAs per feature group that have work (at most max_ctas, at least min_rows of cost each)
};
struct SegWorkView {
  SegWork* st;
  int32_t* build_slot;  // [max_slots + 1]: the k-th built slot
  int64_t* row_start;   // [max_slots + 1]: rows of the built slots before the k-th (the total at n_built)
};
// Where the work list of a level of max_slots slots sits in seg_hist_scratch_bytes(max_slots) of scratch.
SegWorkView seg_work_view(void* scratch, int32_t max_slots);
// launch_hist_zero for the slots of a level's work list (st->n_built of them, build_slot[k]), at most
// max_built: a CTA row per built slot instead of per slot.
void launch_hist_zero_built(const SegWork* st, const int32_t* build_slot, int32_t max_built, int32_t F,
                            uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, cudaStream_t s,
                            const uint32_t* cnt0, const int32_t* n_bins);
// S: the columns the lanes read (slots of the row blocks; F in the column layout).
// filtered: the level's slots are counted through filters (a node's rows inside its pair's segment).
// reg_begin >= 0: slots from reg_begin on are register slots of at most reg_codes codes (squared error only).
SegHistPlan plan_seg_histograms(int64_t N, int32_t S, int32_t max_slots, int32_t max_build, bool with_h = false,
                                bool filtered = false, int32_t reg_begin = -1, int32_t reg_codes = 0);
size_t seg_hist_scratch_bytes(int32_t max_slots);
int launch_seg_histograms(const SegHistPlan& plan, const uint8_t* bins, int64_t ldb, int64_t N, int32_t F,
                          const void* g, int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                          int32_t max_slots, const uint8_t* build_flag, const gbdt_segment* seg,
                          const gbdt_filter* filters, void* scratch, uint32_t* hist_cnt, int64_t* hist_q,
                          int64_t* hist_h, cudaStream_t s, bool row_blocks = false, const uint32_t* floc = nullptr,
                          const uint32_t* slot_src = nullptr, const uint32_t* root_cnt = nullptr,
                          const int32_t* n_bins = nullptr, bool work_ready = false);
// With register groups in the plan, n_bins (device) must be given.
// row_blocks: ldb is the row-block pitch, floc the feature locators and slot_src each slot's features
// (plan_row_block_slots; null: slot s holds feature s); a lane accumulates its slot's byte, the joint
// code of a 4-bit slot, and the flush splits it into the two features' bins.  hist_h: plan.with_h.
// root_cnt (row blocks, fp64 g, a one-slot level only): the slot's count histogram [F][256], known
// beforehand (the root's counts depend on the bins alone); it is copied in and the kernel adds only
// G (and H), one shared atomic fewer per row and slot.
// Stable partition of the per-position data of every split slot (bins columns, g, original row
// id) from *_in to *_out; slots without a split record leaf_of_row[orig] = their node id.
size_t move_scratch_bytes(int64_t N, int32_t max_slots);
void launch_move_rows(const uint8_t* bins_in, uint8_t* bins_out, int64_t ldb, int64_t N, int32_t F,
                      const void* g_in, void* g_out, int g_size, const uint32_t* orig_in, uint32_t* orig_out,
                      const uint8_t* go_right, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, const gbdt_split* splits, gbdt_segment* seg_out,
                      uint16_t* leaf_of_row, void* scratch, int32_t* err, cudaStream_t s);
// ---- training-internal row-block layout (see rb_offset, and loc_slot for 4-bit slots) ----
// Bytes of a row-block copy of N rows x S slots, and the conversion from the column layout:
// slot_src (null: slot s holds feature s) from plan_row_block_slots; with n_bins every bin of the
// N rows is checked against its feature's n_bins (kErrBinRange in err).
size_t row_block_bytes(int64_t N, int32_t S);
void launch_cols_to_row_blocks(const uint8_t* cols, int64_t ldb, int64_t N, int32_t S, const uint32_t* slot_src,
                               const int32_t* n_bins, uint8_t* rb, int32_t* err, cudaStream_t s);
// Host: the slots of a row-block copy.  With pack, features with n_bins <= 16 pair up in feature order
// (the first of a pair in the low nibble, an unpaired one keeps a whole byte); every other feature has a
// slot of its own.  Writes loc[F] (locators) and src[S] (per slot: first feature | second << 16, second
// 0xffff for a whole-byte slot); returns S.
int plan_row_block_slots(const int32_t* n_bins, int32_t F, bool pack, uint32_t* loc, uint32_t* src);
// The same with register slots (regs): features with at most kRegMaxCodes bins are taken out of the
// ordinary plan and placed after it, paired in feature order when pack is on and the two bin counts
// multiply to at most kRegMaxCodes; *reg_begin receives the first register slot (S: none) and *reg_codes
// the most codes of a register slot.
int plan_row_block_slots_ex(const int32_t* n_bins, int32_t F, bool pack, bool regs, uint32_t* loc, uint32_t* src,
                            int* reg_begin, int* reg_codes);
// The tensor map the pair move reads a row-block buffer of S slots through.
int make_row_block_map(CUtensorMap* map, const uint8_t* rb, int64_t N, int32_t S);
// Record leaves without moving data: every row of the level (its child when its slot splits, its
// own node when it does not), or with frozen_only only the rows of slots that do not split.  Needs
// route from the level's splits; bins in the row-block layout; scratch is move_scratch_bytes.
// setup_done: the kernel before has done rows_setup_slot_tiles' setup (rows.cuh) on this scratch; the
// same holds for the two pair launchers below with rows_setup_pairs.
void launch_leaf_rows(const uint8_t* bins_rb, int64_t pitch, const uint32_t* floc, int64_t N,
                      const uint32_t* orig_in, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, bool frozen_only, uint16_t* leaf_of_row, void* scratch, cudaStream_t s,
                      bool setup_done = false);
// Odd level, after its splits: move the rows of every sibling pair (still in their parent's order)
// straight into the next level's order (four grandchild runs per pair); rows of children that do not
// split record them as their leaf.  route_prev/pair_parent: the level above; seg_next: the next
// level's segments.  Bins in the row-block layout, read through map_in (make_row_block_map of
// bins_rb_in, S slots; floc the feature locators); g is fp64.  Scratch: move_scratch_bytes(N, max_slots).
void launch_move_pairs(const CUtensorMap& map_in, const uint8_t* bins_rb_in, uint8_t* bins_rb_out, int64_t pitch,
                       const uint32_t* floc, int64_t N, int32_t S, const double* g_in, double* g_out,
                       const uint32_t* orig_in, uint32_t* orig_out, const gbdt_level* level, int32_t max_slots,
                       const gbdt_segment* seg, const Route* route_cur, const Route* route_prev,
                       const int32_t* pair_parent, const gbdt_segment* seg_next, uint16_t* leaf_of_row, void* scratch,
                       int32_t* err, cudaStream_t s, bool setup_done = false);
// Odd last split level: every row of every pair records its leaf; nothing moves.
void launch_leaf_pairs(const uint8_t* bins_rb, int64_t pitch, const uint32_t* floc, int64_t N,
                       const uint32_t* orig_in, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                       const Route* route_cur, const Route* route_prev, const int32_t* pair_parent,
                       const gbdt_segment* seg_next, uint16_t* leaf_of_row, void* scratch, cudaStream_t s,
                       bool setup_done = false);

// node_of_row[r] = left_node + (bins[feature][r] > bin) for rows of slots with a split.
void launch_route_rows(const uint8_t* bins, int64_t ldb, int64_t N, const Route* route, const gbdt_level* level,
                       int32_t max_slots, uint16_t* node_of_row, int32_t* err, cudaStream_t s);

}  // namespace gbdt
