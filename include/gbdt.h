/*
 * gbdt.h -- C ABI of the GB300 (sm_103a) level-wise histogram GBDT library.
 *
 * The library trains gradient-boosted decision trees with the squared-error
 * objective (or, as an option, the logistic one), growing each tree level by
 * level over uint8-binned features.
 * Its entry points follow the ComputeBackend contract of "Module Design:
 * Training Core" (MPSBoost spec), s.4 Backend Interface: the caller passes
 * plain views and preallocated outputs, the core decides when to call, the
 * backend decides how to compute; split search and partition are exposed as
 * the "fine-grained capability interfaces" that section anticipates.
 *
 * Conventions for every entry point
 *   - Return value: GBDT_OK (0) or a negative GBDT_ERR_* code; on error
 *     gbdt_last_error() returns a message for the calling thread.
 *   - Array arguments are DEVICE pointers owned by the caller unless the
 *     comment says "host".  The library allocates no memory: scratch space is
 *     the caller's workspace `ws` of `ws_bytes` bytes, sized by the matching
 *     *_workspace_size function; too small a workspace gives
 *     GBDT_ERR_WORKSPACE.  Workspace pointers must be 256-byte aligned.
 *   - Work is queued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream), except where a function says
 *     it synchronises.
 *   - Arguments are validated before any launch; an invalid argument returns
 *     GBDT_ERR_INVALID_ARG and queues nothing.
 *   - Consistency checks that only the device can make (a histogram that does
 *     not add up to its node's totals, a partition whose counts differ from
 *     its split records, a level larger than its bound; "Module Design:
 *     Training Core" s.5, the Failed state) are recorded in a device error
 *     word.  Every asynchronous call that takes a workspace keeps that word in
 *     the workspace's first 4 bytes: the call clears it when it is queued and
 *     its kernels OR error bits into it, so after the call the word describes
 *     that call.  gbdt_workspace_status reads it back; gbdt_train and
 *     gbdt_quantize read their own and return the error themselves.  A caller
 *     that never asks does not pay for the check (no synchronisation).
 *   - Binned features are column-major uint8: feature j occupies
 *     bins[j*ldb .. j*ldb + N); ldb >= N, ldb % 16 == 0 and the base pointer
 *     16-byte aligned, so every column is read with 16-byte vector loads.
 *     Bytes N..ldb-1 of a column are never interpreted.
 *   - Gradients are accumulated in histograms as exact 64-bit fixed point:
 *     q = round-half-even(g * 2^S) with one exponent S per call sequence
 *     (gbdt_gradient_scale), so histogram sums are independent of thread
 *     order and sibling subtraction is exact.  For squared error H is the row
 *     count (h = 1), so no H array is stored.  For the logistic objective H
 *     has its own fixed-point histogram hist_h with a second exponent S_h
 *     (fixed_exp then points at two int32: S, S_h).
 *
 * Histogram layout: hist_cnt[slot][feature][256] (uint32) and
 * hist_q[slot][feature][256] (int64, fixed point with exponent S); G of an
 * entry is hist_q * 2^-S; with the logistic objective also
 * hist_h[slot][feature][256] (int64), H = hist_h * 2^-S_h.
 */
#ifndef GBDT_H_
#define GBDT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBDT_OK 0
#define GBDT_ERR_INVALID_ARG (-1) /* bad pointer, size, alignment or parameter */
#define GBDT_ERR_NONFINITE (-2)   /* NaN or Inf in features or labels */
#define GBDT_ERR_WORKSPACE (-3)   /* workspace smaller than *_workspace_size */
#define GBDT_ERR_CUDA (-4)        /* a CUDA runtime call failed */
#define GBDT_ERR_INTERNAL (-5)    /* a kernel detected an inconsistency */

#define GBDT_MAX_BINS 256
#define GBDT_MAX_DEPTH 12

#define GBDT_DTYPE_F32 0
#define GBDT_DTYPE_F64 1

/* Objectives.  Squared error ("Module Design: Training Core" s.2): g = pred -
 * label, h = 1, initial prediction mean(label).  Logistic ("Gradient boosted
 * trees (spec model)", binary cross-entropy of sigmoid(pred) against a 0/1
 * target): g = sigmoid(pred) - label, h = p (1 - p) with p = sigmoid(pred),
 * labels must be 0 or 1, initial prediction (margin) 0.  Predictions are
 * margins for both. */
#define GBDT_OBJECTIVE_SQUARED_ERROR 0
#define GBDT_OBJECTIVE_LOGISTIC 1

/* Training parameters; rules of "Module Design: Training Core" s.3:
 * min_samples_leaf >= 1, min_child_weight >= 0, reg_lambda >= 0, gamma >= 0,
 * every floating parameter finite; here also 0 <= max_depth <= GBDT_MAX_DEPTH
 * and n_trees >= 0. */
typedef struct gbdt_params {
  int32_t n_trees;
  int32_t max_depth;        /* root at depth 0; nodes at depth max_depth are leaves */
  double learning_rate;     /* shrinkage applied to each tree's output */
  double reg_lambda;        /* lambda in score G^2/(H+lambda) and weight -G/(H+lambda) */
  double gamma;             /* subtracted from every split gain */
  int32_t min_samples_leaf; /* rows each child must hold */
  double min_child_weight;  /* H each child must hold */
  int32_t num_leaves;       /* leaf budget per tree, 0: none.  Levels split while all of their valid splits
                               fit the budget; at the first level where they would not, the top
                               K = num_leaves - (leaves so far + the level's nodes) candidates by (gain desc,
                               node index asc) split and their children are leaves (the ExaBoost page's
                               depth-capped final partial level).  1 is invalid. */
  int32_t objective;        /* GBDT_OBJECTIVE_SQUARED_ERROR (0) or GBDT_OBJECTIVE_LOGISTIC (1) */
  int32_t bin_packing;      /* GBDT_BIN_PACKING_4BIT (0): in gbdt_train's internal copies of the bins,
                               features with n_bins <= 16 are stored two per byte (4 bits each, the
                               ExaBoost page's packed bins); GBDT_BIN_PACKING_OFF (1): one byte each.
                               Results are identical either way. */
  int32_t hist_registers;   /* GBDT_HIST_REGISTERS_OFF (0): every level histogram is accumulated with shared-memory
                               atomics; GBDT_HIST_REGISTERS_ON (1), squared error only: features with at most 8
                               bins (two of them in one slot when their bin counts multiply to at most 8) are
                               accumulated per code in registers instead (the ExaBoost page's register-
                               accumulation construct body).  Results are identical either way. */
} gbdt_params; /* 64 bytes */

#define GBDT_BIN_PACKING_4BIT 0
#define GBDT_BIN_PACKING_OFF 1
#define GBDT_HIST_REGISTERS_OFF 0
#define GBDT_HIST_REGISTERS_ON 1

/* One tree node, "Module Design: Training Core" s.3 Tree Model: feature,
 * threshold bin, child indices, leaf value, gain and a leaf flag.  Trees are
 * breadth-first: the root is node 0 and the children of a split are appended
 * left then right in the order of their parent's index.  Rows with
 * bin <= threshold_bin go left. */
typedef struct gbdt_node {
  int32_t feature;       /* -1 for a leaf */
  int32_t threshold_bin; /* -1 for a leaf */
  int32_t left;          /* -1 for a leaf */
  int32_t right;         /* -1 for a leaf */
  double leaf_value;     /* weight(G,H) = -G/(H+lambda) of the node's rows */
  double gain;           /* gain of the split; 0 for a leaf */
  uint8_t is_leaf;       /* 1 for a leaf */
  uint8_t reserved[7];
} gbdt_node; /* 40 bytes */

/* Per-level descriptor (device memory).  A level's nodes are the BFS indices
 * [node_begin, node_begin + n_slots); slot s is node node_begin + s.  A row is
 * active at the level iff its node id lies in that range. */
typedef struct gbdt_level {
  int32_t node_begin;
  int32_t n_slots;
} gbdt_level;

/* Result of the split search for one slot (device memory). */
typedef struct gbdt_split {
  int32_t feature;    /* -1: no valid candidate with gain > 0 (the node stays a leaf) */
  int32_t bin;        /* threshold bin: bin <= this goes left */
  double gain;        /* gain of the chosen candidate */
  int64_t q_left;     /* fixed-point G of the left child */
  int64_t q_total;    /* fixed-point G of the node */
  uint32_t cnt_left;  /* rows (= H for squared error) of the left child */
  uint32_t cnt_total; /* rows (= H for squared error) of the node */
  int64_t h_left;     /* logistic: fixed-point H (exponent S_h) of the left child; else 0 */
  int64_t h_total;    /* logistic: fixed-point H of the node; else 0 */
} gbdt_split; /* 56 bytes */

/* A contiguous run of the row-index array that holds one node's rows. */
typedef struct gbdt_segment {
  int64_t start;
  int64_t count;
} gbdt_segment;

/* A row filter for one slot: the slot's rows are those of its segment whose
 * decision (bins[feature][p] > bin) equals side (0: left, 1: right), i.e. one
 * child of a split whose rows have not been partitioned yet.  feature < 0: no
 * filter (every row of the segment). */
typedef struct gbdt_filter {
  int32_t feature;
  int32_t bin;
  int32_t side;
  int32_t reserved;
} gbdt_filter;

/* Library diagnostics ("Module Design: Training Core" s.4, diagnostics()).
 * Filled by gbdt_train when a non-NULL pointer is passed; device times are
 * CUDA-event times on the training stream, summed over all launches of each
 * kernel family; bytes are algorithmic bytes (what the launch must move). */
typedef struct gbdt_diagnostics {
  int64_t hist_launches;     /* histogram-construction launches */
  double hist_ms;            /* their total device time */
  double hist_bytes;         /* their algorithmic bytes */
  int64_t hist_rows;         /* rows read for directly built histograms, summed */
  double part_ms;            /* device time of the row partitions (data moves) */
  double part_bytes;         /* their algorithmic bytes */
  double total_ms;           /* device time of the whole training call */
  int64_t kernel_launches;   /* kernels launched by the call */
  int32_t trees_at_full_size; /* trees that reached 2^max_depth leaves */
  int32_t reserved;
  double hist_level_bytes;   /* the same launches' bytes by the level formula, as if every row of
                                the level's nodes were read once: rows x (F + 8 B gradient + 2 B
                                node id) + built histograms x F x 256 x 12 B (20 B with H); the
                                histogram reads fewer (hist_bytes: the smaller children's rows at a
                                level after a move, both children's rows at the others) */
} gbdt_diagnostics;

/* Message of the last error on the calling thread ("" if none). */
const char* gbdt_last_error(void);

/* Library version string. */
const char* gbdt_version(void);

/* Number of kernels this library has launched in the process so far
 * (monotonic; a caller takes differences around a region of interest). */
int64_t gbdt_kernel_launch_count(void);

/* gbdt_workspace_status: the device error word of the last call queued with
 * workspace ws (see the conventions above).  Copies the word to the host on
 * `stream` and synchronises the stream; *bits (host, may be NULL) receives it.
 * Returns GBDT_OK when it is 0, else GBDT_ERR_INTERNAL with a message naming
 * each check that failed (GBDT_ERR_INVALID_ARG when the only failure is a bin
 * at or above its feature's n_bins).  ws: the 256-byte aligned device
 * workspace that was passed to the call. */
int gbdt_workspace_status(const void* ws, int32_t* bits, void* stream);

/* Parameter rules of "Module Design: Training Core" s.3 (see gbdt_params);
 * GBDT_OK or GBDT_ERR_INVALID_ARG.  Host only, queues nothing. */
int gbdt_validate_params(const gbdt_params* p);

/* ---------------------------------------------------------------------------
 * gbdt_quantize: exact quantile binning of fp32 features to uint8 bins.
 * The pages name the "Quantized" state ("Module Design: Training Core" s.5)
 * but not the rule; this library's rule, for feature j with v its N values
 * sorted ascending (-0.0 read as +0.0) and U distinct values:
 *   U <= max_bins: edges are the U-1 smallest distinct values;
 *   U >  max_bins: e_k = v[ceil(k*N/max_bins) - 1], k = 1..max_bins-1, keeping
 *                  the strictly increasing ones and dropping one equal to v[N-1].
 * bin(x) = number of edges strictly below x, so x <= edges[b] means bin <= b,
 * which is routing "x > threshold goes right" of "Gradient boosted trees (spec
 * model)", Tree representation, with threshold edges[b].
 *   X      [F][ldx] fp32 column-major, ldx >= N (feature j at X + j*ldx)
 *   bins   [F][ldb] uint8 output
 *   edges  [F][max_bins-1] fp32 output; unused entries are +INFINITY
 *   n_bins [F] int32 output, |edges|+1 per feature
 * 2 <= max_bins <= 256, 1 <= N < 2^31.  NaN/Inf in X: GBDT_ERR_NONFINITE and
 * no output written.  Synchronises the stream once (the finiteness check).
 * ------------------------------------------------------------------------- */
size_t gbdt_quantize_workspace_size(int64_t N, int32_t F);
int gbdt_quantize(const float* X, int64_t ldx, int64_t N, int32_t F, int32_t max_bins, uint8_t* bins,
                  int64_t ldb, float* edges, int32_t* n_bins, void* ws, size_t ws_bytes, void* stream);

/* gbdt_quantize_host: gbdt_quantize of features that are in HOST memory.
 *   X_host [F][ldx] fp32 (host; page-locked memory lets the copies overlap)
 *   X_dev  [F][ldx] fp32 (device, caller-owned): receives the copy of X_host
 * The same rule and outputs as gbdt_quantize (workspace: gbdt_quantize_workspace_size).
 * The columns are copied in batches on a stream the call creates and
 * destroys, each after the work already queued on `stream`; each batch is
 * binned as soon as its copy has landed, so the copy of later columns runs
 * under the sort of earlier ones.  NaN/Inf in X: GBDT_ERR_NONFINITE, found
 * after the outputs were written (do not use them).  Synchronises the stream
 * once, at the end; X_host may be released when the call returns.
 * ------------------------------------------------------------------------- */
int gbdt_quantize_host(const float* X_host, int64_t ldx, int64_t N, int32_t F, int32_t max_bins, float* X_dev,
                       uint8_t* bins, int64_t ldb, float* edges, int32_t* n_bins, void* ws, size_t ws_bytes,
                       void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_compute_gradients: squared error, "Module Design: Training Core" s.2:
 * g_i = pred_i - label_i (FP64), h_i = 1 (implicit).  Also computes the
 * fixed-point exponent S of these g into *fixed_exp (device int32), as
 * gbdt_gradient_scale does.
 *   pred [N] fp64, label [N] fp32, g [N] fp64 output.
 * ------------------------------------------------------------------------- */
size_t gbdt_gradients_workspace_size(int64_t N);
int gbdt_compute_gradients(const double* pred, const float* label, int64_t N, double* g, int32_t* fixed_exp,
                           void* ws, size_t ws_bytes, void* stream);

/* gbdt_compute_gradients_objective: g of either objective (GBDT_OBJECTIVE_*).
 * Squared error is gbdt_compute_gradients.  Logistic ("Gradient boosted trees
 * (spec model)", BCE with a sigmoid): g_i = sigmoid(pred_i) - label_i, with
 * sigmoid(x) = 1 / (1 + exp(-x)) in FP64; fixed_exp (device) receives two
 * int32: S of the g and S_h of the hessians h_i = |g_i| (1 - |g_i|), which for
 * a 0/1 label equal p (1 - p) (p = g for label 0, 1 + g for label 1), so h
 * needs no array of its own.  Labels are not checked here (gbdt_train checks
 * that they are 0 or 1).  Workspace: gbdt_gradients_workspace_size. */
int gbdt_compute_gradients_objective(const double* pred, const float* label, int64_t N, int32_t objective,
                                     double* g, int32_t* fixed_exp, void* ws, size_t ws_bytes, void* stream);

/* gbdt_gradient_scale: exponent S for gradients g [N] (g_dtype F32 or F64):
 * S = 62 - ceil(log2 N) - E where max|g| < 2^E (S = 0 if all g are 0), so the
 * sum of |round(g*2^S)| over any set of rows is below 2^62. */
int gbdt_gradient_scale(const void* g, int32_t g_dtype, int64_t N, int32_t* fixed_exp, void* ws, size_t ws_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_build_histograms: per-bin count and fixed-point G of every slot of a
 * level that has build_flag[slot] = 1, over all features, in one call
 * ("Module Design: Training Core" s.6 step 2 and s.7: count/G/H per bin).
 *   bins [F][ldb] uint8; g [N] of g_dtype; fixed_exp: device int32 S
 *   node_of_row [N] uint16: BFS node id of each row
 *   level: device gbdt_level; max_slots: host bound on level->n_slots
 *   build_flag [max_slots] uint8 (device); max_build: host bound on the number
 *     of flagged slots
 *   hist_cnt/hist_q [max_slots][F][256]: the flagged slots are overwritten;
 *     other slots are not touched.
 * 1 <= max_slots <= 4096.  Device check (error word, gbdt_workspace_status):
 * level->n_slots > max_slots (the extra slots are ignored).
 * ------------------------------------------------------------------------- */
size_t gbdt_histograms_workspace_size(int64_t N, int32_t F, int32_t max_slots);
int gbdt_build_histograms(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g, int32_t g_dtype,
                          const int32_t* fixed_exp, const uint16_t* node_of_row, const gbdt_level* level,
                          int32_t max_slots, const uint8_t* build_flag, int32_t max_build, uint32_t* hist_cnt,
                          int64_t* hist_q, void* ws, size_t ws_bytes, void* stream);

/* gbdt_subtract_histograms: sibling subtraction ("Module Design: Training
 * Core" s.6 step 2: the larger child's histogram is the parent's minus the
 * smaller one's).  Slots come in sibling pairs (2p, 2p+1); for
 * p < level->n_slots/2 the slot of the pair with build_flag = 0 receives
 * parent - built, where the parent is slot pair_parent[p] of prev_cnt/prev_q
 * (the previous level's histograms).  Exact (integer).  pair_parent
 * [max_slots/2] int32 (device).  ws (optional, may be NULL): a workspace of
 * gbdt_subtract_histograms_workspace_size() bytes whose error word records a
 * built count above its parent's (gbdt_workspace_status); with NULL that
 * check is not recorded. */
size_t gbdt_subtract_histograms_workspace_size(void);
int gbdt_subtract_histograms(const uint32_t* prev_cnt, const int64_t* prev_q, const int32_t* pair_parent,
                             const uint8_t* build_flag, const gbdt_level* level, int32_t max_slots, int32_t F,
                             uint32_t* hist_cnt, int64_t* hist_q, void* ws, size_t ws_bytes, void* stream);
/* The same with H histograms (logistic): prev_h and hist_h, both non-NULL,
 * are subtracted like prev_q and hist_q. */
int gbdt_subtract_histograms_h(const uint32_t* prev_cnt, const int64_t* prev_q, const int64_t* prev_h,
                               const int32_t* pair_parent, const uint8_t* build_flag, const gbdt_level* level,
                               int32_t max_slots, int32_t F, uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h,
                               void* ws, size_t ws_bytes, void* stream);

/* gbdt_build_histograms_segmented: the same per-bin count and fixed-point G
 * of every flagged slot of a level ("Module Design: Training Core" s.6 step 2,
 * s.7), for rows already grouped by node: the rows of slot s are the
 * positions segments[s].start .. + segments[s].count of every column of
 * bins [F][ldb] and of g (as gbdt_partition_rows leaves them), restricted by
 * filters[s] when filters is not NULL (a child whose rows still sit inside
 * its parent's segment: the segment is then the parent's).  Only the flagged
 * segments are read (with sibling subtraction, the smaller child of each
 * pair); the flagged rows are cut into equal shares, one per CTA and up to
 * 64 features of shared-memory histograms per CTA.  segments, filters
 * [max_slots] (device; filters may be NULL); other arguments and outputs as
 * gbdt_build_histograms.  Workspace: gbdt_histograms_segmented_workspace_size. */
#define GBDT_LAYOUT_COLUMNS 0    /* bins [F][ldb]: feature j's row p at j * ldb + p */
#define GBDT_LAYOUT_ROW_BLOCKS 1 /* feature j's row p at (p / 32) * pitch + 32 * j + p % 32 */

/* The row-block layout of binned features (the layout gbdt_train keeps its
 * per-level copies in; the pages have no counterpart): the 32 rows of a row
 * block are contiguous per feature and the features of a row block are
 * contiguous, so 32 lanes reading 32 rows of 32 consecutive features read one
 * contiguous kilobyte.  pitch = 32 * (F rounded up to a multiple of 4) bytes
 * per row block; a buffer holds ceil(N / 32) row blocks, 32-byte aligned.
 * gbdt_bins_to_row_blocks converts column-major bins [F][ldb] (asynchronous);
 * bytes of the last row block past N are copied as they are. */
int64_t gbdt_row_block_pitch(int32_t F);

/* gbdt_row_block_slots (HOST only, no GPU): the slots of gbdt_train's internal
 * row-block copies for features with n_bins [F] (host) and a GBDT_BIN_PACKING_*
 * mode.  With GBDT_BIN_PACKING_4BIT, features with n_bins <= 16 pair up in
 * feature order in one 32-byte slot, the first of a pair in the low nibble of
 * each byte and the second in the high nibble (a last unpaired one keeps a whole
 * byte); every other feature has a slot of its own, slots numbered in the order
 * of their first feature.  loc [F] (host) receives slot | nibble << 16 (nibble
 * 0: whole byte, 1: low, 2: high); src [F] (host) receives, for each slot s <
 * the returned count, first feature | second feature << 16 (0xffff: none).
 * Returns the slot count (pitch = 32 x slots), or GBDT_ERR_INVALID_ARG. */
int32_t gbdt_row_block_slots(const int32_t* n_bins, int32_t F, int32_t packing, uint32_t* loc, uint32_t* src);
/* gbdt_row_block_slots_ex (HOST only, no GPU): the same plan with a GBDT_HIST_REGISTERS_* mode, the one
 * gbdt_train uses (squared error).  With GBDT_HIST_REGISTERS_ON the features with at most 8 bins leave the
 * ordinary plan and get register slots after it, in feature order: two share a slot (the first in the
 * low nibble) when the packing mode is 4-bit and their bin counts multiply to at most 8, else one takes
 * a whole byte.  *reg_begin (host) receives the first register slot (the returned count when there are
 * none).  Returns the slot count, or GBDT_ERR_INVALID_ARG. */
int32_t gbdt_row_block_slots_ex(const int32_t* n_bins, int32_t F, int32_t packing, int32_t hist_registers,
                                uint32_t* loc, uint32_t* src, int32_t* reg_begin);
size_t gbdt_row_block_bytes(int64_t N, int32_t F);
int gbdt_bins_to_row_blocks(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, uint8_t* out, void* stream);

size_t gbdt_histograms_segmented_workspace_size(int32_t max_slots);
/* layout: GBDT_LAYOUT_COLUMNS (ldb >= N, ldb % 16 == 0) or GBDT_LAYOUT_ROW_BLOCKS
 * (ldb = gbdt_row_block_pitch(F), bins 32-byte aligned). */
int gbdt_build_histograms_segmented(const uint8_t* bins, int64_t ldb, int32_t layout, int64_t N, int32_t F,
                                    const void* g, int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                                    int32_t max_slots, const uint8_t* build_flag, int32_t max_build,
                                    const gbdt_segment* segments, const gbdt_filter* filters, uint32_t* hist_cnt,
                                    int64_t* hist_q, void* ws, size_t ws_bytes, void* stream);
/* The same with the logistic objective's H histogram: hist_h [max_slots][F][256]
 * (non-NULL) receives the fixed-point sums of h = |g| (1 - |g|) (the hessian
 * of a row whose g is sigmoid(pred) - label, label 0 or 1, see
 * gbdt_compute_gradients_objective) with exponent fixed_exp[1]; fixed_exp[0]
 * is S of g.  Up to 32 features of shared-memory histograms per CTA. */
int gbdt_build_histograms_segmented_h(const uint8_t* bins, int64_t ldb, int32_t layout, int64_t N, int32_t F,
                                      const void* g, int32_t g_dtype, const int32_t* fixed_exp,
                                      const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag,
                                      int32_t max_build, const gbdt_segment* segments, const gbdt_filter* filters,
                                      uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, void* ws,
                                      size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_find_splits: best split of every slot of a level, "Module Design:
 * Training Core" s.2-s.3.  For feature j and threshold b = 0..n_bins[j]-2 the
 * left side is bins <= b (prefix over bins), the right side is node minus
 * left.  Valid iff both sides have cnt >= min_samples_leaf,
 * H >= min_child_weight and H > 0.  gain = 0.5*((s_L + s_R) - s_P) - gamma
 * with s = G*G/(H+lambda), FP64, no contraction.  Best = strictly larger
 * gain, then smaller feature, then smaller bin; a slot splits iff its best
 * valid gain is > 0 (else out[slot].feature = -1).  Node totals are the sums
 * over feature 0's bins below n_bins[0] (the same for every feature); bins at
 * or above a feature's n_bins are never read (they may hold anything).
 *   out [max_slots] gbdt_split (device); p: host pointer.
 * Work is spread over (slot, feature) pairs, then reduced per slot; since the
 * comparison is a total order the result does not depend on that split.
 * Device check (error word, gbdt_workspace_status): a feature whose
 * histogram does not add up to the node totals of feature 0.
 * ------------------------------------------------------------------------- */
size_t gbdt_find_splits_workspace_size(int32_t F, int32_t max_slots);
int gbdt_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int32_t* fixed_exp, int32_t F,
                     const int32_t* n_bins, const gbdt_level* level, int32_t max_slots, const gbdt_params* p,
                     gbdt_split* out, void* ws, size_t ws_bytes, void* stream);
/* The same with H from an H histogram (logistic): H = hist_h * 2^-fixed_exp[1]
 * (hist_h non-NULL, 16-byte aligned).  min_samples_leaf applies to the row
 * counts, min_child_weight and H > 0 to H; out[].h_left/h_total are filled. */
int gbdt_find_splits_h(const uint32_t* hist_cnt, const int64_t* hist_q, const int64_t* hist_h,
                       const int32_t* fixed_exp, int32_t F, const int32_t* n_bins, const gbdt_level* level,
                       int32_t max_slots, const gbdt_params* p, gbdt_split* out, void* ws, size_t ws_bytes,
                       void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_partition: "Module Design: Training Core" s.6 step 5.  The k-th slot
 * (in slot order) whose split has feature >= 0 gets the child slots 2k (left)
 * and 2k+1 (right) of the next level, whose node_begin is
 * level->node_begin + level->n_slots.  For such a slot s:
 *   - rows r of s get node_of_row[r] = child node (left iff
 *     bins[feature][r] <= bin);
 *   - its segment seg_in[s] of idx_in is written to idx_out at the same
 *     positions, left rows first, each side in input order (stable);
 *   - seg_out[2k], seg_out[2k+1] are the children's segments.
 * Segments of slots without a split are copied unchanged to idx_out.
 * next_level (device) receives {node_begin + n_slots, 2*splits}.  Positions
 * outside the level's segments are not written.  Device check (error word,
 * gbdt_workspace_status): a split slot whose rows going left differ from its
 * record's cnt_left (the rows are still placed by the counts the kernels
 * compute, so every write stays inside the slot's segment).
 * ------------------------------------------------------------------------- */
size_t gbdt_partition_workspace_size(int64_t N, int32_t max_slots);
int gbdt_partition(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const gbdt_split* splits,
                   const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg_in, const uint32_t* idx_in,
                   uint16_t* node_of_row, uint32_t* idx_out, gbdt_segment* seg_out, gbdt_level* next_level,
                   void* ws, size_t ws_bytes, void* stream);

/* gbdt_partition_rows: "Module Design: Training Core" s.6 step 5 carried out
 * on the data itself.  For every slot whose split has feature >= 0, the
 * positions seg_in[s] of every per-position array -- bins [F][ldb] (uint8),
 * g [N] (g_dtype), orig [N] (uint32, the original row id) -- are copied to the
 * same positions of the *_out arrays, rows going left first, each side in
 * input order (stable).  A row goes right iff bins[feature][p] > bin, or, when
 * go_right [N] (uint8, device) is given, iff go_right[p] != 0.  The k-th
 * splitting slot (slot order) gets seg_out[2k] (left), seg_out[2k+1] (right);
 * next_level (optional) receives {node_begin + n_slots, 2*splits}.  Slots
 * without a split are not copied; if leaf_of_row [original rows] (uint16) is
 * given, leaf_of_row[orig_in[p]] = node_begin + s for their positions.
 * Inputs and outputs must not alias.  Device check as gbdt_partition. */
size_t gbdt_partition_rows_workspace_size(int64_t N, int32_t max_slots);
int gbdt_partition_rows(const uint8_t* bins_in, uint8_t* bins_out, int64_t ldb, int64_t N, int32_t F,
                        const void* g_in, void* g_out, int32_t g_dtype, const uint32_t* orig_in, uint32_t* orig_out,
                        const uint8_t* go_right, const gbdt_split* splits, const gbdt_level* level,
                        int32_t max_slots, const gbdt_segment* seg_in, gbdt_segment* seg_out,
                        gbdt_level* next_level, uint16_t* leaf_of_row, void* ws, size_t ws_bytes, void* stream);

/* gbdt_partition_noalloc: gbdt_partition without a workspace argument.  The
 * pages have no counterpart; this entry point exists for callers that cannot
 * allocate device memory at the point where they partition -- code that runs
 * inside another framework's fixed memory pool, a plugin that has no access
 * to the host application's allocator, or a latency-critical loop where a
 * cudaMalloc (which can synchronise the device) is not allowed.  It calls no
 * allocator: its scratch is a 128 KiB array in the library's device memory,
 * which every GPU that loads the library holds until the process exits.
 * Limits of that scratch: N <= 16,777,216 rows and max_slots <= 1024; larger
 * sizes return GBDT_ERR_INVALID_ARG with a message naming the limit.
 * The first call on each device (and again in a new context of that device,
 * e.g. after cudaDeviceReset) looks the array's device address up, with that
 * device current; make that first call before any stream capture.
 * All calls on a device share the one array, and it keeps the previous
 * call's contents: each call clears what must start at zero (its error
 * word), but calls that overlap on the GPU (different streams, or host
 * threads) race on it and must be serialised by the caller.  Arguments and
 * results are as gbdt_partition. */
int gbdt_partition_noalloc(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const gbdt_split* splits,
                           const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg_in,
                           const uint32_t* idx_in, uint16_t* node_of_row, uint32_t* idx_out,
                           gbdt_segment* seg_out, gbdt_level* next_level, void* stream);
/* gbdt_partition_noalloc_status: the device error word of the last
 * gbdt_partition_noalloc call on the current device (its checks are those of
 * gbdt_partition), which lives in the built-in scratch array.  Copies it to
 * the host on `stream` and synchronises the stream; *bits (host, may be NULL)
 * receives it.  Returns GBDT_OK or GBDT_ERR_INTERNAL as gbdt_workspace_status.
 * Allocates nothing. */
int gbdt_partition_noalloc_status(int32_t* bits, void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_update_predictions: "Module Design: Training Core" s.6 step 7 and
 * "Gradient boosted trees (spec model)", forward pass:
 * pred[i] = pred[i] + (lr * leaf_value[leaf_of_row[i]]) (product rounded
 * first).  leaf_value [n_leaf_values] fp64, leaf_of_row [N] uint16.
 * ------------------------------------------------------------------------- */
int gbdt_update_predictions(double* pred, const uint16_t* leaf_of_row, const double* leaf_value,
                            int32_t n_leaf_values, int64_t N, double lr, void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_predict: batched prediction on raw fp32 features ("Gradient boosted
 * trees (spec model)", Forward pass: init + learning_rate * sum of tree
 * outputs; Tree representation: x > threshold goes right).  The threshold of a
 * split (feature j, bin b) is edges[j][b] from gbdt_quantize, so routing raw
 * values is exactly the training's routing on bins; the sum is taken tree by
 * tree, pred + (learning_rate * leaf_value) with the product rounded first, so
 * the predictions of the training rows equal gbdt_train's pred_out bit for
 * bit.  A NaN compares false and goes left.
 *   X [F][ldx] fp32 column-major (device); edges [F][max_bins-1] (device) as
 *   gbdt_quantize wrote them; nodes [n_trees][max_nodes] gbdt_node (device,
 *   the layout gbdt_train returns: BFS, right = left + 1); nodes_per_tree
 *   [n_trees] int32 (device; NULL: every slot is a node): the nodes a tree
 *   uses are its first nodes_per_tree[t] slots; out [N] fp64.
 * Every used internal node is checked (feature < F, bin < max_bins - 1,
 * children a pair after the node among the used nodes); a bad node or count
 * makes the call return GBDT_ERR_INVALID_ARG (out is then unspecified).  Workspace:
 * gbdt_predict_workspace_size(n_trees, max_nodes).  Synchronises the stream
 * once at the end (to report model errors).
 * ------------------------------------------------------------------------- */
size_t gbdt_predict_workspace_size(int32_t n_trees, int32_t max_nodes);
int gbdt_predict(const float* X, int64_t ldx, int64_t N, int32_t F, const float* edges, int32_t max_bins,
                 const gbdt_node* nodes, const int32_t* nodes_per_tree, int32_t n_trees, int32_t max_nodes,
                 double init_pred, double learning_rate, double* out, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * gbdt_train: whole training run ("Module Design: Training Core" s.6).
 *   bins [F][ldb] uint8, n_bins [F] int32 (1..256), label [N] fp32 (device);
 *     every bin of feature j must be below n_bins[j] (checked: GBDT_ERR_INVALID_ARG)
 *   p: host pointer
 *   pred_out [N] fp64 (device): predictions (margins) after the last tree
 *   init_pred_out: host double, the initial prediction: mean(label) for
 *     squared error, 0 for the logistic objective
 *   nodes_out: HOST array [n_trees][2^(max_depth+1)-1] gbdt_node; tree t's
 *     nodes are nodes_out[t*(2^(max_depth+1)-1) + i], i < nodes_per_tree[t]
 *   nodes_per_tree: HOST [n_trees] int32
 *   diag: optional HOST diagnostics (NULL to skip the timing events)
 * Synchronises the stream twice: after the input checks (n_bins range, finite
 * labels) and at the end.  With n_trees >= 4 the launches of one tree are
 * captured once per call into a CUDA graph (on a stream the call creates and
 * destroys) and trees 1 .. n_trees-2 replay it on `stream` (with diag, its
 * timing events are nodes of that graph on a branch of their own, recorded on
 * a second stream the call creates, pointed at each tree's events); the
 * results are the same as launching tree by tree (which the failure-injection
 * hook uses).  On any error after parameter validation nodes_out
 * is left untouched and nodes_per_tree[*] = 0 (no partial model, s.5 State
 * Machine).
 * NaN/Inf labels: GBDT_ERR_NONFINITE; with the logistic objective a label
 * other than 0 or 1: GBDT_ERR_INVALID_ARG.  1 <= N < 2^31, 1 <= F <= 4096.
 * ------------------------------------------------------------------------- */
size_t gbdt_train_workspace_size(int64_t N, int32_t F, const gbdt_params* p);
int gbdt_train(const uint8_t* bins, int64_t ldb, const int32_t* n_bins, int64_t N, int32_t F, const float* label,
               const gbdt_params* p, double* pred_out, double* init_pred_out, gbdt_node* nodes_out,
               int32_t* nodes_per_tree, gbdt_diagnostics* diag, void* ws, size_t ws_bytes, void* stream);

/* Testing hook for "Module Design: Training Core" s.5 ("Failed must not
 * export a model"): while after_levels >= 0, gbdt_train fails with
 * GBDT_ERR_INTERNAL on the host after that many levels, leaving nodes_out
 * untouched; -1 (the initial state) disables it.  Process-wide. */
void gbdt_debug_inject_failure(int32_t after_levels);

#ifdef __cplusplus
}
#endif
#endif /* GBDT_H_ */
