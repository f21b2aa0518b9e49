/*
 * gbdt_oracle.c -- CPU oracle for level-wise histogram GBDT with squared error.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, FP64 restatement of
 * what the training method computes.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library, and it never reads anything the CUDA
 * path produced except the optional lockstep guide of orc_train (see there),
 * which can only choose between candidates this file itself rates as tied.
 *
 * Sources (page titles and sections):
 *   [MPS-TC]  "Module Design: Training Core" (MPSBoost spec)
 *             s.2 Single Mathematical Semantics  -- g, h, score, weight, gain
 *             s.3 Tree Model                      -- flat BFS nodes, frozen
 *                                                    tie-break, validity, routing,
 *                                                    parameter rules
 *             s.6 Tree Growth                     -- level-wise growth steps 1-7
 *             s.7 CPU Oracle                      -- FP64 count/G/H per bin in
 *                                                    row-index order
 *   [LEAN]    "Gradient boosted trees (spec model)" (TorchLean)
 *             Forward pass -- init + learning_rate * sum of tree outputs;
 *             Tree representation -- goRight := x > threshold.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - Quantile binning (the pages name a "Quantized" state only): exact order
 *     statistics, see orc_quantize.
 *   - The node total G_P is the row-order sum over the node's rows; G_R and
 *     H_R are parent minus left; the gain is evaluated as
 *     0.5*((s_L + s_R) - s_P) - gamma with s = G*G/(H+lambda), no fused
 *     multiply-add (build with -ffp-contract=off).
 *   - "meet minimum" reads as >=.
 *   - Depth D: root at depth 0, nodes at depth D are leaves.
 *   - Initial prediction: mean of the labels, FP64 sum in row order / N.
 *   - Prediction update: pred + (lr * w), product rounded first.
 *
 * Parity pins: every function here is checked by tests that do not call it
 * back (brute force, closed forms, the CART special case, invariants,
 * hand-computed trees).  No function in this file is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENONFINITE (-2)
#define ORC_ENOMEM (-3)

#define ORC_NBINS 256      /* histogram width: every bin index a uint8 can hold */
#define ORC_NEAR_MAX 8     /* near-tied candidates recorded per node */
#define ORC_NEAR_REL 1e-12 /* relative gain gap that counts as a near-tie */

typedef struct {
  int32_t n_trees;
  int32_t max_depth;
  double learning_rate;
  double reg_lambda;
  double gamma;
  int32_t min_samples_leaf;
  double min_child_weight;
  int32_t num_leaves; /* leaf budget per tree; 0: none (see orc_train) */
  int32_t objective;  /* 0: squared error; 1: logistic (see orc_gradients_objective) */
  int32_t n_threads;  /* OpenMP threads over features; results do not depend on it */
} orc_params;

typedef struct {
  int32_t feature;       /* -1 for a leaf */
  int32_t threshold_bin; /* -1 for a leaf; bin <= threshold_bin goes left */
  int32_t left, right;   /* BFS child indices, -1 for a leaf */
  double leaf_value;     /* weight(G,H) of the node (used for leaves) */
  double gain;           /* gain of the chosen split, 0 for a leaf */
  int32_t is_leaf;
  int32_t depth;
} orc_node;

typedef struct {
  int64_t n_rows;
  double G, H, A; /* row-order sums of g, h and |g| over the node's rows */
  double best_gain, second_gain; /* over distinct partitions; -INFINITY if none */
  int32_t n_near;                /* candidates within ORC_NEAR_REL of the best */
  int32_t near_feature[ORC_NEAR_MAX];
  int32_t near_bin[ORC_NEAR_MAX];
  int32_t adopted;        /* the guide's choice replaced ours: 1 within ORC_NEAR_REL, 2 within the
                             rounding bound of the tie quanta only (see orc_train) */
  int32_t guide_mismatch; /* 1: the guide disagreed outside both */
  double guide_gap;       /* where the guide differed: our best gain minus the guide's candidate's */
  double guide_bound;     /* the rounding bound that gap was held against (0 without tie quanta) */
} orc_node_info;

typedef struct {
  int32_t valid;   /* 1 if a valid candidate exists */
  int32_t feature; /* best candidate (valid == 1) */
  int32_t bin;
  double gain;
  int64_t cnt_left;
  double G_left, H_left;
  double second_gain; /* best gain over other distinct partitions */
  int32_t n_near;
  int32_t near_feature[ORC_NEAR_MAX];
  int32_t near_bin[ORC_NEAR_MAX];
} orc_split;

/* ------------------------------------------------------------------------ */
/* [MPS-TC] s.2: score, weight and gain, evaluated in the stated order.     */
/* ------------------------------------------------------------------------ */
static double orc_score(double G, double H, double lambda) { return (G * G) / (H + lambda); }

double orc_weight(double G, double H, double lambda) { return -G / (H + lambda); }

double orc_gain(double GL, double HL, double GR, double HR, double GP, double HP, double lambda,
                double gamma) {
  double sL = orc_score(GL, HL, lambda);
  double sR = orc_score(GR, HR, lambda);
  double sP = orc_score(GP, HP, lambda);
  return 0.5 * ((sL + sR) - sP) - gamma;
}

/* ------------------------------------------------------------------------ */
/* Parity harness: how far a candidate's gain can move when another program   */
/* sums the same per-row g (and h) with a bounded rounding per row.  Not part  */
/* of the method; orc_train's lockstep guide uses it to tell rounding ties     */
/* from real disagreements.                                                    */
/* ------------------------------------------------------------------------ */
/* gamma_n = n u / (1 - n u), u = 2^-53: the classical bound on the error of a sum of n terms
 * accumulated one by one in FP64, relative to the sum of their magnitudes. */
static double sum_error_factor(int64_t n) {
  const double nu = (double)n * 0x1p-53;
  return nu < 0.5 ? nu / (1.0 - nu) : INFINITY;
}

/* Bound on |s(G', H') - s(G, H)| for s = G^2 / (H + lambda), |G' - G| <= dG, |H' - H| <= dH:
 * |G'^2 - G^2| <= 2|G| dG + dG^2 over a denominator of at least H + lambda - dH, plus
 * G^2 |1/(H' + lambda) - 1/(H + lambda)| <= G^2 dH / ((H + lambda)(H + lambda - dH)). */
static double score_spread(double G, double H, double dG, double dH, double lambda) {
  const double hl = H + lambda, lo = hl - dH;
  if (!(lo > 0.0)) return INFINITY;
  return (2.0 * fabs(G) * dG + dG * dG) / lo + G * G * dH / (hl * lo);
}

/* Bound on how far a candidate's gain, 0.5 ((s_L + s_R) - s_P) - gamma, computed by this oracle
 * and by another program from the same rows can differ.  The other program's per-row rounding of g
 * is at most qg (of h, qh; 0 when H is a count); this oracle's row-order sums of n terms are off by
 * at most gamma_(n + bins) times the sum of magnitudes (A for G, H_P for h >= 0; a side's
 * magnitudes are at most the node's); each side's conversions add one rounding of its sums, and the
 * gain's own evaluation a few roundings of its scores on each program. */
static double gain_spread(double GL, double HL, int64_t nL, double GP, double HP, int64_t nP, double A, double qg,
                          double qh, int h_counts, double lambda) {
  const double u = 0x1p-53;
  const double GR = GP - GL, HR = HP - HL;
  const double dGL = (double)nL * qg + sum_error_factor(nL + ORC_NBINS) * A + u * fabs(GL);
  const double dGP = (double)nP * qg + sum_error_factor(nP) * A + u * fabs(GP);
  const double dGR = dGP + dGL + u * fabs(GR);
  double dHL = 0.0, dHP = 0.0, dHR = 0.0;
  if (!h_counts) {
    dHL = (double)nL * qh + sum_error_factor(nL + ORC_NBINS) * HP + u * HL;
    dHP = (double)nP * qh + sum_error_factor(nP) * HP + u * HP;
    dHR = dHP + dHL + u * fabs(HR);
  }
  const double sL = orc_score(GL, HL, lambda), sR = orc_score(GR, HR, lambda), sP = orc_score(GP, HP, lambda);
  return 0.5 * (score_spread(GL, HL, dGL, dHL, lambda) + score_spread(GR, HR, dGR, dHR, lambda) +
                score_spread(GP, HP, dGP, dHP, lambda)) +
         8.0 * u * (fabs(sL) + fabs(sR) + fabs(sP));
}

/* [MPS-TC] s.3: parameter rules. */
int orc_validate_params(const orc_params* p) {
  if (!p) return ORC_EINVAL;
  if (p->n_trees < 0 || p->max_depth < 0 || p->max_depth > 15) return ORC_EINVAL;
  if (!isfinite(p->learning_rate) || !isfinite(p->reg_lambda) || !isfinite(p->gamma) ||
      !isfinite(p->min_child_weight))
    return ORC_EINVAL;
  if (p->min_samples_leaf < 1 || p->min_child_weight < 0.0 || p->reg_lambda < 0.0 || p->gamma < 0.0)
    return ORC_EINVAL;
  if (p->num_leaves < 0 || p->num_leaves == 1) return ORC_EINVAL;
  if (p->objective != 0 && p->objective != 1) return ORC_EINVAL;
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Quantile binning (reading; the pages only name the "Quantized" state).   */
/* ------------------------------------------------------------------------ */
static int cmp_float(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  return (x < y) ? -1 : (x > y) ? 1 : 0;
}

/*
 * For each feature j, with v the N values sorted ascending (-0.0 read as
 * +0.0) and U the number of distinct values:
 *   U <= B : edges are the U-1 smallest distinct values (one bin per value);
 *   U >  B : for k = 1..B-1 take e_k = v[ceil(k*N/B) - 1]; keep the strictly
 *            increasing subsequence; drop an edge equal to v[N-1].
 * bin(x) = number of edges strictly below x, so x <= edges[b] means bin <= b,
 * which matches routing "x > threshold goes right" ([LEAN] Tree representation)
 * with threshold = edges[b].  Unused edge slots are +INFINITY.
 * X is column-major [F][N]; bins is [F][N]; edges is [F][max_bins-1].
 */
int orc_quantize(const float* X, int64_t N, int32_t F, int32_t max_bins, int32_t n_threads,
                 uint8_t* bins, float* edges, int32_t* n_bins) {
  if (!X || !bins || !edges || !n_bins || N < 1 || F < 1 || max_bins < 2 || max_bins > 256)
    return ORC_EINVAL;
  for (int64_t i = 0; i < N * (int64_t)F; ++i)
    if (!isfinite(X[i])) return ORC_ENONFINITE;
  const int32_t B = max_bins;
  int status = ORC_OK;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
#endif
  for (int32_t j = 0; j < F; ++j) {
    float* v = (float*)malloc((size_t)N * sizeof(float));
    if (!v) {
      status = ORC_ENOMEM;
      continue;
    }
    const float* col = X + (int64_t)j * N;
    for (int64_t i = 0; i < N; ++i) v[i] = (col[i] == 0.0f) ? 0.0f : col[i];
    qsort(v, (size_t)N, sizeof(float), cmp_float);
    int64_t U = 1;
    for (int64_t i = 1; i < N; ++i)
      if (v[i] != v[i - 1]) ++U;
    float* e = edges + (int64_t)j * (B - 1);
    int32_t ne = 0;
    if (U <= B) {
      for (int64_t i = 0; i < N && ne < U - 1; ++i)
        if (i == 0 || v[i] != v[i - 1]) e[ne++] = v[i];
    } else {
      for (int32_t k = 1; k <= B - 1; ++k) {
        /* ceil(k*N/B) - 1 in integer arithmetic */
        int64_t pk = ((int64_t)k * N + B - 1) / B - 1;
        float ek = v[pk];
        if (ne > 0 && !(ek > e[ne - 1])) continue; /* keep strictly increasing */
        if (ek == v[N - 1]) continue;              /* an edge at the maximum is empty above */
        e[ne++] = ek;
      }
    }
    for (int32_t k = ne; k < B - 1; ++k) e[k] = INFINITY;
    n_bins[j] = ne + 1;
    uint8_t* bj = bins + (int64_t)j * N;
    for (int64_t i = 0; i < N; ++i) {
      float x = col[i];
      int32_t c = 0;
      while (c < ne && e[c] < x) ++c; /* count of edges strictly below x */
      bj[i] = (uint8_t)c;
    }
    free(v);
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* [MPS-TC] s.2: gradients of squared error.                                */
/* ------------------------------------------------------------------------ */
int orc_gradients(const double* pred, const float* label, int64_t N, double* g, double* h) {
  if (!pred || !label || !g || N < 0) return ORC_EINVAL;
  for (int64_t i = 0; i < N; ++i) {
    g[i] = pred[i] - (double)label[i];
    if (h) h[i] = 1.0;
  }
  return ORC_OK;
}

/* Gradients of the objective at the margins pred.  0, squared error ([MPS-TC]
 * s.2): g = pred - label, h = 1.  1, logistic ("Gradient boosted trees
 * (spec model)", binary cross-entropy with a sigmoid and its gradient
 * sigmoid(pred) - target): p = 1 / (1 + exp(-pred)), g = p - label, and the
 * second derivative of the loss in the margin, h = p (1 - p). */
int orc_gradients_objective(const double* pred, const float* label, int64_t N, int32_t objective, double* g,
                            double* h) {
  if (objective == 0) return orc_gradients(pred, label, N, g, h);
  if (objective != 1 || !pred || !label || !g || N < 0) return ORC_EINVAL;
  for (int64_t i = 0; i < N; ++i) {
    const double p = 1.0 / (1.0 + exp(-pred[i]));
    g[i] = p - (double)label[i];
    if (h) h[i] = p * (1.0 - p);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [MPS-TC] s.7: per-bin count/G/H in supplied row-index order, FP64.       */
/* ------------------------------------------------------------------------ */
/*
 * Histogram of one node: rows[0..n) in the order given.  cnt/G/H are
 * [F][256]; A_out (optional) receives sum |g| over the node's rows.
 */
static void node_histogram(const uint8_t* bins, int64_t N, int32_t F, const double* g, const double* h,
                           const int64_t* rows, int64_t n, uint32_t* cnt, double* G, double* H, int32_t n_threads) {
  memset(cnt, 0, sizeof(uint32_t) * (size_t)F * ORC_NBINS);
  memset(G, 0, sizeof(double) * (size_t)F * ORC_NBINS);
  memset(H, 0, sizeof(double) * (size_t)F * ORC_NBINS);
  (void)n_threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(n_threads > 0 ? n_threads : 1)
#endif
  for (int32_t j = 0; j < F; ++j) {
    const uint8_t* col = bins + (int64_t)j * N;
    uint32_t* c = cnt + (int64_t)j * ORC_NBINS;
    double* gg = G + (int64_t)j * ORC_NBINS;
    double* hh = H + (int64_t)j * ORC_NBINS;
    for (int64_t k = 0; k < n; ++k) {
      int64_t r = rows[k];
      int b = col[r];
      c[b] += 1u;
      gg[b] += g[r];
      hh[b] += h ? h[r] : 1.0;
    }
  }
}

/*
 * Histograms of every slot of a level in one call: slot_of_row[r] in
 * [0, n_slots) selects the slot of row r (any other value: row inactive).
 * Rows are visited in ascending index order, which is the supplied order.
 * cnt/G/H are [n_slots][F][256]; n/Gt/Ht/At (optional) are per-slot row
 * counts and row-order sums of g, h and |g|.  h: per-row hessians, or NULL
 * for h = 1 (squared error).
 */
int orc_histograms(const uint8_t* bins, int64_t N, int32_t F, const double* g, const double* h,
                   const int32_t* slot_of_row, int32_t n_slots, uint32_t* cnt, double* G, double* H, int64_t* n,
                   double* Gt, double* Ht, double* At) {
  if (!bins || !g || !slot_of_row || !cnt || !G || !H || N < 0 || F < 1 || n_slots < 0) return ORC_EINVAL;
  const size_t per = (size_t)F * ORC_NBINS;
  memset(cnt, 0, sizeof(uint32_t) * per * (size_t)n_slots);
  memset(G, 0, sizeof(double) * per * (size_t)n_slots);
  memset(H, 0, sizeof(double) * per * (size_t)n_slots);
  if (n) memset(n, 0, sizeof(int64_t) * (size_t)n_slots);
  if (Gt) memset(Gt, 0, sizeof(double) * (size_t)n_slots);
  if (Ht) memset(Ht, 0, sizeof(double) * (size_t)n_slots);
  if (At) memset(At, 0, sizeof(double) * (size_t)n_slots);
  for (int64_t r = 0; r < N; ++r) {
    int32_t s = slot_of_row[r];
    if (s < 0 || s >= n_slots) continue;
    if (n) n[s] += 1;
    if (Gt) Gt[s] += g[r];
    const double hr = h ? h[r] : 1.0;
    if (Ht) Ht[s] += hr;
    if (At) At[s] += fabs(g[r]);
    for (int32_t j = 0; j < F; ++j) {
      size_t o = (size_t)s * per + (size_t)j * ORC_NBINS + bins[(int64_t)j * N + r];
      cnt[o] += 1u;
      G[o] += g[r];
      H[o] += hr;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [MPS-TC] s.3: split search under the frozen rule.                         */
/* ------------------------------------------------------------------------ */
/*
 * One node, histograms cnt/G/H [F][256], node totals (n_P, G_P, H_P).
 * For feature j and threshold b = 0..n_bins[j]-2: left = bins <= b, with
 * G_L, H_L, cnt_L the running prefix sums in bin order; G_R = G_P - G_L,
 * H_R = H_P - H_L, cnt_R = n_P - cnt_L.  A candidate is valid iff both sides
 * have cnt >= min_samples_leaf, H >= min_child_weight and H > 0; invalid
 * candidates never enter the comparison.  Best: strictly larger gain, then
 * smaller feature, then smaller bin (scan order with replace-if-strictly-
 * better gives exactly that).  The caller splits iff valid and gain > 0.
 *
 * Near-tie bookkeeping (for parity reports only): a threshold whose bin is
 * empty gives the same partition as the threshold one below it, so it is not
 * a distinct partition and is skipped for second_gain / the near list.
 */
int orc_best_split(const uint32_t* cnt, const double* G, const double* H, int32_t F, const int32_t* n_bins,
                   int64_t n_P, double G_P, double H_P, const orc_params* p, orc_split* out) {
  if (!cnt || !G || !H || !n_bins || !p || !out || F < 1) return ORC_EINVAL;
  memset(out, 0, sizeof(*out));
  out->feature = -1;
  out->bin = -1;
  out->gain = -INFINITY;
  out->second_gain = -INFINITY;
  const double lambda = p->reg_lambda, gamma = p->gamma, mcw = p->min_child_weight;
  const int64_t msl = p->min_samples_leaf;
  /* pass 1: the winner */
  for (int32_t j = 0; j < F; ++j) {
    const uint32_t* c = cnt + (int64_t)j * ORC_NBINS;
    const double* gg = G + (int64_t)j * ORC_NBINS;
    const double* hh = H + (int64_t)j * ORC_NBINS;
    double GL = 0.0, HL = 0.0;
    int64_t cL = 0;
    int32_t nb = n_bins[j];
    if (nb > ORC_NBINS) nb = ORC_NBINS;
    for (int32_t b = 0; b <= nb - 2; ++b) {
      GL += gg[b];
      HL += hh[b];
      cL += c[b];
      int64_t cR = n_P - cL;
      double GR = G_P - GL, HR = H_P - HL;
      if (!(cL >= msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;
      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);
      if (!out->valid || gain > out->gain) {
        out->valid = 1;
        out->feature = j;
        out->bin = b;
        out->gain = gain;
        out->cnt_left = cL;
        out->G_left = GL;
        out->H_left = HL;
      }
    }
  }
  if (!out->valid) return ORC_OK;
  /* pass 2: runner-up over distinct partitions and the near-tie list */
  const double g1 = out->gain;
  for (int32_t j = 0; j < F; ++j) {
    const uint32_t* c = cnt + (int64_t)j * ORC_NBINS;
    const double* gg = G + (int64_t)j * ORC_NBINS;
    const double* hh = H + (int64_t)j * ORC_NBINS;
    double GL = 0.0, HL = 0.0;
    int64_t cL = 0;
    int32_t nb = n_bins[j];
    if (nb > ORC_NBINS) nb = ORC_NBINS;
    for (int32_t b = 0; b <= nb - 2; ++b) {
      GL += gg[b];
      HL += hh[b];
      cL += c[b];
      if (b > 0 && c[b] == 0) continue; /* same partition as threshold b-1 */
      int64_t cR = n_P - cL;
      double GR = G_P - GL, HR = H_P - HL;
      if (!(cL >= msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;
      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);
      int is_best = (j == out->feature && b == out->bin);
      if (!is_best && gain > out->second_gain) out->second_gain = gain;
      if (fabs(g1 - gain) < ORC_NEAR_REL * fabs(g1) || is_best) {
        if (out->n_near < ORC_NEAR_MAX) {
          out->near_feature[out->n_near] = j;
          out->near_bin[out->n_near] = b;
        }
        out->n_near++;
      }
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [MPS-TC] s.6: level-wise depth-limited growth; [LEAN] forward pass.       */
/* ------------------------------------------------------------------------ */
/*
 * Trains n_trees trees.  bins [F][N] column-major, n_bins [F], label [N].
 * Outputs: pred [N] (after the last tree), *init_pred, nodes
 * [n_trees][2^(max_depth+1)-1] in BFS order, nodes_per_tree [n_trees],
 * optional info (same shape as nodes), optional leaf_of_row [N] (the BFS
 * index of each row's leaf in the last tree).
 *
 * guide (optional, [n_trees][max_nodes][2] = feature, bin; feature -1 = leaf)
 * is the lockstep rule of the parity harness: where this oracle's choice at
 * a node differs from the guide's and the guide's (feature, bin) is a valid
 * candidate whose gain this oracle rates within ORC_NEAR_REL of its best, the
 * guide's candidate is taken (info.adopted = 1).  With tie_quanta
 * ([n_trees][2]: the other program's per-row rounding bound of g and of h, h
 * 0 when H is a row count) the guide's candidate is also taken when the gap
 * is within gain_spread of both candidates, i.e. rounding of the same rows'
 * sums could reorder them (info.adopted = 2); likewise a node whose best gain
 * is within its spread of 0 may split or not as the guide says.  Any other
 * disagreement is recorded (info.guide_mismatch = 1) and this oracle keeps
 * its own choice.
 * pred_in (optional, [N]): start from these predictions instead of the
 * initial value (*init_pred still receives the initial value).
 */
int orc_train(const uint8_t* bins, const int32_t* n_bins, int64_t N, int32_t F, const float* label,
              const orc_params* p, const int32_t* guide, const double* tie_quanta, const double* pred_in,
              double* pred, double* init_pred, orc_node* nodes, int32_t* nodes_per_tree, orc_node_info* info,
              int32_t* leaf_of_row) {
  if (!bins || !n_bins || !label || !pred || !init_pred || !nodes || !nodes_per_tree || N < 1 || F < 1)
    return ORC_EINVAL;
  int rc = orc_validate_params(p);
  if (rc != ORC_OK) return rc;
  for (int32_t j = 0; j < F; ++j)
    if (n_bins[j] < 1 || n_bins[j] > ORC_NBINS) return ORC_EINVAL;
  for (int64_t i = 0; i < N; ++i)
    if (!isfinite(label[i])) return ORC_ENONFINITE;
  const int logistic = p->objective == 1;
  if (logistic)
    for (int64_t i = 0; i < N; ++i)
      if (label[i] != 0.0f && label[i] != 1.0f) return ORC_EINVAL; /* binary labels */

  const int32_t D = p->max_depth;
  const int32_t max_nodes = (int32_t)((1u << (D + 1)) - 1u);
  const double lambda = p->reg_lambda;

  double* g = (double*)malloc(sizeof(double) * (size_t)N);
  double* hv = logistic ? (double*)malloc(sizeof(double) * (size_t)N) : NULL;
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)N); /* rows grouped by node */
  int64_t* scratch = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
  int64_t* seg_start = (int64_t*)malloc(sizeof(int64_t) * (size_t)max_nodes);
  int64_t* seg_count = (int64_t*)malloc(sizeof(int64_t) * (size_t)max_nodes);
  uint32_t* cnt = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)F * ORC_NBINS);
  double* G = (double*)malloc(sizeof(double) * (size_t)F * ORC_NBINS);
  double* H = (double*)malloc(sizeof(double) * (size_t)F * ORC_NBINS);
  const int32_t max_level = (int32_t)(1u << D); /* nodes of the widest level */
  int32_t* lvl_do = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_level);
  int32_t* lvl_keep = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_level);
  int32_t* lvl_f = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_level);
  int32_t* lvl_b = (int32_t*)malloc(sizeof(int32_t) * (size_t)max_level);
  double* lvl_gain = (double*)malloc(sizeof(double) * (size_t)max_level);
  if (!g || (logistic && !hv) || !order || !scratch || !seg_start || !seg_count || !cnt || !G || !H || !lvl_do ||
      !lvl_keep || !lvl_f || !lvl_b || !lvl_gain) {
    free(hv);
    free(g), free(order), free(scratch), free(seg_start), free(seg_count), free(cnt), free(G), free(H);
    free(lvl_do), free(lvl_keep), free(lvl_f), free(lvl_b), free(lvl_gain);
    return ORC_ENOMEM;
  }

  /* initial prediction: mean label, FP64 sum in row order (squared error); margin 0, probability
   * one half (logistic; a reading: the pages fix no initial value for it) */
  double sum = 0.0;
  for (int64_t i = 0; i < N; ++i) sum += (double)label[i];
  const double init = logistic ? 0.0 : sum / (double)N;
  *init_pred = init;
  for (int64_t i = 0; i < N; ++i) pred[i] = pred_in ? pred_in[i] : init;

  for (int32_t t = 0; t < p->n_trees; ++t) {
    orc_node* tn = nodes + (int64_t)t * max_nodes;
    orc_node_info* ti = info ? info + (int64_t)t * max_nodes : NULL;
    const int32_t* tg = guide ? guide + (int64_t)t * max_nodes * 2 : NULL;
    orc_gradients_objective(pred, label, N, p->objective, g, hv);

    for (int64_t i = 0; i < N; ++i) order[i] = i;
    int32_t n_nodes = 1;
    seg_start[0] = 0;
    seg_count[0] = N;
    int32_t level_begin = 0, level_end = 1;
    int32_t leaves_done = 0; /* nodes of earlier levels that stayed leaves */
    int32_t last = D;        /* the level whose nodes are leaves without a search */
    for (int32_t d = 0; d <= last; ++d) {
      const int32_t nl = level_end - level_begin;
      /* phase 1: every node of the level searches its best split */
      for (int32_t v = level_begin; v < level_end; ++v) {
        const int64_t* rows = order + seg_start[v];
        const int64_t n = seg_count[v];
        double GP = 0.0, HP = 0.0, A = 0.0;
        for (int64_t k = 0; k < n; ++k) {
          GP += g[rows[k]];
          HP += hv ? hv[rows[k]] : 1.0;
          A += fabs(g[rows[k]]);
        }
        orc_node* nd = &tn[v];
        nd->feature = -1;
        nd->threshold_bin = -1;
        nd->left = -1;
        nd->right = -1;
        nd->leaf_value = orc_weight(GP, HP, lambda);
        nd->gain = 0.0;
        nd->is_leaf = 1;
        nd->depth = d;
        if (ti) {
          memset(&ti[v], 0, sizeof(ti[v]));
          ti[v].n_rows = n;
          ti[v].G = GP;
          ti[v].H = HP;
          ti[v].A = A;
          ti[v].best_gain = -INFINITY;
          ti[v].second_gain = -INFINITY;
        }
        lvl_do[v - level_begin] = 0;
        if (d == last) continue; /* depth limit (or budget): leaf without search */

        node_histogram(bins, N, F, g, hv, rows, n, cnt, G, H, p->n_threads);
        orc_split sp;
        orc_best_split(cnt, G, H, F, n_bins, n, GP, HP, p, &sp);
        int do_split = sp.valid && sp.gain > 0.0;
        int32_t f = sp.feature, b = sp.bin;
        double gain = sp.gain;
        if (ti) {
          ti[v].best_gain = sp.valid ? sp.gain : -INFINITY;
          ti[v].second_gain = sp.second_gain;
          ti[v].n_near = sp.n_near;
          for (int k = 0; k < ORC_NEAR_MAX; ++k) {
            ti[v].near_feature[k] = sp.near_feature[k];
            ti[v].near_bin[k] = sp.near_bin[k];
          }
        }
        if (tg && (do_split || tg[2 * v] >= 0) && (!do_split || tg[2 * v] != f || tg[2 * v + 1] != b)) {
          /* the guide differs from this oracle: rate its choice with this oracle's own sums.  Only two
           * different split candidates are a mismatch here; a split where the guide has a leaf (or the
           * reverse) is adopted when rounding allows it, else left to the check after the leaf budget */
          const int own_split = do_split;
          const double* tq = tie_quanta ? tie_quanta + 2 * (int64_t)t : NULL;
          const int h_counts = !logistic;
          const double spread_best =
              sp.valid && tq ? gain_spread(sp.G_left, sp.H_left, sp.cnt_left, GP, HP, n, A, tq[0], tq[1], h_counts,
                                           lambda)
                             : 0.0;
          int32_t gf = tg[2 * v], gb = tg[2 * v + 1];
          int kind = 0;
          double gap = 0.0, bound = 0.0, gain_g = 0.0;
          if (gf >= 0) {
            if (gf < F && gb >= 0 && gb <= n_bins[gf] - 2) {
              const uint32_t* cc = cnt + (int64_t)gf * ORC_NBINS;
              const double* gg = G + (int64_t)gf * ORC_NBINS;
              const double* hh = H + (int64_t)gf * ORC_NBINS;
              double GL = 0.0, HL = 0.0;
              int64_t cL = 0;
              for (int32_t q = 0; q <= gb; ++q) {
                GL += gg[q];
                HL += hh[q];
                cL += cc[q];
              }
              const double GR = GP - GL, HR = HP - HL;
              const int64_t cR = n - cL;
              const int valid = cL >= p->min_samples_leaf && cR >= p->min_samples_leaf && HL >= p->min_child_weight &&
                                HR >= p->min_child_weight && HL > 0.0 && HR > 0.0;
              if (valid) {
                gain_g = orc_gain(GL, HL, GR, HR, GP, HP, lambda, p->gamma);
                const double spread_g = tq ? gain_spread(GL, HL, cL, GP, HP, n, A, tq[0], tq[1], h_counts, lambda)
                                           : 0.0;
                if (do_split) {  /* both split, on different candidates */
                  gap = gain - gain_g;
                  bound = spread_best + spread_g;
                  if (gap <= ORC_NEAR_REL * fabs(gain)) kind = 1;
                  else if (tq && gap <= bound) kind = 2;
                } else {  /* the guide splits where this oracle's best gain is not above 0 */
                  gap = -gain_g;
                  bound = spread_g;
                  if (tq && gain_g > -spread_g && (!sp.valid || sp.gain - gain_g <= spread_best + spread_g)) kind = 2;
                }
              }
            }
            if (kind) {
              f = gf;
              b = gb;
              gain = gain_g;
              do_split = 1;
            }
          } else if (do_split) {  /* the guide makes a leaf where this oracle's best gain is above 0 */
            gap = gain;
            bound = spread_best;
            if (tq && gain <= spread_best) {
              kind = 2;
              do_split = 0;
            }
          }
          if (ti) {
            ti[v].guide_gap = gap;
            ti[v].guide_bound = bound;
            if (kind) ti[v].adopted = kind;
            else if (gf >= 0 && own_split) ti[v].guide_mismatch = 1;
          }
        }
        lvl_do[v - level_begin] = do_split;
        lvl_f[v - level_begin] = f;
        lvl_b[v - level_begin] = b;
        lvl_gain[v - level_begin] = gain;
      }
      /* phase 2: leaf budget (a reading of the ExaBoost page's depth-capped final partial
       * level).  If applying every split of this level would leave more than num_leaves leaves,
       * keep the first K = num_leaves - (leaves so far + this level's nodes) candidates in the
       * order (gain desc, node index asc), and make this the last level that splits. */
      if (p->num_leaves > 0 && d < last) {
        int32_t C = 0;
        for (int32_t i = 0; i < nl; ++i) C += lvl_do[i];
        const int32_t K = p->num_leaves - (leaves_done + nl);
        if (C > K) {
          for (int32_t i = 0; i < nl; ++i) {
            if (!lvl_do[i]) continue;
            int32_t rank = 0;
            for (int32_t j = 0; j < nl; ++j)
              if (lvl_do[j] && (lvl_gain[j] > lvl_gain[i] || (lvl_gain[j] == lvl_gain[i] && j < i))) ++rank;
            lvl_keep[i] = rank < K;
          }
          for (int32_t i = 0; i < nl; ++i) lvl_do[i] = lvl_do[i] && lvl_keep[i];
          last = d + 1;
        }
      }
      /* phase 3: apply the splits in node order */
      for (int32_t v = level_begin; v < level_end; ++v) {
        const int32_t i = v - level_begin;
        if (tg && d < D && ((tg[2 * v] >= 0) != (lvl_do[i] != 0)) && ti) ti[v].guide_mismatch = 1;
        if (!lvl_do[i]) {
          ++leaves_done;
          continue;
        }
        const int32_t f = lvl_f[i], b = lvl_b[i];
        const int64_t* rows = order + seg_start[v];
        const int64_t n = seg_count[v];
        orc_node* nd = &tn[v];

        /* stable partition of the node's rows: bin <= b left, others right */
        const uint8_t* col = bins + (int64_t)f * N;
        int64_t* dst = scratch + seg_start[v];
        int64_t w = 0;
        for (int64_t k = 0; k < n; ++k)
          if (col[rows[k]] <= b) dst[w++] = rows[k];
        const int64_t nlc = w;
        for (int64_t k = 0; k < n; ++k)
          if (!(col[rows[k]] <= b)) dst[w++] = rows[k];
        memcpy(order + seg_start[v], dst, sizeof(int64_t) * (size_t)n);

        int32_t L = n_nodes++, R = n_nodes++;
        nd->feature = f;
        nd->threshold_bin = b;
        nd->left = L;
        nd->right = R;
        nd->gain = lvl_gain[i];
        nd->is_leaf = 0;
        seg_start[L] = seg_start[v];
        seg_count[L] = nlc;
        seg_start[R] = seg_start[v] + nlc;
        seg_count[R] = n - nlc;
      }
      level_begin = level_end;
      level_end = n_nodes;
      if (level_begin == level_end) break;
    }
    nodes_per_tree[t] = n_nodes;

    /* [MPS-TC] s.6 step 7 / [LEAN] forward: pred += lr * w of the row's leaf */
    for (int32_t v = 0; v < n_nodes; ++v) {
      if (!tn[v].is_leaf) continue;
      const double step = p->learning_rate * tn[v].leaf_value;
      const int64_t* rows = order + seg_start[v];
      for (int64_t k = 0; k < seg_count[v]; ++k) {
        pred[rows[k]] = pred[rows[k]] + step;
        if (leaf_of_row && t == p->n_trees - 1) leaf_of_row[rows[k]] = v;
      }
    }
  }
  free(g), free(order), free(scratch), free(seg_start), free(seg_count), free(cnt), free(G), free(H);
  free(lvl_do), free(lvl_keep), free(lvl_f), free(lvl_b), free(lvl_gain);
  free(hv);
  return ORC_OK;
}

/*
 * Stable partition of one level's row-index segments (the oracle's own
 * restatement of the partition step, [MPS-TC] s.6 step 5).  For slot s with
 * split_feature[s] >= 0 the rows idx_in[seg_start[s] .. +seg_count[s]) are
 * written to idx_out at the same offset, those with bin <= split_bin[s] first,
 * both groups in their input order.  Slots without a split are copied.
 */
int orc_partition(const uint8_t* bins, int64_t N, int32_t n_slots, const int32_t* split_feature,
                  const int32_t* split_bin, const int64_t* seg_start, const int64_t* seg_count,
                  const int64_t* idx_in, int64_t* idx_out, int64_t* left_count) {
  if (!bins || !split_feature || !split_bin || !seg_start || !seg_count || !idx_in || !idx_out) return ORC_EINVAL;
  for (int32_t s = 0; s < n_slots; ++s) {
    const int64_t* in = idx_in + seg_start[s];
    int64_t* out = idx_out + seg_start[s];
    const int64_t n = seg_count[s];
    if (split_feature[s] < 0) {
      memcpy(out, in, sizeof(int64_t) * (size_t)n);
      if (left_count) left_count[s] = 0;
      continue;
    }
    const uint8_t* col = bins + (int64_t)split_feature[s] * N;
    int64_t w = 0;
    for (int64_t k = 0; k < n; ++k)
      if (col[in[k]] <= split_bin[s]) out[w++] = in[k];
    if (left_count) left_count[s] = w;
    for (int64_t k = 0; k < n; ++k)
      if (!(col[in[k]] <= split_bin[s])) out[w++] = in[k];
  }
  return ORC_OK;
}

/* [MPS-TC] s.6 step 7: pred_i + (lr * leaf_value[node_of_row[i]]). */
int orc_update_predictions(double* pred, const double* leaf_value, const int32_t* node_of_row, int64_t N,
                           double lr) {
  if (!pred || !leaf_value || !node_of_row) return ORC_EINVAL;
  for (int64_t i = 0; i < N; ++i) {
    const double step = lr * leaf_value[node_of_row[i]];
    pred[i] = pred[i] + step;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [LEAN] "Gradient boosted trees (spec model)", Forward pass and Tree        */
/* representation: the prediction of a row is init + learning_rate * (sum of */
/* its tree outputs), a tree sending x right when x > threshold.  On raw      */
/* features the threshold of split (feature j, bin b) is the edge             */
/* edges[j][b]: by the quantize rule bin(x) = #{edges < x}, so x > edges[b]   */
/* exactly when bin(x) > b, the training routing.  The sum is taken tree by   */
/* tree as in training ([MPS-TC] s.6 step 7): pred + (lr * leaf value).  A    */
/* NaN compares false and goes left.                                          */
int orc_predict(const float* X, int64_t N, int32_t F, const float* edges, int32_t max_bins, const orc_node* nodes,
                int32_t n_trees, int32_t max_nodes, double init, double lr, double* out) {
  if (!X || !edges || !out || N < 0 || F < 1 || max_bins < 2 || n_trees < 0 || (n_trees > 0 && !nodes) ||
      max_nodes < 1)
    return ORC_EINVAL;
  for (int64_t i = 0; i < N; ++i) {
    double pred = init;
    for (int32_t t = 0; t < n_trees; ++t) {
      const orc_node* tn = nodes + (int64_t)t * max_nodes;
      int32_t v = 0;
      for (int32_t steps = 0; !tn[v].is_leaf; ++steps) {
        if (steps > 64 || tn[v].feature < 0 || tn[v].feature >= F || tn[v].left < 0 || tn[v].right >= max_nodes)
          return ORC_EINVAL;
        const float x = X[(int64_t)tn[v].feature * N + i];
        const float thr = edges[(int64_t)tn[v].feature * (max_bins - 1) + tn[v].threshold_bin];
        v = x > thr ? tn[v].right : tn[v].left;
      }
      const double step = lr * tn[v].leaf_value;
      pred = pred + step;
    }
    out[i] = pred;
  }
  return ORC_OK;
}
