// Split search of every slot of a level.
//
// "Module Design: Training Core" s.2: score(G,H) = G^2/(H+lambda),
// gain = 0.5*(score_L + score_R - score_P) - gamma; s.3: strict FP64 gain >,
// ties to the smaller feature then the smaller bin, invalid candidates never
// compared, split only on gain > 0, bin <= threshold goes left.
//
// Two phases.  Screen: one warp per (slot, feature); a lane holds 8
// consecutive bins, the warp forms prefix sums of (count, fixed-point G) with
// shuffles and screens every threshold in FP32 with a proven error margin,
// keeping the few that could reach the feature's maximum.  Select: one CTA per
// slot applies the same margin across all of the slot's features and
// evaluates only the survivors in FP64 with explicitly rounded operations (no
// contraction), reducing under the frozen rule.  FP64 is scarce on this GPU,
// so a node evaluates one or two thresholds in FP64 instead of one per
// feature.  The comparison (gain desc, feature asc, bin asc) is a total order
// on distinct candidates, so the result does not depend on the reduction
// order.  With the logistic objective H comes from the H histograms (fixed
// point with its own exponent) instead of the row counts; min_samples_leaf
// still applies to the counts.
#include <cmath>

#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kSplitThreads = 64;  // two warps: one feature each
constexpr int kSplitWarps = kSplitThreads / 32;

struct Cand {
  double gain;
  int feature;
  int bin;
  uint32_t cnt_left;
  int64_t q_left;
  int64_t qh_left;  // logistic: fixed-point H of the left side
};

// true if a is strictly preferred to b under the frozen rule
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  if (a.feature < 0) return false;
  if (b.feature < 0) return true;
  if (a.gain > b.gain) return true;
  if (a.gain < b.gain) return false;
  if (a.feature != b.feature) return a.feature < b.feature;
  return a.bin < b.bin;
}

__device__ __forceinline__ Cand shfl_cand(const Cand& c, int src) {
  Cand o;
  o.gain = __shfl_sync(0xffffffffu, c.gain, src);
  o.feature = __shfl_sync(0xffffffffu, c.feature, src);
  o.bin = __shfl_sync(0xffffffffu, c.bin, src);
  o.cnt_left = __shfl_sync(0xffffffffu, c.cnt_left, src);
  o.q_left = __shfl_sync(0xffffffffu, c.q_left, src);
  o.qh_left = __shfl_sync(0xffffffffu, c.qh_left, src);
  return o;
}

// |q| as a float within 3 ulps: the two 32-bit halves of |q|, both
// non-negative (no cancellation), converted and combined with one FMA.
__device__ __forceinline__ float abs_to_float(int64_t q) {
  const uint64_t a = q < 0 ? static_cast<uint64_t>(0) - static_cast<uint64_t>(q) : static_cast<uint64_t>(q);
  return __fmaf_rn(__uint2float_rn(static_cast<uint32_t>(a >> 32)), 4294967296.0f,
                   __uint2float_rn(static_cast<uint32_t>(a)));
}

__device__ __forceinline__ double score(double G, double H, double lambda) {
  return __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, lambda));
}

// Sum over the warp of the bins below nb (a lane holds bins 8 lane .. 8 lane + 7; lanes wholly at or above
// nb load nothing, the bins of a lane's last word at or above nb are masked out).
__device__ __forceinline__ long long warp_sum8(const int64_t* __restrict__ q, int lane, int nb) {
  long long s = 0;
  if (lane * 8 < nb) {
    const longlong2* qp = reinterpret_cast<const longlong2*>(q + lane * 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      longlong2 v = qp[i];
      s += (lane * 8 + 2 * i < nb ? v.x : 0) + (lane * 8 + 2 * i + 1 < nb ? v.y : 0);
    }
  }
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Node totals from feature 0 (every row has one bin per feature, below that feature's n_bins): warp-wide
// sums over its bins below nb0.  h (may be null): the H histogram, summed into *th.  Bins at or above a
// feature's n_bins are never read (the histogram passes do not write them).
__device__ __forceinline__ void node_totals(const uint32_t* __restrict__ cnt, const int64_t* __restrict__ q,
                                            const int64_t* __restrict__ h, int lane, int nb0, uint32_t* tc,
                                            long long* tq, long long* th) {
  uint32_t c = 0;
  if (lane * 8 < nb0) {
    const uint4* cp = reinterpret_cast<const uint4*>(cnt + lane * 8);
    const uint4 c0 = cp[0], c1 = cp[1];
    const uint32_t v[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) c += lane * 8 + i < nb0 ? v[i] : 0u;
  }
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  *tc = c;
  *tq = warp_sum8(q, lane, nb0);
  *th = h ? warp_sum8(h, lane, nb0) : 0;
}

// Eight bins of one lane (bins 8 lane .. 8 lane + 7) as inclusive prefix sums
// within the lane; returns the lane's exclusive offset over the warp and the
// feature's total (lane 31's inclusive sum) through *total.
// A threshold that survived its feature's FP32 screen.
constexpr int kSurv = 4;  // survivors kept per (slot, feature)
struct Surv {
  float x;            // its FP32 screening value; -1: empty entry
  int32_t bin;
  uint32_t cnt_left;
  int32_t exact;      // 1: gain holds its FP64 gain (its feature had more than kSurv survivors)
  int64_t q_left;
  int64_t qh_left;
  double gain;
};

// score of the node: G^2 / (H + lambda) from its fixed-point totals (H = count unless kH).
static_assert(sizeof(Surv) == 40, "Surv is five 8-byte words");
// A survivor written by another CTA of the same launch, read through L2.
__device__ __forceinline__ Surv load_surv(const Surv* p) {
  const long long* w = reinterpret_cast<const long long*>(p);
  long long v[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) v[i] = __ldcg(w + i);
  Surv s;
  memcpy(&s, v, sizeof(s));
  return s;
}

template <bool kH>
__device__ __forceinline__ double node_score(int64_t tot_q, uint32_t tot_cnt, int64_t tot_h, double inv,
                                             double inv_h, double lambda) {
  const double GP = static_cast<double>(tot_q) * inv;
  const double HP = kH ? static_cast<double>(tot_h) * inv_h : static_cast<double>(tot_cnt);
  return score(GP, HP, lambda);
}

// FP64 gain of the threshold whose left side holds (qL, cL, qhL) of the node totals, each
// operation rounded once: 0.5 * ((s_L + s_R) - s_P) - gamma.
template <bool kH>
__device__ __forceinline__ double exact_gain(int64_t qL, uint32_t cL, int64_t qhL, int64_t tot_q, uint32_t tot_cnt,
                                             int64_t tot_h, double inv, double inv_h, double sP, double lambda,
                                             double gamma) {
  const uint32_t cR = tot_cnt - cL;
  const int64_t qR = static_cast<int64_t>(static_cast<uint64_t>(tot_q) - static_cast<uint64_t>(qL));
  const int64_t qhR = static_cast<int64_t>(static_cast<uint64_t>(tot_h) - static_cast<uint64_t>(qhL));
  const double HL = kH ? static_cast<double>(qhL) * inv_h : static_cast<double>(cL);
  const double HR = kH ? static_cast<double>(qhR) * inv_h : static_cast<double>(cR);
  const double GL = static_cast<double>(qL) * inv;
  const double GR = static_cast<double>(qR) * inv;
  const double sL = score(GL, HL, lambda), sR = score(GR, HR, lambda);
  return __dsub_rn(__dmul_rn(0.5, __dsub_rn(__dadd_rn(sL, sR), sP)), gamma);
}

template <typename T>
__device__ __forceinline__ T lane_prefix8(T (&v)[8], int lane, T* total) {
#pragma unroll
  for (int i = 1; i < 8; ++i) v[i] += v[i - 1];
  T x = v[7];
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v[7];
}

// Where a slot's histogram comes from in training: a slot that was not built (the larger child of its
// pair) is its parent's histogram (the previous level's, pair_parent[slot / 2]) minus its built sibling's
// (slot ^ 1); the screen forms it, bin by bin, and also stores it (the next level subtracts from it).
// pc null: every slot's histogram is in place (the ABI call).
struct SubSrc {
  const uint32_t* pc;
  const int64_t* pq;
  const int64_t* ph;
  const int32_t* pair_parent;
  const uint8_t* build_flag;
};

// Screen of feature f of a slot (one warp).  Writes the feature's survivors of
// the FP32 screen to surv[slot][f][0 .. kSurv): in bin order, or, when more than
// kSurv survive (long runs of empty bins can tie), the best of them evaluated in
// FP64 as one exact entry.  kH: H from hist_h with exponent fixed_exp[1]
// (logistic), else H = the row count.  tot_*: the node totals.
template <bool kH, bool kNarrow>
__device__ __forceinline__ void screen_feature(const uint32_t* hist_cnt, const int64_t* hist_q,
                                               const int64_t* hist_h, const int32_t* __restrict__ fixed_exp,
                                               int32_t F, const int32_t* __restrict__ n_bins, int slot, int f, int lane,
                                               uint32_t tot_cnt, long long tot_q, long long tot_h, double lambda,
                                               double gamma, int32_t msl, double mcw, int64_t mcw_ceil,
                                               Surv* __restrict__ surv, int32_t* __restrict__ err, const SubSrc& src) {
  // kNarrow: this thread alone holds the whole feature (at most 8 bins: its bins 0..7), so every sum,
  // maximum and survivor count below is the thread's own; otherwise the warp holds it, 8 bins per lane
  const int sub = kNarrow ? 0 : lane;  // this thread's bins: 8 sub .. 8 sub + 7
  const int64_t base = static_cast<int64_t>(slot) * F * kBins;
  const int64_t off = base + static_cast<int64_t>(f) * kBins + sub * 8;
  int nb = n_bins[f];
  nb = nb < 1 ? 1 : (nb > kBins ? kBins : nb);
  // only the bins below nb are read (the histogram passes do not write the others): a lane wholly at or
  // above nb loads nothing, the bins of a lane's word at or above nb read as 0
  uint32_t c[8];
  long long q[8], qh[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = 0, q[i] = 0, qh[i] = 0;
  auto load8 = [&](const uint32_t* hc, const int64_t* hq, const int64_t* hh, int64_t o, uint32_t (&cc)[8],
                   long long (&qq)[8], long long (&hv)[8]) {
    const uint4* cp = reinterpret_cast<const uint4*>(hc + o);
    const longlong2* qp = reinterpret_cast<const longlong2*>(hq + o);
    const uint4 a = cp[0], b = cp[1];
    cc[0] = a.x, cc[1] = a.y, cc[2] = a.z, cc[3] = a.w, cc[4] = b.x, cc[5] = b.y, cc[6] = b.z, cc[7] = b.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const longlong2 v = qp[i];
      qq[2 * i] = v.x;
      qq[2 * i + 1] = v.y;
    }
    if (kH) {
      const longlong2* hp = reinterpret_cast<const longlong2*>(hh + o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const longlong2 v = hp[i];
        hv[2 * i] = v.x;
        hv[2 * i + 1] = v.y;
      }
    }
  };
  if (sub * 8 < nb) {
    if (src.pc && !src.build_flag[slot]) {  // parent minus the built sibling, stored for the next level
      const int64_t fo = static_cast<int64_t>(f) * kBins + sub * 8;
      const int64_t op = static_cast<int64_t>(src.pair_parent[slot >> 1]) * F * kBins + fo;
      const int64_t ob = static_cast<int64_t>(slot ^ 1) * F * kBins + fo;
      uint32_t bc[8];
      long long bq[8], bh[8];
      load8(src.pc, src.pq, src.ph, op, c, q, qh);
      load8(hist_cnt, hist_q, hist_h, ob, bc, bq, bh);
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        bad |= bc[i] > c[i] && sub * 8 + i < nb;
        c[i] -= bc[i];
        q[i] = static_cast<long long>(static_cast<unsigned long long>(q[i]) - static_cast<unsigned long long>(bq[i]));
        if (kH)
          qh[i] = static_cast<long long>(static_cast<unsigned long long>(qh[i]) - static_cast<unsigned long long>(bh[i]));
      }
      if (bad) raise_error(err, kErrHistTotals);
      uint4* cs = reinterpret_cast<uint4*>(const_cast<uint32_t*>(hist_cnt) + off);
      longlong2* qs = reinterpret_cast<longlong2*>(const_cast<int64_t*>(hist_q) + off);
      cs[0] = make_uint4(c[0], c[1], c[2], c[3]);
      cs[1] = make_uint4(c[4], c[5], c[6], c[7]);
#pragma unroll
      for (int i = 0; i < 4; ++i) qs[i] = make_longlong2(q[2 * i], q[2 * i + 1]);
      if (kH) {
        longlong2* hs = reinterpret_cast<longlong2*>(const_cast<int64_t*>(hist_h) + off);
#pragma unroll
        for (int i = 0; i < 4; ++i) hs[i] = make_longlong2(qh[2 * i], qh[2 * i + 1]);
      }
    } else {
      load8(hist_cnt, hist_q, hist_h, off, c, q, qh);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (sub * 8 + i >= nb) c[i] = 0, q[i] = 0, qh[i] = 0;
  }
  // A threshold whose own bin is empty has the same left side (count, G, H) as the threshold before
  // it, hence the same gain, and loses the tie to that smaller bin: only thresholds at non-empty bins
  // are candidates (runs of empty bins would otherwise all tie and survive the screen together).
  uint32_t filled = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) filled |= (c[i] != 0 ? 1u : 0u) << i;
  // prefix sums over the bins; the feature's totals must equal the node totals
  uint32_t fc, ce;
  long long fq, fh = 0, qe, he;
  if constexpr (kNarrow) {
#pragma unroll
    for (int i = 1; i < 8; ++i) c[i] += c[i - 1], q[i] += q[i - 1], qh[i] += qh[i - 1];
    ce = 0, qe = 0, he = 0;
    fc = c[7], fq = q[7], fh = kH ? qh[7] : 0;
  } else {
    ce = lane_prefix8(c, lane, &fc);
    qe = lane_prefix8(q, lane, &fq);
    he = kH ? lane_prefix8(qh, lane, &fh) : 0;
  }
  if ((kNarrow || lane == 0) && (fc != tot_cnt || fq != tot_q || (kH && fh != tot_h))) raise_error(err, kErrHistTotals);

  // Screening in FP32.  Within a node the gain is a non-decreasing function of
  // x = qL^2/(HL+lambda) + qR^2/(HR+lambda) (fixed-point units; score_P,
  // gamma and the scale are the node's constants).  x is a sum of two
  // non-negative terms, so its FP32 value (|q| converted within 3 ulps, the
  // division within 2 ulps, H + lambda, the square and the sum rounded once
  // each) is within 12 * 2^-24 relative of the exact one; every candidate
  // that could reach the FP64 maximum (ties included) has
  // x32 >= max x32 * (1 - 2^-16), and only those are evaluated in FP64.  The
  // chosen candidate is the one a full FP64 scan would choose.
  // With H from the H histogram (kH) the screen uses the node-relative form
  // (qL 2^-31)^2 / (qhL / qhP + lambda / HP), a positive multiple of the same
  // x, whose terms stay in FP32's range however small H is (|qL| 2^-31 <= 2^31,
  // qhL / qhP >= 2^-62); its conversions and one more division keep it within
  // 20 * 2^-24 relative, far inside the margin.  (lambda / HP beyond FP32's
  // range makes every term 0: every candidate is then kept.)
  // an integer count c satisfies c >= msl, c >= mcw and c > 0 iff c >= cnt_min; a fixed-point H
  // qh * 2^-S_h satisfies H >= mcw and H > 0 iff qh >= qh_min (mcw * 2^S_h is exact in FP64)
  const int64_t cnt_min = max(max(static_cast<int64_t>(msl), int64_t(1)), mcw_ceil);
  int64_t qh_min = 1;
  if (kH) {
    const double m = ceil(ldexp(mcw, fixed_exp[1]));
    qh_min = m >= 9.2e18 ? INT64_MAX : max(int64_t(1), static_cast<int64_t>(m));
  }
  const float lam = static_cast<float>(lambda);
  const float hpf = kH ? abs_to_float(tot_h) : 1.0f;
  const float lamn = kH ? static_cast<float>(lambda / (static_cast<double>(tot_h) * ldexp(1.0, -fixed_exp[1]))) : 0.0f;
  float x32[8];
  uint32_t ok = 0;
  float xmax = -1.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int b = sub * 8 + i;
    const uint32_t cL = ce + c[i];
    const int64_t qL = qe + q[i];
    const uint32_t cR = tot_cnt - cL;
    const int64_t qR = static_cast<int64_t>(static_cast<uint64_t>(tot_q) - static_cast<uint64_t>(qL));
    const int64_t qhL = kH ? he + qh[i] : 0;
    const int64_t qhR = kH ? static_cast<int64_t>(static_cast<uint64_t>(tot_h) - static_cast<uint64_t>(qhL)) : 0;
    x32[i] = 0.0f;
    if (b > nb - 2 || !(filled >> i & 1u)) continue;
    // validity in integers (the FP64 pipe is scarce): H = count, so count >= msl, H >= mcw and H > 0
    // are count >= cnt_min; with H from its histogram, H >= mcw and H > 0 are qh >= qh_min
    if (kH ? !(static_cast<int64_t>(cL) >= msl && static_cast<int64_t>(cR) >= msl && qhL >= qh_min && qhR >= qh_min)
           : !(static_cast<int64_t>(cL) >= cnt_min && static_cast<int64_t>(cR) >= cnt_min))
      continue;
    float x;
    if (kH) {
      const float gl = abs_to_float(qL) * 0x1p-31f, gr = abs_to_float(qR) * 0x1p-31f;
      const float hl = __fdividef(abs_to_float(qhL), hpf), hr = __fdividef(abs_to_float(qhR), hpf);
      x = __fadd_rn(__fdividef(__fmul_rn(gl, gl), __fadd_rn(hl, lamn)),
                    __fdividef(__fmul_rn(gr, gr), __fadd_rn(hr, lamn)));
    } else {
      const float gl = abs_to_float(qL), gr = abs_to_float(qR);
      x = __fadd_rn(__fdividef(__fmul_rn(gl, gl), __fadd_rn(static_cast<float>(cL), lam)),
                    __fdividef(__fmul_rn(gr, gr), __fadd_rn(static_cast<float>(cR), lam)));
    }
    x32[i] = x;
    ok |= 1u << i;
    xmax = fmaxf(xmax, x);
  }
  if constexpr (!kNarrow)
    for (int o = 16; o > 0; o >>= 1) xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, o));
  const float keep = xmax - xmax * 1.52587890625e-05f;  // xmax * (1 - 2^-16)
  uint32_t sv = 0;  // this lane's survivors
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((ok >> i & 1u) && x32[i] >= keep) sv |= 1u << i;
  const int mine = __popc(sv);
  int before = mine, total = mine;  // inclusive prefix over lanes (lanes hold consecutive bins)
  if constexpr (!kNarrow) {
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, before, o);
      if (lane >= o) before += v;
    }
    total = __shfl_sync(0xffffffffu, before, 31);
  }
  before -= mine;
  Surv* out = surv + (static_cast<int64_t>(slot) * F + f) * kSurv;
  if (total <= kSurv) {
    int k = before;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!(sv >> i & 1u)) continue;
      const uint32_t cL = ce + c[i];
      out[k++] = Surv{x32[i], sub * 8 + i, cL, 0, qe + q[i], kH ? he + qh[i] : 0, 0.0};
    }
    if constexpr (kNarrow) {
      for (int e = total; e < kSurv; ++e) out[e] = Surv{-1.0f, -1, 0, 0, 0, 0, 0.0};
    } else {
      if (lane >= total && lane < kSurv) out[lane] = Surv{-1.0f, -1, 0, 0, 0, 0, 0.0};
    }
    return;
  }
  // more survivors than entries: evaluate them all in FP64 here and keep the best
  const double inv = ldexp(1.0, -fixed_exp[0]), inv_h = kH ? ldexp(1.0, -fixed_exp[1]) : 1.0;
  const double sP = node_score<kH>(tot_q, tot_cnt, tot_h, inv, inv_h, lambda);
  Cand lb{-INFINITY, -1, -1, 0, 0, 0};
  float lx = -1.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!(sv >> i & 1u)) continue;
    const uint32_t cL = ce + c[i];
    const int64_t qL = qe + q[i], qhL = kH ? he + qh[i] : 0;
    const double gain = exact_gain<kH>(qL, cL, qhL, tot_q, tot_cnt, tot_h, inv, inv_h, sP, lambda, gamma);
    if (lb.feature < 0 || gain > lb.gain) lb = Cand{gain, f, sub * 8 + i, cL, qL, qhL}, lx = x32[i];
  }
  if constexpr (kNarrow) {
    out[0] = Surv{lx, lb.bin, lb.cnt_left, 1, lb.q_left, lb.qh_left, lb.gain};
    for (int e = 1; e < kSurv; ++e) out[e] = Surv{-1.0f, -1, 0, 0, 0, 0, 0.0};
  } else {
    for (int o = 16; o > 0; o >>= 1) {
      const Cand other = shfl_cand(lb, lane ^ o);
      const float ox = __shfl_xor_sync(0xffffffffu, lx, o);
      if (better(other, lb)) lb = other, lx = ox;
    }
    if (lane == 0) out[0] = Surv{lx, lb.bin, lb.cnt_left, 1, lb.q_left, lb.qh_left, lb.gain};
    if (lane >= 1 && lane < kSurv) out[lane] = Surv{-1.0f, -1, 0, 0, 0, 0, 0.0};
  }
}

// Select for one slot (the whole 64-thread CTA).  The FP32 margin holds across the slot's features
// (x is the same monotone proxy of the gain everywhere in a node), so only survivors within it of
// the largest screening value of the slot are evaluated in FP64 (exact entries carry their gain),
// then reduced under the frozen rule.  The survivors were written by other CTAs: they are read
// through L2 (ld.global.cg).
template <bool kH>
__device__ __forceinline__ void select_slot(const uint32_t* __restrict__ hist_cnt, const int64_t* __restrict__ hist_q,
                                            const int64_t* __restrict__ hist_h, const int32_t* __restrict__ fixed_exp,
                                            int32_t F, int slot, uint32_t tot_cnt, long long tot_q, long long tot_h,
                                            double lambda, double gamma, const Surv* __restrict__ surv,
                                            gbdt_split* __restrict__ out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ Cand s_best[kSplitWarps];
  __shared__ float s_x[kSplitWarps];
  const Surv* sv = surv + static_cast<int64_t>(slot) * F * kSurv;
  const int n = F * kSurv;
  float xmax = -1.0f;
#pragma unroll 4
  for (int e = threadIdx.x; e < n; e += blockDim.x) xmax = fmaxf(xmax, __ldcg(&sv[e].x));
  for (int o = 16; o > 0; o >>= 1) xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, o));
  if (lane == 0) s_x[warp] = xmax;
  __syncthreads();
  for (int w = 0; w < kSplitWarps; ++w) xmax = fmaxf(xmax, s_x[w]);
  const float keep = xmax - xmax * 1.52587890625e-05f;  // xmax * (1 - 2^-16)
  const double inv = ldexp(1.0, -fixed_exp[0]), inv_h = kH ? ldexp(1.0, -fixed_exp[1]) : 1.0;
  double sP = 0.0;
  bool have_sP = false;
  Cand best{-INFINITY, -1, -1, 0, 0, 0};
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const Surv c = load_surv(sv + e);
    if (c.bin < 0 || c.x < keep) continue;
    double gain = c.gain;
    if (!c.exact) {
      if (!have_sP) sP = node_score<kH>(tot_q, tot_cnt, tot_h, inv, inv_h, lambda), have_sP = true;
      gain = exact_gain<kH>(c.q_left, c.cnt_left, c.qh_left, tot_q, tot_cnt, tot_h, inv, inv_h, sP, lambda, gamma);
    }
    const Cand cd{gain, e / kSurv, c.bin, c.cnt_left, c.q_left, c.qh_left};
    if (better(cd, best)) best = cd;
  }
  for (int o = 16; o > 0; o >>= 1) {
    Cand other = shfl_cand(best, lane ^ o);
    if (better(other, best)) best = other;
  }
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    Cand b = s_best[0];
    for (int w = 1; w < kSplitWarps; ++w)
      if (better(s_best[w], b)) b = s_best[w];
    gbdt_split r;
    const bool split = b.feature >= 0 && b.gain > 0.0;
    r.feature = split ? b.feature : -1;
    r.bin = split ? b.bin : -1;
    r.gain = split ? b.gain : 0.0;
    r.q_left = split ? b.q_left : 0;
    r.cnt_left = split ? b.cnt_left : 0;
    r.q_total = tot_q;
    r.cnt_total = tot_cnt;
    r.h_left = split ? b.qh_left : 0;
    r.h_total = kH ? tot_h : 0;
    out[slot] = r;
  }
}

// One CTA of two warps per (slot, pair of features): each warp screens one feature; the CTA that
// finishes a slot last (a per-slot counter, which that CTA resets to 0 for the next launch)
// selects the slot's split.  No CTA waits for another.
template <bool kH>
__global__ void __launch_bounds__(kSplitThreads)
    split_kernel(const uint32_t* hist_cnt, const int64_t* hist_q, const int64_t* hist_h,
                 const int32_t* __restrict__ fixed_exp, int32_t F, const int32_t* __restrict__ n_bins,
                 const gbdt_level* __restrict__ level, int32_t max_slots, double lambda, double gamma, int32_t msl,
                 double mcw, int64_t mcw_ceil, Surv* __restrict__ surv, int32_t* __restrict__ slot_done,
                 gbdt_split* __restrict__ out, int32_t* __restrict__ err, const int32_t* __restrict__ fsched,
                 int32_t n_wide, int32_t n_narrow, const SlotTotals* __restrict__ totals, SubSrc src) {
  const int slot = blockIdx.x;
  const int n_slots = min(level->n_slots, max_slots);
  if (slot >= n_slots) return;  // every CTA of this slot
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the features of this CTA: the first ceil(n_wide / 2) CTAs of a slot take two wide features (a warp
  // each), the others kSplitThreads narrow ones (a thread each); fsched (null: every feature wide, in
  // order) lists the wide features, then the narrow ones
  const int wide_ctas = (n_wide + kSplitWarps - 1) / kSplitWarps;
  const bool narrow = static_cast<int>(blockIdx.y) >= wide_ctas;
  int f = -1;
  if (!narrow) {
    const int j = blockIdx.y * kSplitWarps + warp;
    if (j < n_wide) f = fsched ? fsched[j] : j;
  } else {
    const int j = (blockIdx.y - wide_ctas) * kSplitThreads + threadIdx.x;
    if (j < n_narrow) f = fsched[n_wide + j];
  }
  const int64_t base = static_cast<int64_t>(slot) * F * kBins;
  uint32_t tot_cnt;
  long long tot_q, tot_h;
  if (totals) {  // the expected totals: every feature's histogram is checked against them below
    const SlotTotals t = totals[slot];
    tot_cnt = t.cnt;
    tot_q = t.q;
    tot_h = kH ? t.qh : 0;
  } else {
    const int nb0 = min(max(n_bins[0], 1), kBins);
    node_totals(hist_cnt + base, hist_q + base, kH ? hist_h + base : nullptr, lane, nb0, &tot_cnt, &tot_q, &tot_h);
  }
  if (f >= 0 && narrow)
    screen_feature<kH, true>(hist_cnt, hist_q, hist_h, fixed_exp, F, n_bins, slot, f, lane, tot_cnt, tot_q, tot_h,
                             lambda, gamma, msl, mcw, mcw_ceil, surv, err, src);
  else if (f >= 0)  // warp-uniform
    screen_feature<kH, false>(hist_cnt, hist_q, hist_h, fixed_exp, F, n_bins, slot, f, lane, tot_cnt, tot_q, tot_h,
                              lambda, gamma, msl, mcw, mcw_ceil, surv, err, src);
  __shared__ int s_last;
  __threadfence();  // this CTA's survivors are visible device-wide before it is counted
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&slot_done[slot], 1) == static_cast<int>(gridDim.y) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  select_slot<kH>(hist_cnt, hist_q, hist_h, fixed_exp, F, slot, tot_cnt, tot_q, tot_h, lambda, gamma, surv, out);
  if (threadIdx.x == 0) slot_done[slot] = 0;
}

}  // namespace

// Scratch: the per-slot counters (kMaxSlots of them, at a fixed place so that every level's launch
// finds them zero), then the survivors [max_slots][F][kSurv].
constexpr size_t kCounterBytes = sizeof(int32_t) * kMaxSlots;

size_t find_splits_scratch_bytes(int32_t F, int32_t max_slots) {
  return kCounterBytes + sizeof(Surv) * kSurv * static_cast<size_t>(F) * static_cast<size_t>(max_slots);
}

int32_t* split_counters(void* scratch, int32_t F, int32_t max_slots) {
  (void)F, (void)max_slots;
  return static_cast<int32_t*>(scratch);
}

void launch_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int64_t* hist_h,
                        const int32_t* fixed_exp, int32_t F, const int32_t* n_bins, const gbdt_level* level,
                        int32_t max_slots, const gbdt_params& p, gbdt_split* out, void* scratch, int32_t* err,
                        cudaStream_t s, const int32_t* fsched, int32_t n_narrow, const SlotTotals* totals,
                        const uint32_t* prev_cnt, const int64_t* prev_q, const int64_t* prev_h,
                        const int32_t* pair_parent, const uint8_t* build_flag) {
  const SubSrc src{prev_cnt, prev_q, prev_h, pair_parent, build_flag};
  int32_t* done = split_counters(scratch, F, max_slots);
  Surv* surv = reinterpret_cast<Surv*>(static_cast<char*>(scratch) + kCounterBytes);
  if (!fsched) n_narrow = 0;
  const int n_wide = F - n_narrow;
  const int ctas = (n_wide + kSplitWarps - 1) / kSplitWarps + (n_narrow + kSplitThreads - 1) / kSplitThreads;
  dim3 grid(static_cast<unsigned>(max_slots), static_cast<unsigned>(ctas));
  // ceil(min_child_weight) for the count test (counts are below 2^32)
  const double cm = std::ceil(p.min_child_weight);
  const int64_t mcw_ceil = cm > 8.0e9 ? int64_t(8000000000) : static_cast<int64_t>(cm);
  if (hist_h)
    split_kernel<true><<<grid, kSplitThreads, 0, s>>>(hist_cnt, hist_q, hist_h, fixed_exp, F, n_bins, level,
                                                      max_slots, p.reg_lambda, p.gamma, p.min_samples_leaf,
                                                      p.min_child_weight, mcw_ceil, surv, done, out, err, fsched,
                                                      n_wide, n_narrow, totals, src);
  else
    split_kernel<false><<<grid, kSplitThreads, 0, s>>>(hist_cnt, hist_q, nullptr, fixed_exp, F, n_bins, level,
                                                       max_slots, p.reg_lambda, p.gamma, p.min_samples_leaf,
                                                       p.min_child_weight, mcw_ceil, surv, done, out, err, fsched,
                                                      n_wide, n_narrow, totals, src);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

int validate_params(const gbdt_params* p);

extern "C" size_t gbdt_find_splits_workspace_size(int32_t F, int32_t max_slots) {
  return find_splits_scratch_bytes(F, max_slots) + kWsAlign;
}

extern "C" int gbdt_find_splits_h(const uint32_t* hist_cnt, const int64_t* hist_q, const int64_t* hist_h,
                                  const int32_t* fixed_exp, int32_t F, const int32_t* n_bins, const gbdt_level* level,
                                  int32_t max_slots, const gbdt_params* p, gbdt_split* out, void* ws,
                                  size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(hist_cnt && hist_q && fixed_exp && n_bins && level && p && out, "gbdt_find_splits: null pointer");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096 && max_slots >= 1 && max_slots <= kMaxSlots,
                 "gbdt_find_splits: sizes out of range");
  GBDT_CHECK_ARG(aligned(hist_cnt, 16) && aligned(hist_q, 16) && aligned(hist_h, 16),
                 "gbdt_find_splits: histograms must be 16-byte aligned");
  int rc = validate_params(p);
  if (rc != GBDT_OK) return rc;
  if (!ws || ws_bytes < gbdt_find_splits_workspace_size(F, max_slots) || !aligned(ws, kWsAlign)) {
    set_error("gbdt_find_splits: workspace needs %zu bytes", gbdt_find_splits_workspace_size(F, max_slots));
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the workspace: the call's error word (gbdt_workspace_status), then the search's scratch
  int32_t* err = static_cast<int32_t*>(ws);
  void* scratch = static_cast<char*>(ws) + kWsAlign;
  GBDT_CUDA(cudaMemsetAsync(err, 0, sizeof(int32_t), s));
  GBDT_CUDA(cudaMemsetAsync(split_counters(scratch, F, max_slots), 0, sizeof(int32_t) * max_slots, s));
  launch_find_splits(hist_cnt, hist_q, hist_h, fixed_exp, F, n_bins, level, max_slots, *p, out, scratch, err, s);
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" int gbdt_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int32_t* fixed_exp, int32_t F,
                                const int32_t* n_bins, const gbdt_level* level, int32_t max_slots,
                                const gbdt_params* p, gbdt_split* out, void* ws, size_t ws_bytes, void* stream) {
  return gbdt_find_splits_h(hist_cnt, hist_q, nullptr, fixed_exp, F, n_bins, level, max_slots, p, out, ws, ws_bytes,
                            stream);
}
