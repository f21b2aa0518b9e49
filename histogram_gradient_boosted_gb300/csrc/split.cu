// Split search of every slot of a level.
//
// "Module Design: Training Core" s.2: score(G,H) = G^2/(H+lambda),
// gain = 0.5*(score_L + score_R - score_P) - gamma; s.3: strict FP64 gain >,
// ties to the smaller feature then the smaller bin, invalid candidates never
// compared, split only on gain > 0, bin <= threshold goes left.
//
// One CTA per slot, one warp per feature at a time.  A lane holds 8
// consecutive bins; the warp forms prefix sums of (count, fixed-point G) with
// shuffles, evaluates every threshold in FP64 with explicitly rounded
// operations (no contraction), and reduces to the best candidate.  The
// comparison (gain desc, feature asc, bin asc) is a total order on distinct
// candidates, so the result does not depend on the reduction order.
#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitWarps = kSplitThreads / 32;

struct Cand {
  double gain;
  int feature;
  int bin;
  uint32_t cnt_left;
  int64_t q_left;
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
  return o;
}

__device__ __forceinline__ double score(double G, double H, double lambda) {
  return __ddiv_rn(__dmul_rn(G, G), __dadd_rn(H, lambda));
}

__global__ void __launch_bounds__(kSplitThreads)
    find_splits_kernel(const uint32_t* __restrict__ hist_cnt, const int64_t* __restrict__ hist_q,
                       const int32_t* __restrict__ fixed_exp, int32_t F, const int32_t* __restrict__ n_bins,
                       const gbdt_level* __restrict__ level, int32_t max_slots, double lambda, double gamma,
                       int32_t msl, double mcw, gbdt_split* __restrict__ out, int32_t* __restrict__ err) {
  const int slot = blockIdx.x;
  const int n_slots = min(level->n_slots, max_slots);
  if (slot >= n_slots) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = *fixed_exp;
  const double inv = ldexp(1.0, -S);
  __shared__ uint32_t s_tot_cnt;
  __shared__ long long s_tot_q;
  __shared__ Cand s_best[kSplitWarps];
  const int64_t base = static_cast<int64_t>(slot) * F * kBins;

  // node totals: sums over the bins of feature 0
  if (warp == 0) {
    const uint4* cp = reinterpret_cast<const uint4*>(hist_cnt + base + lane * 8);
    const longlong2* qp = reinterpret_cast<const longlong2*>(hist_q + base + lane * 8);
    uint4 c0 = cp[0], c1 = cp[1];
    uint32_t c = c0.x + c0.y + c0.z + c0.w + c1.x + c1.y + c1.z + c1.w;
    long long q = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      longlong2 v = qp[i];
      q += v.x + v.y;
    }
    for (int o = 16; o > 0; o >>= 1) {
      c += __shfl_xor_sync(0xffffffffu, c, o);
      q += __shfl_xor_sync(0xffffffffu, q, o);
    }
    if (lane == 0) {
      s_tot_cnt = c;
      s_tot_q = q;
    }
  }
  __syncthreads();
  const uint32_t tot_cnt = s_tot_cnt;
  const int64_t tot_q = s_tot_q;
  const double GP = static_cast<double>(tot_q) * inv;
  const double HP = static_cast<double>(tot_cnt);
  const double sP = score(GP, HP, lambda);

  Cand best{-INFINITY, -1, -1, 0, 0};
  for (int f = warp; f < F; f += kSplitWarps) {
    const int64_t off = base + static_cast<int64_t>(f) * kBins + lane * 8;
    const uint4* cp = reinterpret_cast<const uint4*>(hist_cnt + off);
    const longlong2* qp = reinterpret_cast<const longlong2*>(hist_q + off);
    uint32_t c[8];
    long long q[8];
    {
      uint4 a = cp[0], b = cp[1];
      c[0] = a.x, c[1] = a.y, c[2] = a.z, c[3] = a.w, c[4] = b.x, c[5] = b.y, c[6] = b.z, c[7] = b.w;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        longlong2 v = qp[i];
        q[2 * i] = v.x;
        q[2 * i + 1] = v.y;
      }
    }
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      c[i] += c[i - 1];
      q[i] += q[i - 1];
    }
    // exclusive warp scan of the lane totals
    uint32_t ci = c[7];
    long long qi = q[7];
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t cv = __shfl_up_sync(0xffffffffu, ci, o);
      long long qv = __shfl_up_sync(0xffffffffu, qi, o);
      if (lane >= o) {
        ci += cv;
        qi += qv;
      }
    }
    const uint32_t ce = ci - c[7];
    const long long qe = qi - q[7];
    // the feature's total must equal the node total (every row has one bin per feature)
    const uint32_t fc = __shfl_sync(0xffffffffu, ci, 31);
    const long long fq = __shfl_sync(0xffffffffu, qi, 31);
    if (lane == 0 && (fc != tot_cnt || fq != tot_q)) raise_error(err, kErrHistTotals);

    int nb = n_bins[f];
    nb = nb < 1 ? 1 : (nb > kBins ? kBins : nb);
    Cand lb{-INFINITY, -1, -1, 0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = lane * 8 + i;
      if (b > nb - 2) break;
      const uint32_t cL = ce + c[i];
      const int64_t qL = qe + q[i];
      const uint32_t cR = tot_cnt - cL;
      const int64_t qR = static_cast<int64_t>(static_cast<uint64_t>(tot_q) - static_cast<uint64_t>(qL));
      const double HL = static_cast<double>(cL), HR = static_cast<double>(cR);
      if (!(static_cast<int64_t>(cL) >= msl && static_cast<int64_t>(cR) >= msl && HL >= mcw && HR >= mcw &&
            HL > 0.0 && HR > 0.0))
        continue;
      const double GL = static_cast<double>(qL) * inv;
      const double GR = static_cast<double>(qR) * inv;
      const double sL = score(GL, HL, lambda), sR = score(GR, HR, lambda);
      const double gain = __dsub_rn(__dmul_rn(0.5, __dsub_rn(__dadd_rn(sL, sR), sP)), gamma);
      if (lb.feature < 0 || gain > lb.gain) lb = Cand{gain, f, b, cL, qL};
    }
    for (int o = 16; o > 0; o >>= 1) {
      Cand other = shfl_cand(lb, lane ^ o);
      if (better(other, lb)) lb = other;
    }
    if (better(lb, best)) best = lb;
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
    out[slot] = r;
  }
}

}  // namespace

void launch_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int32_t* fixed_exp, int32_t F,
                        const int32_t* n_bins, const gbdt_level* level, int32_t max_slots, const gbdt_params& p,
                        gbdt_split* out, int32_t* err, cudaStream_t s) {
  find_splits_kernel<<<max_slots, kSplitThreads, 0, s>>>(hist_cnt, hist_q, fixed_exp, F, n_bins, level, max_slots,
                                                          p.reg_lambda, p.gamma, p.min_samples_leaf,
                                                          p.min_child_weight, out, err);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

int validate_params(const gbdt_params* p);

extern "C" int gbdt_find_splits(const uint32_t* hist_cnt, const int64_t* hist_q, const int32_t* fixed_exp, int32_t F,
                                const int32_t* n_bins, const gbdt_level* level, int32_t max_slots,
                                const gbdt_params* p, gbdt_split* out, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(hist_cnt && hist_q && fixed_exp && n_bins && level && p && out, "gbdt_find_splits: null pointer");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096 && max_slots >= 1 && max_slots <= kMaxSlots,
                 "gbdt_find_splits: sizes out of range");
  GBDT_CHECK_ARG(aligned(hist_cnt, 16) && aligned(hist_q, 16), "gbdt_find_splits: histograms must be 16-byte aligned");
  int rc = validate_params(p);
  if (rc != GBDT_OK) return rc;
  launch_find_splits(hist_cnt, hist_q, fixed_exp, F, n_bins, level, max_slots, *p, out, nullptr,
                     static_cast<cudaStream_t>(stream));
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}
