// Level histogram construction and sibling subtraction.
//
// "Module Design: Training Core" s.6 step 2 (build node histograms for the
// active nodes of a level) and s.7 (count/G/H per bin; H = count for squared
// error since h = 1).  All flagged slots of a level are built in one launch.
//
// Design (GB300):
//  * bins are column-major uint8; each thread owns 16 consecutive rows and
//    reads them with one 16-byte load per feature;
//  * each CTA privatises the histograms of a group of slots x features in
//    shared memory and merges them into global memory once, at its end;
//  * G is accumulated as exact fixed point (q = rint(g*2^S), int64) using only
//    32-bit shared atomics, because 64-bit shared atomics are emulated and
//    several times slower on this part: per entry a count word, a low word
//    that detects its own carry from the value atomicAdd returns, and a high
//    word that is touched only when the high half of q plus that carry is
//    non-zero.  Integer sums make the result independent of thread order;
//  * the larger sibling is parent minus the smaller one (exact on integers).
#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kHistThreads = 1024;
constexpr int kRowsPerThread = 16;
constexpr int kMaxGroupEntries = 64 * kBins;  // slots x features x bins per CTA
constexpr size_t kHistSmemCap = 227 * 1024 - 1024;  // opt-in limit minus the kernel's static shared memory

// Exclusive ranks of flagged slots; s_rank[s] = rank or -1.  Returns the flag count.
__device__ int rank_flags(const uint8_t* __restrict__ flag, int n_slots, int16_t* s_rank, int* s_scratch) {
  const int per = (n_slots + blockDim.x - 1) / blockDim.x;
  const int b0 = threadIdx.x * per;
  const int b1 = min(n_slots, b0 + per);
  int c = 0;
  for (int s = b0; s < b1; ++s) c += flag[s] ? 1 : 0;
  // block exclusive scan over threads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = c;
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_scratch[lane] : 0;
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    if (lane < nw) s_scratch[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) s_scratch[32] = wi;        // total
  }
  __syncthreads();
  int r = s_scratch[warp] + incl - c;
  for (int s = b0; s < b1; ++s) {
    if (flag[s]) {
      s_rank[s] = static_cast<int16_t>(r);
      ++r;
    } else {
      s_rank[s] = -1;
    }
  }
  const int total = s_scratch[32];
  __syncthreads();
  return total;
}

template <typename GT>
__device__ __forceinline__ void load_g16(const GT* __restrict__ g, int64_t r0, int64_t N, double* out);

template <>
__device__ __forceinline__ void load_g16<double>(const double* __restrict__ g, int64_t r0, int64_t N, double* out) {
  if (r0 + kRowsPerThread <= N) {
    const double2* p = reinterpret_cast<const double2*>(g + r0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      double2 v = __ldg(p + i);
      out[2 * i] = v.x;
      out[2 * i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) out[i] = (r0 + i < N) ? g[r0 + i] : 0.0;
  }
}

template <>
__device__ __forceinline__ void load_g16<float>(const float* __restrict__ g, int64_t r0, int64_t N, double* out) {
  if (r0 + kRowsPerThread <= N) {
    const float4* p = reinterpret_cast<const float4*>(g + r0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 v = __ldg(p + i);
      out[4 * i] = v.x;
      out[4 * i + 1] = v.y;
      out[4 * i + 2] = v.z;
      out[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) out[i] = (r0 + i < N) ? static_cast<double>(g[r0 + i]) : 0.0;
  }
}

// Add q (and one row) to shared entry e using 32-bit atomics only.
__device__ __forceinline__ void add_entry(uint32_t* s_cnt, uint32_t* s_lo, int32_t* s_hi, int e, int64_t q) {
  atomicAdd(s_cnt + e, 1u);
  const uint32_t ql = static_cast<uint32_t>(static_cast<uint64_t>(q));
  int32_t qh = static_cast<int32_t>(q >> 32);
  const uint32_t old = atomicAdd(s_lo + e, ql);
  qh += (old + ql < old) ? 1 : 0;  // carry out of the low word
  if (qh != 0) atomicAdd(s_hi + e, qh);
}

template <typename GT>
__global__ void __launch_bounds__(kHistThreads, 1)
    hist_build_kernel(const uint8_t* __restrict__ bins, int64_t ldb, int64_t N, int32_t F, const GT* __restrict__ g,
                      const int32_t* __restrict__ fixed_exp, const uint16_t* __restrict__ node_of_row,
                      const gbdt_level* __restrict__ level, int32_t max_slots, const uint8_t* __restrict__ build_flag,
                      int32_t group_slots, int32_t group_feats, int32_t n_fgroups, int32_t n_chunks,
                      int64_t rows_per_chunk, uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q,
                      int32_t* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int entries = group_slots * group_feats * kBins;
  uint32_t* s_cnt = reinterpret_cast<uint32_t*>(smem);
  uint32_t* s_lo = s_cnt + entries;
  int32_t* s_hi = reinterpret_cast<int32_t*>(s_lo + entries);
  int16_t* s_rank = reinterpret_cast<int16_t*>(s_hi + entries);   // [max_slots]
  int32_t* s_slot = reinterpret_cast<int32_t*>(s_rank + ((max_slots + 7) & ~7));  // [group_slots]
  __shared__ int s_scratch[33];

  const int chunk = blockIdx.x % n_chunks;
  const int fgroup = (blockIdx.x / n_chunks) % n_fgroups;
  const int sgroup = blockIdx.x / (n_chunks * n_fgroups);

  const int node_begin = level->node_begin;
  int n_slots = level->n_slots;
  if (n_slots > max_slots) {
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(err, kErrLevelSize);
    n_slots = max_slots;
  }
  const int n_build = rank_flags(build_flag, n_slots, s_rank, s_scratch);
  const int k_lo = sgroup * group_slots;
  if (k_lo >= n_build) return;  // no built slot in this group (uniform per block)
  const int f_lo = fgroup * group_feats;
  const int nf = min(group_feats, F - f_lo);
  if (nf <= 0) return;

  for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
    const int r = s_rank[s];
    if (r >= k_lo && r < k_lo + group_slots) s_slot[r - k_lo] = s;
  }
  for (int e = threadIdx.x; e < entries; e += blockDim.x) {
    s_cnt[e] = 0;
    s_lo[e] = 0;
    s_hi[e] = 0;
  }
  __syncthreads();

  const int S = *fixed_exp;
  const double scale = ldexp(1.0, S);
  const int64_t c0 = static_cast<int64_t>(chunk) * rows_per_chunk;
  const int64_t c1 = min(N, c0 + rows_per_chunk);

  for (int64_t r0 = c0 + static_cast<int64_t>(threadIdx.x) * kRowsPerThread; r0 < c1;
       r0 += static_cast<int64_t>(blockDim.x) * kRowsPerThread) {
    // group-local slot index of each of the 16 rows, -1 if the row is not ours
    int k[kRowsPerThread];
    bool any = false;
    if (r0 + kRowsPerThread <= N) {
      const uint4* np = reinterpret_cast<const uint4*>(node_of_row + r0);
      uint4 a = __ldg(np), b = __ldg(np + 1);
      uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        k[2 * i] = static_cast<int>(w[i] & 0xffffu);
        k[2 * i + 1] = static_cast<int>(w[i] >> 16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) k[i] = (r0 + i < N) ? static_cast<int>(node_of_row[r0 + i]) : -1;
    }
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int slot = k[i] - node_begin;
      int kk = -1;
      if (k[i] >= 0 && slot >= 0 && slot < n_slots) {
        const int r = s_rank[slot];
        if (r >= k_lo && r < k_lo + group_slots) kk = r - k_lo;
      }
      k[i] = kk;
      any |= kk >= 0;
    }
    if (!any) continue;
    double gv[kRowsPerThread];
    load_g16<GT>(g, r0, N, gv);
    int64_t q[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) q[i] = to_fixed(gv[i], scale);

    for (int fl = 0; fl < nf; ++fl) {
      const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bins + static_cast<int64_t>(f_lo + fl) * ldb + r0));
      const uint32_t words[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        if (k[i] >= 0) {
          const int b = (words[i >> 2] >> (8 * (i & 3))) & 0xff;
          add_entry(s_cnt, s_lo, s_hi, ((k[i] * group_feats + fl) << 8) | b, q[i]);
        }
      }
    }
  }
  __syncthreads();

  // merge into global memory: one 32-bit and one 64-bit atomic per non-empty entry
  const int n_local = min(group_slots, n_build - k_lo);
  const int used = n_local * group_feats * kBins;
  for (int e = threadIdx.x; e < used; e += blockDim.x) {
    const uint32_t c = s_cnt[e];
    if (c == 0) continue;
    const int b = e & 0xff;
    const int fl = (e >> 8) % group_feats;
    const int kk = (e >> 8) / group_feats;
    if (fl >= nf) continue;
    const int64_t v = static_cast<int64_t>(s_hi[e]) * 4294967296ll + static_cast<int64_t>(s_lo[e]);
    const int64_t o = (static_cast<int64_t>(s_slot[kk]) * F + (f_lo + fl)) * kBins + b;
    atomicAdd(hist_cnt + o, c);
    atomicAdd(reinterpret_cast<unsigned long long*>(hist_q + o), static_cast<unsigned long long>(v));
  }
}

// Both passes below take four consecutive bins of one feature per thread (16-byte loads and stores; a
// slot's F x 256 entries are a multiple of 4 and every slot starts 16-byte aligned).  n_bins (may be
// null): only the bins below each feature's n_bins are touched (the training's histogram passes never
// write the others and its split search never reads them); null: every bin.
__device__ __forceinline__ bool quad_used(const int32_t* __restrict__ n_bins, int64_t e) {
  return !n_bins || static_cast<int>(e & (kBins - 1)) < n_bins[e >> 8];
}

__global__ void __launch_bounds__(256)
    hist_zero_kernel(const gbdt_level* __restrict__ level, int32_t max_slots, const uint8_t* __restrict__ build_flag,
                     int32_t F, uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q,
                     int64_t* __restrict__ hist_h, const uint32_t* __restrict__ cnt0,
                     const int32_t* __restrict__ n_bins) {
  const int n_slots = min(level->n_slots, max_slots);
  const int slot = blockIdx.y;
  if (slot >= n_slots || !build_flag[slot]) return;
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;
  const int64_t e = 4 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (e >= per_slot || !quad_used(n_bins, e)) return;
  const int64_t o = slot * per_slot + e;
  *reinterpret_cast<uint4*>(hist_cnt + o) =
      (cnt0 && slot == 0) ? *reinterpret_cast<const uint4*>(cnt0 + e) : make_uint4(0, 0, 0, 0);
  const longlong2 z = make_longlong2(0, 0);
  reinterpret_cast<longlong2*>(hist_q + o)[0] = z;
  reinterpret_cast<longlong2*>(hist_q + o)[1] = z;
  if (hist_h) {
    reinterpret_cast<longlong2*>(hist_h + o)[0] = z;
    reinterpret_cast<longlong2*>(hist_h + o)[1] = z;
  }
}

// The same for the k-th slot of a level's work list (blockIdx.y = k < st->n_built).
__global__ void __launch_bounds__(256)
    hist_zero_built_kernel(const SegWork* __restrict__ st, const int32_t* __restrict__ build_slot, int32_t F,
                           uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q, int64_t* __restrict__ hist_h,
                           const uint32_t* cnt0, const int32_t* __restrict__ n_bins) {
  if (static_cast<int>(blockIdx.y) >= st->n_built) return;
  const int slot = build_slot[blockIdx.y];
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;
  const int64_t e = 4 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (e >= per_slot || !quad_used(n_bins, e)) return;
  const int64_t o = slot * per_slot + e;
  *reinterpret_cast<uint4*>(hist_cnt + o) =
      (cnt0 && slot == 0) ? *reinterpret_cast<const uint4*>(cnt0 + e) : make_uint4(0, 0, 0, 0);
  const longlong2 z = make_longlong2(0, 0);
  reinterpret_cast<longlong2*>(hist_q + o)[0] = z;
  reinterpret_cast<longlong2*>(hist_q + o)[1] = z;
  if (hist_h) {
    reinterpret_cast<longlong2*>(hist_h + o)[0] = z;
    reinterpret_cast<longlong2*>(hist_h + o)[1] = z;
  }
}

__device__ __forceinline__ longlong2 sub2(longlong2 a, longlong2 b) {
  return make_longlong2(static_cast<long long>(static_cast<unsigned long long>(a.x) - static_cast<unsigned long long>(b.x)),
                        static_cast<long long>(static_cast<unsigned long long>(a.y) - static_cast<unsigned long long>(b.y)));
}

__global__ void __launch_bounds__(256)
    hist_subtract_kernel(const uint32_t* __restrict__ prev_cnt, const int64_t* __restrict__ prev_q,
                         const int64_t* __restrict__ prev_h, const int32_t* __restrict__ pair_parent,
                         const uint8_t* __restrict__ build_flag, const gbdt_level* __restrict__ level,
                         int32_t max_slots, int32_t F, uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q,
                         int64_t* __restrict__ hist_h, int32_t* __restrict__ err, const int32_t* __restrict__ n_bins) {
  const int n_slots = min(level->n_slots, max_slots);
  const int p = blockIdx.x;
  if (2 * p + 1 >= n_slots) return;
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;
  const int64_t e = 4 * (static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x);
  if (e >= per_slot || !quad_used(n_bins, e)) return;
  const int built = build_flag[2 * p] ? 2 * p : 2 * p + 1;
  const int other = built ^ 1;
  const int parent = pair_parent[p];
  const int64_t op = parent * per_slot + e, ob = built * per_slot + e, oo = other * per_slot + e;
  const uint4 pc = *reinterpret_cast<const uint4*>(prev_cnt + op);
  const uint4 bc = *reinterpret_cast<const uint4*>(hist_cnt + ob);
  const longlong2 pq0 = reinterpret_cast<const longlong2*>(prev_q + op)[0];
  const longlong2 pq1 = reinterpret_cast<const longlong2*>(prev_q + op)[1];
  const longlong2 bq0 = reinterpret_cast<const longlong2*>(hist_q + ob)[0];
  const longlong2 bq1 = reinterpret_cast<const longlong2*>(hist_q + ob)[1];
  // bins of a quad at or above n_bins hold anything: only the used ones are checked
  const int nb = n_bins ? n_bins[e >> 8] : kBins;
  const int b0 = static_cast<int>(e & (kBins - 1));
  const bool bad = (bc.x > pc.x && b0 < nb) || (bc.y > pc.y && b0 + 1 < nb) || (bc.z > pc.z && b0 + 2 < nb) ||
                   (bc.w > pc.w && b0 + 3 < nb);
  *reinterpret_cast<uint4*>(hist_cnt + oo) = make_uint4(pc.x - bc.x, pc.y - bc.y, pc.z - bc.z, pc.w - bc.w);
  reinterpret_cast<longlong2*>(hist_q + oo)[0] = sub2(pq0, bq0);
  reinterpret_cast<longlong2*>(hist_q + oo)[1] = sub2(pq1, bq1);
  if (hist_h) {
    const longlong2 ph0 = reinterpret_cast<const longlong2*>(prev_h + op)[0];
    const longlong2 ph1 = reinterpret_cast<const longlong2*>(prev_h + op)[1];
    const longlong2 bh0 = reinterpret_cast<const longlong2*>(hist_h + ob)[0];
    const longlong2 bh1 = reinterpret_cast<const longlong2*>(hist_h + ob)[1];
    reinterpret_cast<longlong2*>(hist_h + oo)[0] = sub2(ph0, bh0);
    reinterpret_cast<longlong2*>(hist_h + oo)[1] = sub2(ph1, bh1);
  }
  if (bad) raise_error(err, kErrHistTotals);
}

template <typename K>
cudaError_t set_smem_attr(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

}  // namespace

HistPlan plan_histograms(int64_t N, int32_t F, int32_t max_slots, int32_t max_build) {
  HistPlan p{};
  const int nb = max_build < 1 ? 1 : max_build;
  const int max_entries_groups = kMaxGroupEntries / kBins;  // slots x features per CTA
  p.group_slots = nb < max_entries_groups ? nb : max_entries_groups;
  int gf = max_entries_groups / p.group_slots;
  if (gf > F) gf = F;
  p.n_fgroups = ceil_div(F, gf);
  p.group_feats = ceil_div(F, p.n_fgroups);  // balance features over groups
  p.n_sgroups = ceil_div(nb, p.group_slots);
  const int types = p.n_sgroups * p.n_fgroups;
  const int target = sm_count() * 2;
  int chunks = ceil_div(target, types);
  const int64_t min_rows = 16 * kHistThreads;  // at least one row per thread per chunk
  int64_t rpc = (N + chunks - 1) / chunks;
  if (rpc < min_rows) rpc = min_rows;
  rpc = (rpc + 15) / 16 * 16;
  p.rows_per_chunk = rpc;
  p.n_chunks = ceil_div(N, rpc);
  if (p.n_chunks < 1) p.n_chunks = 1;
  const int entries = p.group_slots * p.group_feats * kBins;
  p.smem = static_cast<size_t>(entries) * 12 + static_cast<size_t>((max_slots + 7) & ~7) * 2 +
           static_cast<size_t>(p.group_slots) * 4 + 16;
  return p;
}

void launch_hist_zero(const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag, int32_t F,
                      uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, cudaStream_t s, const uint32_t* cnt0,
                      const int32_t* n_bins) {
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;  // 4 bins per thread, 256 threads per CTA
  dim3 grid(static_cast<unsigned>((per_slot / 4 + 255) / 256), static_cast<unsigned>(max_slots));
  hist_zero_kernel<<<grid, 256, 0, s>>>(level, max_slots, build_flag, F, hist_cnt, hist_q, hist_h, cnt0, n_bins);
  count_launches();
}

void launch_hist_zero_built(const SegWork* st, const int32_t* build_slot, int32_t max_built, int32_t F,
                            uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, cudaStream_t s,
                            const uint32_t* cnt0, const int32_t* n_bins) {
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;  // 4 bins per thread, 256 threads per CTA
  dim3 grid(static_cast<unsigned>((per_slot / 4 + 255) / 256), static_cast<unsigned>(max_built < 1 ? 1 : max_built));
  hist_zero_built_kernel<<<grid, 256, 0, s>>>(st, build_slot, F, hist_cnt, hist_q, hist_h, cnt0, n_bins);
  count_launches();
}

int launch_hist_build(const HistPlan& plan, const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g,
                      int32_t g_dtype, const int32_t* fixed_exp, const uint16_t* node_of_row,
                      const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag, uint32_t* hist_cnt,
                      int64_t* hist_q, int32_t* err, cudaStream_t s) {
  if (plan.smem > kHistSmemCap) {
    set_error("histogram plan needs %zu bytes of shared memory", plan.smem);
    return GBDT_ERR_INTERNAL;
  }
  if (g_dtype == GBDT_DTYPE_F32) {
    GBDT_CUDA(set_smem_attr(hist_build_kernel<float>, plan.smem));
    hist_build_kernel<float><<<plan.blocks(), kHistThreads, plan.smem, s>>>(
        bins, ldb, N, F, static_cast<const float*>(g), fixed_exp, node_of_row, level, max_slots, build_flag,
        plan.group_slots, plan.group_feats, plan.n_fgroups, plan.n_chunks, plan.rows_per_chunk, hist_cnt, hist_q,
        err);
    count_launches();
  } else {
    GBDT_CUDA(set_smem_attr(hist_build_kernel<double>, plan.smem));
    hist_build_kernel<double><<<plan.blocks(), kHistThreads, plan.smem, s>>>(
        bins, ldb, N, F, static_cast<const double*>(g), fixed_exp, node_of_row, level, max_slots, build_flag,
        plan.group_slots, plan.group_feats, plan.n_fgroups, plan.n_chunks, plan.rows_per_chunk, hist_cnt, hist_q,
        err);
    count_launches();
  }
  return GBDT_OK;
}

void launch_hist_subtract(const uint32_t* prev_cnt, const int64_t* prev_q, const int64_t* prev_h,
                          const int32_t* pair_parent, const uint8_t* build_flag, const gbdt_level* level,
                          int32_t max_slots, int32_t F, uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h,
                          int32_t* err, cudaStream_t s, const int32_t* n_bins) {
  const int pairs = max_slots / 2;
  if (pairs < 1) return;
  const int64_t per_slot = static_cast<int64_t>(F) * kBins;  // 4 bins per thread, 256 threads per CTA
  dim3 grid(static_cast<unsigned>(pairs), static_cast<unsigned>((per_slot / 4 + 255) / 256));
  hist_subtract_kernel<<<grid, 256, 0, s>>>(prev_cnt, prev_q, prev_h, pair_parent, build_flag, level, max_slots, F,
                                             hist_cnt, hist_q, hist_h, err, n_bins);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

namespace {
// Workspace of gbdt_build_histograms: the error word, then what the grouping path needs (per-slot
// counts, cursors and segments, the grouped row-block and gradient buffers, the segmented
// histograms' scratch).  A workspace with the error word alone selects the node-id scan.
struct HistWs {
  int32_t* err;
  uint32_t* count;
  uint32_t* cursor;
  gbdt_segment* seg;
  uint8_t* rb;
  void* g;
  void* seg_scratch;
};
HistWs carve_hist(void* ws, size_t bytes, int64_t N, int32_t F, int32_t max_slots, size_t* need) {
  Carve c(ws, bytes);
  HistWs w{};
  w.err = c.take<int32_t>(1);
  const size_t cap = group_rows_capacity(N, max_slots);
  w.count = c.take<uint32_t>(max_slots);
  w.cursor = c.take<uint32_t>(max_slots);
  w.seg = c.take<gbdt_segment>(max_slots);
  w.rb = c.take<uint8_t>(static_cast<size_t>(rb_blocks(static_cast<int64_t>(cap))) * rb_pitch(F));
  w.g = c.take<double>(cap);
  w.seg_scratch = c.take<unsigned char>(seg_hist_scratch_bytes(max_slots));
  *need = c.used;
  return w;
}
}  // namespace

extern "C" size_t gbdt_histograms_workspace_size(int64_t N, int32_t F, int32_t max_slots) {
  if (N < 1 || F < 1 || max_slots < 1) return kWsAlign;
  size_t need = 0;
  carve_hist(nullptr, 0, N, F, max_slots, &need);
  return need;
}

extern "C" int gbdt_build_histograms(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g,
                                     int32_t g_dtype, const int32_t* fixed_exp, const uint16_t* node_of_row,
                                     const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag,
                                     int32_t max_build, uint32_t* hist_cnt, int64_t* hist_q, void* ws,
                                     size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && g && fixed_exp && node_of_row && level && build_flag && hist_cnt && hist_q,
                 "gbdt_build_histograms: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31), "gbdt_build_histograms: N out of range");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096, "gbdt_build_histograms: F out of range");
  GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins, 16), "gbdt_build_histograms: bins need ldb >= N, "
                 "ldb %% 16 == 0 and a 16-byte aligned base");
  GBDT_CHECK_ARG(aligned(node_of_row, 16) && aligned(g, 16), "gbdt_build_histograms: node_of_row and g must be "
                 "16-byte aligned");
  GBDT_CHECK_ARG(g_dtype == GBDT_DTYPE_F32 || g_dtype == GBDT_DTYPE_F64, "gbdt_build_histograms: bad g dtype");
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kMaxSlots, "gbdt_build_histograms: max_slots out of range");
  GBDT_CHECK_ARG(max_build >= 1 && max_build <= max_slots, "gbdt_build_histograms: max_build out of range");
  if (!ws || ws_bytes < kWsAlign || !aligned(ws, kWsAlign)) {
    set_error("gbdt_build_histograms: workspace too small or misaligned");
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t need = 0;
  const HistWs w = carve_hist(ws, ws_bytes, N, F, max_slots, &need);
  int32_t* err = w.err;  // the call's error word (gbdt_workspace_status)
  GBDT_CUDA(cudaMemsetAsync(err, 0, sizeof(int32_t), s));
  if (max_build >= 2 && ws_bytes >= need) {
    // rows grouped by slot first, then the node-contiguous histogram kernel on the grouped copy
    const int g_size = g_dtype == GBDT_DTYPE_F64 ? 8 : 4;
    launch_group_rows(bins, ldb, N, F, g, g_size, node_of_row, level, max_slots, build_flag, w.count, w.cursor,
                      w.seg, w.rb, w.g, err, s);
    const int64_t cap = static_cast<int64_t>(group_rows_capacity(N, max_slots));
    const SegHistPlan plan = plan_seg_histograms(cap, F, max_slots, max_build, false, false);
    int rc = launch_seg_histograms(plan, w.rb, rb_pitch(F), cap, F, w.g, g_dtype, fixed_exp, level, max_slots,
                                   build_flag, w.seg, nullptr, w.seg_scratch, hist_cnt, hist_q, nullptr, s, true);
    if (rc != GBDT_OK) return rc;
    GBDT_LAUNCH_CHECK();
    return GBDT_OK;
  }
  const HistPlan plan = plan_histograms(N, F, max_slots, max_build);
  launch_hist_zero(level, max_slots, build_flag, F, hist_cnt, hist_q, nullptr, s);
  int rc = launch_hist_build(plan, bins, ldb, N, F, g, g_dtype, fixed_exp, node_of_row, level, max_slots,
                             build_flag, hist_cnt, hist_q, err, s);
  if (rc != GBDT_OK) return rc;
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" size_t gbdt_subtract_histograms_workspace_size(void) { return kWsAlign; }

extern "C" int gbdt_subtract_histograms_h(const uint32_t* prev_cnt, const int64_t* prev_q, const int64_t* prev_h,
                                          const int32_t* pair_parent, const uint8_t* build_flag,
                                          const gbdt_level* level, int32_t max_slots, int32_t F, uint32_t* hist_cnt,
                                          int64_t* hist_q, int64_t* hist_h, void* ws, size_t ws_bytes,
                                          void* stream) {
  clear_error();
  GBDT_CHECK_ARG(prev_cnt && prev_q && pair_parent && build_flag && level && hist_cnt && hist_q,
                 "gbdt_subtract_histograms: null pointer");
  GBDT_CHECK_ARG((prev_h == nullptr) == (hist_h == nullptr), "gbdt_subtract_histograms: prev_h and hist_h must both "
                 "be given or both be NULL");
  GBDT_CHECK_ARG(max_slots >= 2 && max_slots <= kMaxSlots && F >= 1 && F <= 4096,
                 "gbdt_subtract_histograms: sizes out of range");
  if (ws && (ws_bytes < gbdt_subtract_histograms_workspace_size() || !aligned(ws, kWsAlign))) {
    set_error("gbdt_subtract_histograms: workspace too small or misaligned");
    return GBDT_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* err = static_cast<int32_t*>(ws);  // optional: the call's error word (gbdt_workspace_status)
  if (err) GBDT_CUDA(cudaMemsetAsync(err, 0, sizeof(int32_t), s));
  launch_hist_subtract(prev_cnt, prev_q, prev_h, pair_parent, build_flag, level, max_slots, F, hist_cnt, hist_q,
                       hist_h, err, s);
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" int gbdt_subtract_histograms(const uint32_t* prev_cnt, const int64_t* prev_q, const int32_t* pair_parent,
                                        const uint8_t* build_flag, const gbdt_level* level, int32_t max_slots,
                                        int32_t F, uint32_t* hist_cnt, int64_t* hist_q, void* ws, size_t ws_bytes,
                                        void* stream) {
  return gbdt_subtract_histograms_h(prev_cnt, prev_q, nullptr, pair_parent, build_flag, level, max_slots, F, hist_cnt,
                                    hist_q, nullptr, ws, ws_bytes, stream);
}
