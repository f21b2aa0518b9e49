// Exact quantile binning of fp32 features into uint8 bins.
//
// The pages name the "Quantized" state ("Module Design: Training Core" s.5)
// without its rule; the rule used here is stated in gbdt.h.  It is made of
// order statistics and comparisons only, so it is reproducible bit for bit.
//
// First one pass over every value: its finiteness and, per column, whether it has at most max_bins
// distinct values (a hash set of the values in each CTA's shared memory, merged per column).  A column
// with at most max_bins distinct values takes its edges from that set and is never sorted.  The other
// columns, per batch: map each value to an order-preserving uint32 key (-0.0 read as +0.0), sort the
// column with a stable 4-pass LSD radix sort (8-bit digits; tile counts, a scan over tiles per (column,
// digit) and over digits per column, and a stable scatter that ranks equal digits inside a warp with 8
// ballots), and read the order statistics off the sorted keys.  Then every value is binned by binary
// search over its column's edges.
#include <algorithm>
#include <vector>

#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kQThreads = 256;
constexpr int kQTile = 4096;  // keys per radix tile
constexpr int kQRounds = kQTile / kQThreads;
constexpr size_t kQBatchBudget = size_t(2) << 30;  // bytes of key buffers per batch

__device__ __forceinline__ uint32_t f2key(float x) {
  const uint32_t b = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void finite_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int32_t F, int32_t* flag) {
  bool bad = false;
  for (int j = blockIdx.y; j < F; j += gridDim.y)
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x)
      bad |= !isfinite(X[j * ldx + i]);
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
}

// ---- distinct values (at most B per column are tracked)
constexpr int kSetSlots = 512;        // open-addressing slots of a CTA's set (> 2 * 256: probes stay short)
constexpr int kDistinctCtas = 64;     // CTAs per column of the distinct pass
constexpr int kListCap = kDistinctCtas * 256;  // per column: every CTA's set (each at most 256 values)
constexpr uint32_t kEmptyKey = 0xffffffffu;     // no finite value maps to it

__device__ __forceinline__ uint32_t set_hash(uint32_t k) { return (k * 2654435761u) >> (32 - 9); }

// Grid (kDistinctCtas, columns of the batch).  Each CTA: its rows of column j = j0 + y, their finiteness
// (flag), and the distinct keys among them while there are at most B; more than B in one CTA marks the
// column for sorting (more[j] = 1).  Otherwise the CTA's keys are appended to the column's list
// (list[y][0 .. cnt[j]): the batch's lists, kListCap entries each, room for every CTA's set).
__device__ __forceinline__ bool nonfinite_bits(float v) {  // exponent all ones: Inf or NaN
  return (__float_as_uint(v) & 0x7f800000u) == 0x7f800000u;
}

// Add key k to the CTA's set (open addressing over kSetSlots slots).  More than B keys, or no free slot
// within kMaxProbes (a set of at most B <= 256 keys in 512 slots practically never needs that many),
// set *over: the column is then sorted, which is always correct.
constexpr int kMaxProbes = 32;
__device__ __forceinline__ void set_insert(uint32_t* s_set, int* s_n, int* s_over, uint32_t k, int B) {
  if (*reinterpret_cast<volatile int*>(s_over)) return;
  uint32_t h = set_hash(k);
  for (int probe = 0; probe < kMaxProbes; ++probe, h = (h + 1) & (kSetSlots - 1)) {
    const uint32_t cur = s_set[h];
    if (cur == k) return;
    if (cur == kEmptyKey) {
      const uint32_t old = atomicCAS(&s_set[h], kEmptyKey, k);
      if (old == kEmptyKey) {
        if (atomicAdd(s_n, 1) >= B) *s_over = 1;
        return;
      }
      if (old == k) return;
    }
  }
  *s_over = 1;
}

// kVec: X's columns 16-byte aligned (four values per load).
template <bool kVec>
__global__ void __launch_bounds__(256)
    distinct_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int j0, int B, int32_t* flag,
                    uint32_t* __restrict__ list, uint32_t* __restrict__ cnt, int32_t* __restrict__ more) {
  __shared__ uint32_t s_set[kSetSlots];
  __shared__ int s_n, s_over;
  __shared__ uint32_t s_pos;
  const int j = j0 + blockIdx.y;
  for (int i = threadIdx.x; i < kSetSlots; i += blockDim.x) s_set[i] = kEmptyKey;
  if (threadIdx.x == 0) s_n = 0, s_over = 0;
  __syncthreads();
  const float* x = X + static_cast<int64_t>(j) * ldx;
  // this CTA's rows [r0, r1), a multiple of four of them per CTA
  const int64_t per = (N + 4 * gridDim.x - 1) / (4 * gridDim.x) * 4;
  const int64_t r0 = per * blockIdx.x, r1 = min(N, r0 + per);
  volatile int* over = &s_over;
  bool bad = false;
  int64_t i = r0;
  if (kVec) {
    const int64_t n4 = r1 > r0 ? (r1 - r0) / 4 : 0;
    const float4* x4 = reinterpret_cast<const float4*>(x + r0);
    int64_t q = threadIdx.x;
    for (; q < n4 && !*over; q += blockDim.x) {  // values still counted
      const float4 v = x4[q];
      bad |= nonfinite_bits(v.x) | nonfinite_bits(v.y) | nonfinite_bits(v.z) | nonfinite_bits(v.w);
      set_insert(s_set, &s_n, &s_over, f2key(v.x), B);
      set_insert(s_set, &s_n, &s_over, f2key(v.y), B);
      set_insert(s_set, &s_n, &s_over, f2key(v.z), B);
      set_insert(s_set, &s_n, &s_over, f2key(v.w), B);
    }
    for (; q < n4; q += blockDim.x) {  // more than B values: only the finiteness is left to check
      const float4 v = x4[q];
      bad |= nonfinite_bits(v.x) | nonfinite_bits(v.y) | nonfinite_bits(v.z) | nonfinite_bits(v.w);
    }
    i = r0 + 4 * n4;
  }
  for (i += threadIdx.x; i < r1; i += blockDim.x) {
    const float v = x[i];
    bad |= nonfinite_bits(v);
    if (!*over) set_insert(s_set, &s_n, &s_over, f2key(v), B);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
  if (s_over) {
    if (threadIdx.x == 0) more[j] = 1;
    return;
  }
  if (threadIdx.x == 0) {
    const uint32_t pos = atomicAdd(&cnt[j], static_cast<uint32_t>(s_n));
    s_pos = pos;
    if (pos + s_n > static_cast<uint32_t>(kListCap)) more[j] = 1;
    s_n = 0;  // reused as the write cursor
  }
  __syncthreads();
  const uint32_t pos = s_pos;
  uint32_t* out = list + static_cast<int64_t>(blockIdx.y) * kListCap;
  for (int k = threadIdx.x; k < kSetSlots; k += blockDim.x) {
    const uint32_t key = s_set[k];
    if (key == kEmptyKey) continue;
    const uint32_t at = pos + static_cast<uint32_t>(atomicAdd(&s_n, 1));
    if (at < static_cast<uint32_t>(kListCap)) out[at] = key;
  }
}

// One CTA per column j = j0 + x of the batch: a column not marked for sorting has its list's distinct keys
// counted; U <= B of them: its edges are the U-1 smallest (the largest is no edge), n_bins = U;
// more than B (the CTAs' sets together exceed B): marked for sorting.
__global__ void __launch_bounds__(256)
    distinct_edges_kernel(const uint32_t* __restrict__ list, const uint32_t* __restrict__ cnt, int32_t* __restrict__ more,
                          int j0, int B, float* __restrict__ edges, int32_t* __restrict__ n_bins) {
  __shared__ uint32_t s_set[kSetSlots];
  __shared__ uint32_t s_vals[256];
  __shared__ int s_n, s_over;
  const int j = j0 + blockIdx.x;
  if (more[j]) return;  // CTA-uniform
  for (int i = threadIdx.x; i < kSetSlots; i += blockDim.x) s_set[i] = kEmptyKey;
  if (threadIdx.x == 0) s_n = 0, s_over = 0;
  __syncthreads();
  const uint32_t n = min(cnt[j], static_cast<uint32_t>(kListCap));
  const uint32_t* in = list + static_cast<int64_t>(blockIdx.x) * kListCap;
  for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
    if (*reinterpret_cast<volatile int*>(&s_over)) break;
    const uint32_t k = in[i];
    uint32_t h = set_hash(k);
    bool placed = false;  // found or inserted; a key that finds no slot within kMaxProbes sends the column to the sort
    for (int probe = 0; probe < kMaxProbes && !placed; ++probe, h = (h + 1) & (kSetSlots - 1)) {
      const uint32_t cur = s_set[h];
      if (cur == k) {
        placed = true;
      } else if (cur == kEmptyKey) {
        const uint32_t old = atomicCAS(&s_set[h], kEmptyKey, k);
        if (old == kEmptyKey) {
          const int at = atomicAdd(&s_n, 1);
          if (at < B) s_vals[at] = k;
          else s_over = 1;
          placed = true;
        } else if (old == k) {
          placed = true;
        }
      }
    }
    if (!placed) s_over = 1;
  }
  __syncthreads();
  if (s_over) {
    if (threadIdx.x == 0) more[j] = 1;
    return;
  }
  const int U = s_n;
  float* e = edges + static_cast<int64_t>(j) * (B - 1);
  for (int i = threadIdx.x; i < U; i += blockDim.x) {  // rank among the distinct values
    const uint32_t x = s_vals[i];
    int r = 0;
    for (int m = 0; m < U; ++m) r += s_vals[m] < x ? 1 : 0;
    if (r + 1 < U) e[r] = key2f(x);
  }
  for (int k = U - 1 + threadIdx.x; k < B - 1; k += blockDim.x) e[k] = INFINITY;
  if (threadIdx.x == 0) n_bins[j] = U;
}

// The kernels of the sort take the columns j0 .. j0 + nb - 1 of a batch and skip those that more[]
// (the batch's part: more[j] for column j0 + j) does not mark.
__global__ void keys_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int j0, uint32_t* __restrict__ keys,
                            const int32_t* __restrict__ more) {
  const int j = blockIdx.y;
  if (!more[j]) return;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x)
    keys[j * N + i] = f2key(X[(j0 + j) * ldx + i]);
}

// counts[j][digit][tile]
__global__ void __launch_bounds__(kQThreads)
    radix_count_kernel(const uint32_t* __restrict__ keys, int64_t N, int tiles, int shift,
                       uint32_t* __restrict__ counts, const int32_t* __restrict__ more) {
  __shared__ uint32_t h[256];
  const int j = blockIdx.y, t = blockIdx.x;
  if (!more[j]) return;
  h[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t* k = keys + j * N;
  const int64_t b0 = static_cast<int64_t>(t) * kQTile;
  for (int r = 0; r < kQRounds; ++r) {
    const int64_t i = b0 + r * kQThreads + threadIdx.x;
    if (i < N) atomicAdd(&h[(k[i] >> shift) & 0xff], 1u);
  }
  __syncthreads();
  counts[(static_cast<int64_t>(j) * 256 + threadIdx.x) * tiles + t] = h[threadIdx.x];
}

// In-place exclusive scan over the tiles of one (column, digit) row of the
// counts; the row's total goes to dtot[j][digit].
__global__ void __launch_bounds__(256)
    radix_tile_scan_kernel(uint32_t* __restrict__ counts, int tiles, uint32_t* __restrict__ dtot,
                           const int32_t* __restrict__ more) {
  __shared__ uint32_t s_warp[33];
  __shared__ uint32_t s_carry;
  const int d = blockIdx.x, j = blockIdx.y;
  if (!more[j]) return;
  uint32_t* c = counts + (static_cast<int64_t>(j) * 256 + d) * tiles;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int c0 = 0; c0 < tiles; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const uint32_t v = i < tiles ? c[i] : 0u;
    uint32_t incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
      const uint32_t w = lane < nw ? s_warp[lane] : 0u;
      uint32_t wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      if (lane < nw) s_warp[lane] = wi - w;
      if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    if (i < tiles) c[i] = s_carry + s_warp[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_warp[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) dtot[j * 256 + d] = s_carry;
}

// Exclusive scan of one column's 256 digit totals (in place): the digit's first position.
__global__ void __launch_bounds__(256) radix_digit_scan_kernel(uint32_t* __restrict__ dtot,
                                                               const int32_t* __restrict__ more) {
  __shared__ uint32_t s[256];
  if (!more[blockIdx.x]) return;
  uint32_t* t = dtot + blockIdx.x * 256;
  const uint32_t v = t[threadIdx.x];
  s[threadIdx.x] = v;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {
    const uint32_t a = threadIdx.x >= o ? s[threadIdx.x - o] : 0u;
    __syncthreads();
    s[threadIdx.x] += a;
    __syncthreads();
  }
  t[threadIdx.x] = s[threadIdx.x] - v;
}

// Stable scatter of one tile (kQTile keys): the keys are ranked into shared memory in (digit,
// original order) - taken 256 at a time, equal digits inside a warp ranked with ballots, across warps
// and rounds with counters - and each digit's run of the tile is then written out with consecutive
// addresses (a warp's stores cover one or two runs instead of up to 32).
__global__ void __launch_bounds__(kQThreads)
    radix_scatter_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int64_t N, int tiles, int shift,
                         const uint32_t* __restrict__ offsets, const uint32_t* __restrict__ dbase,
                         const int32_t* __restrict__ more) {
  constexpr int kWarps = kQThreads / 32;
  static_assert(kQThreads == 256, "one thread per digit");
  __shared__ uint32_t s_keys[kQTile];     // the tile's keys, ranked
  __shared__ uint32_t s_start[256];       // each digit's first position in s_keys
  __shared__ uint32_t s_run[256];         // each digit's next position in s_keys
  __shared__ uint32_t s_gbase[256];       // the global position of the tile's first key of each digit
  __shared__ uint32_t s_wc[kWarps][256];  // per-warp count, then per-warp start, of each digit
  __shared__ uint32_t s_warp[kWarps];
  const int j = blockIdx.y, t = blockIdx.x;
  if (!more[j]) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t* k = in + j * N;
  uint32_t* o = out + j * N;
  const int64_t b0 = static_cast<int64_t>(t) * kQTile;
  const int n = static_cast<int>(min(static_cast<int64_t>(kQTile), N - b0));
  uint32_t key[kQRounds];
#pragma unroll
  for (int r = 0; r < kQRounds; ++r) {
    const int li = r * kQThreads + static_cast<int>(threadIdx.x);
    key[r] = li < n ? k[b0 + li] : 0u;
  }
  // the tile's count of each digit, then its exclusive scan over the digits (thread d: digit d)
  s_run[threadIdx.x] = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kQRounds; ++r)
    if (r * kQThreads + static_cast<int>(threadIdx.x) < n) atomicAdd(&s_run[(key[r] >> shift) & 0xff], 1u);
  __syncthreads();
  {
    const uint32_t c = s_run[threadIdx.x];
    uint32_t incl = c;
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    const uint32_t excl = before + incl - c;
    s_start[threadIdx.x] = excl;
    s_run[threadIdx.x] = excl;
    s_gbase[threadIdx.x] =
        dbase[j * 256 + threadIdx.x] + offsets[(static_cast<int64_t>(j) * 256 + threadIdx.x) * tiles + t];
  }
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < kQRounds; ++r) {
    for (int w = 0; w < kWarps; ++w) s_wc[w][threadIdx.x] = 0;
    __syncthreads();
    const bool valid = r * kQThreads + static_cast<int>(threadIdx.x) < n;
    const uint32_t dg = (key[r] >> shift) & 0xff;
    uint32_t peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t bal = __ballot_sync(0xffffffffu, (dg >> b) & 1u);
      peers &= ((dg >> b) & 1u) ? bal : ~bal;
    }
    const uint32_t rank = __popc(peers & lt);
    if (valid && rank == 0) s_wc[warp][dg] = __popc(peers);
    __syncthreads();
    {  // thread d: exclusive prefix over warps of digit d, advance the running position
      const int d = threadIdx.x;
      uint32_t run = s_run[d];
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = s_wc[w][d];
        s_wc[w][d] = run;
        run += c;
      }
      s_run[d] = run;
    }
    __syncthreads();
    if (valid) s_keys[s_wc[warp][dg] + rank] = key[r];
    __syncthreads();  // every thread has read its start before the next round clears them
  }
  for (int i = threadIdx.x; i < n; i += kQThreads) {
    const uint32_t x = s_keys[i];
    const uint32_t dg = (x >> shift) & 0xff;
    const int64_t p = static_cast<int64_t>(s_gbase[dg]) + (i - static_cast<int64_t>(s_start[dg]));
    if (p >= 0 && p < N) o[p] = x;  // always: the tile's counts and the scans agree
  }
}

// One CTA per sorted column (more than B distinct values): the order statistics
// v[ceil(kN/B) - 1], k = 1..B-1, strictly increasing, without one equal to the largest value.
__global__ void __launch_bounds__(256)
    order_edges_kernel(const uint32_t* __restrict__ sorted, int64_t N, int j0, int B, const int32_t* __restrict__ more,
                       float* __restrict__ edges, int32_t* __restrict__ n_bins) {
  const int j = blockIdx.x;
  if (!more[j]) return;
  const uint32_t* v = sorted + j * N;
  __shared__ float s_e[256];
  __shared__ int s_ne;
  float* e = edges + static_cast<int64_t>(j0 + j) * (B - 1);
  for (int k = 1 + threadIdx.x; k <= B - 1; k += blockDim.x) {
    const int64_t pk = (static_cast<int64_t>(k) * N + B - 1) / B - 1;
    s_e[k - 1] = key2f(v[pk]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float vmax = key2f(v[N - 1]);
    int ne = 0;
    for (int k = 0; k < B - 1; ++k) {
      const float ek = s_e[k];
      if (ne > 0 && !(ek > s_e[ne - 1])) continue;  // strictly increasing (s_e[ne-1] already compacted)
      if (ek == vmax) continue;
      s_e[ne++] = ek;
    }
    s_ne = ne;
  }
  __syncthreads();
  const int ne = s_ne;
  for (int k = threadIdx.x; k < B - 1; k += blockDim.x) e[k] = k < ne ? s_e[k] : INFINITY;
  if (threadIdx.x == 0) n_bins[j0 + j] = ne + 1;
}

// Number of the column's edges strictly below x (binary search over the ne edges in shared memory).
__device__ __forceinline__ uint32_t bin_of(const float* s_e, int ne, float x) {
  int lo = 0, hi = ne;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_e[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return static_cast<uint32_t>(lo);
}

// kVec: X's columns 16-byte aligned (X aligned, ldx % 4 == 0): four values per thread per step (one
// 16-byte load, four independent searches, one 4-byte store; bins' columns are 16-byte aligned),
// the last N % 4 values of a column by the first CTA of its row.
template <bool kVec>
__global__ void bin_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int j0, int B,
                           const float* __restrict__ edges, const int32_t* __restrict__ n_bins,
                           uint8_t* __restrict__ bins, int64_t ldb) {
  __shared__ float s_e[256];
  const int j = j0 + blockIdx.y;
  const int ne = n_bins[j] - 1;
  for (int k = threadIdx.x; k < ne; k += blockDim.x) s_e[k] = edges[static_cast<int64_t>(j) * (B - 1) + k];
  __syncthreads();
  const float* xc = X + j * ldx;
  uint8_t* bc = bins + j * ldb;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i0 = 0;
  if (kVec) {
    const int64_t n4 = N / 4;
    for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < n4; q += stride) {
      const float4 x = *reinterpret_cast<const float4*>(xc + 4 * q);
      const uint32_t b = bin_of(s_e, ne, x.x) | bin_of(s_e, ne, x.y) << 8 | bin_of(s_e, ne, x.z) << 16 |
                         bin_of(s_e, ne, x.w) << 24;
      *reinterpret_cast<uint32_t*>(bc + 4 * q) = b;
    }
    if (blockIdx.x != 0) return;
    i0 = 4 * n4;
  }
  for (int64_t i = i0 + (kVec ? 0 : blockIdx.x * static_cast<int64_t>(blockDim.x)) + threadIdx.x; i < N;
       i += kVec ? blockDim.x : stride)
    bc[i] = static_cast<uint8_t>(bin_of(s_e, ne, xc[i]));
}

int batch_columns(int64_t N, int32_t F) {
  const size_t per_col = static_cast<size_t>(N) * 8 + static_cast<size_t>(256) * ceil_div(N, kQTile) * 4 +
                         sizeof(uint32_t) * kListCap;
  int fb = static_cast<int>(kQBatchBudget / (per_col ? per_col : 1));
  return std::max(1, std::min<int>(fb, F));
}

struct QuantWs {
  uint32_t* a;
  uint32_t* b;
  uint32_t* counts;
  uint32_t* dtot;
  uint32_t* list;   // [batch columns][kListCap] distinct keys per column of a batch
  uint32_t* cnt;    // [F] entries of each list
  int32_t* more;    // [F] 1: more than max_bins distinct values (the column is sorted)
  int32_t* flag;
};
QuantWs carve_quant(void* ws, size_t bytes, int64_t N, int32_t F, size_t* need) {
  Carve c(ws, bytes);
  QuantWs w{};
  const int fb = batch_columns(N, F);
  w.a = c.take<uint32_t>(static_cast<size_t>(fb) * N);
  w.b = c.take<uint32_t>(static_cast<size_t>(fb) * N);
  w.counts = c.take<uint32_t>(static_cast<size_t>(fb) * 256 * ceil_div(N, kQTile));
  w.dtot = c.take<uint32_t>(static_cast<size_t>(fb) * 256);
  w.list = c.take<uint32_t>(static_cast<size_t>(fb) * kListCap);
  w.cnt = c.take<uint32_t>(F);
  w.more = c.take<int32_t>(F);
  w.flag = c.take<int32_t>(1);
  *need = c.used;
  return w;
}

// Finiteness and distinct values of columns j0 .. j0 + nb - 1; the edges of those with at most B distinct
// values (the others are marked in w.more for the sort).  w.cnt and w.more of the columns must be zero.
void distinct_batch(const float* X, int64_t ldx, int64_t N, int j0, int nb, int B, float* edges, int32_t* n_bins,
                    const QuantWs& w, cudaStream_t s) {
  if (aligned(X, 16) && ldx % 4 == 0)
    distinct_kernel<true><<<dim3(kDistinctCtas, nb), 256, 0, s>>>(X, ldx, N, j0, B, w.flag, w.list, w.cnt, w.more);
  else
    distinct_kernel<false><<<dim3(kDistinctCtas, nb), 256, 0, s>>>(X, ldx, N, j0, B, w.flag, w.list, w.cnt, w.more);
  count_launches();
  distinct_edges_kernel<<<nb, 256, 0, s>>>(w.list, w.cnt, w.more, j0, B, edges, n_bins);
  count_launches();
}

// Sort and order statistics of the marked columns among j0 .. j0 + nb - 1, then the bins of all of them.
int quantize_batch(const float* X, int64_t ldx, int64_t N, int j0, int nb, int max_bins, uint8_t* bins, int64_t ldb,
                   float* edges, int32_t* n_bins, const QuantWs& w, cudaStream_t s) {
  const int gx = std::min<int64_t>(ceil_div(N, 256), sm_count() * 4);
  const int tiles = ceil_div(N, kQTile);
  const int32_t* more = w.more + j0;
  keys_kernel<<<dim3(gx, nb), 256, 0, s>>>(X, ldx, N, j0, w.a, more);
  count_launches();
  uint32_t* src = w.a;
  uint32_t* dst = w.b;
  for (int pass = 0; pass < 4; ++pass) {
    radix_count_kernel<<<dim3(tiles, nb), kQThreads, 0, s>>>(src, N, tiles, 8 * pass, w.counts, more);
    count_launches();
    radix_tile_scan_kernel<<<dim3(256, nb), 256, 0, s>>>(w.counts, tiles, w.dtot, more);
    count_launches();
    radix_digit_scan_kernel<<<nb, 256, 0, s>>>(w.dtot, more);
    count_launches();
    radix_scatter_kernel<<<dim3(tiles, nb), kQThreads, 0, s>>>(src, dst, N, tiles, 8 * pass, w.counts, w.dtot, more);
    count_launches();
    std::swap(src, dst);
  }
  order_edges_kernel<<<nb, 256, 0, s>>>(src, N, j0, max_bins, more, edges, n_bins);
  count_launches();
  if (aligned(X, 16) && ldx % 4 == 0)
    bin_kernel<true><<<dim3(gx, nb), 256, 0, s>>>(X, ldx, N, j0, max_bins, edges, n_bins, bins, ldb);
  else
    bin_kernel<false><<<dim3(gx, nb), 256, 0, s>>>(X, ldx, N, j0, max_bins, edges, n_bins, bins, ldb);
  count_launches();
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

// Columns per batch when the features arrive from the host: small batches, so that the first batch's
// sort starts after a small part of the copy and every later copy runs under an earlier batch's sort.
constexpr int kHostBatchColumns = 8;

}  // namespace

}  // namespace gbdt

using namespace gbdt;

extern "C" size_t gbdt_quantize_workspace_size(int64_t N, int32_t F) {
  if (N < 1 || F < 1) return 0;
  size_t need = 0;
  carve_quant(nullptr, 0, N, F, &need);
  return need;
}

extern "C" int gbdt_quantize(const float* X, int64_t ldx, int64_t N, int32_t F, int32_t max_bins, uint8_t* bins,
                             int64_t ldb, float* edges, int32_t* n_bins, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(X && bins && edges && n_bins, "gbdt_quantize: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 65535, "gbdt_quantize: sizes out of range");
  GBDT_CHECK_ARG(max_bins >= 2 && max_bins <= GBDT_MAX_BINS, "gbdt_quantize: max_bins must be in 2..256");
  GBDT_CHECK_ARG(ldx >= N && ldb >= N && ldb % 16 == 0 && aligned(bins, 16),
                 "gbdt_quantize: need ldx >= N, ldb >= N, ldb %% 16 == 0 and 16-byte aligned bins");
  size_t need = 0;
  QuantWs w = carve_quant(ws, ws_bytes, N, F, &need);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_quantize: workspace needs %zu bytes", need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GBDT_CUDA(cudaMemsetAsync(w.flag, 0, sizeof(int32_t), s));
  GBDT_CUDA(cudaMemsetAsync(w.cnt, 0, sizeof(uint32_t) * F, s));
  GBDT_CUDA(cudaMemsetAsync(w.more, 0, sizeof(int32_t) * F, s));
  const int gx = std::min<int64_t>(ceil_div(N, 256), sm_count() * 4);
  finite_kernel<<<dim3(gx, std::min(F, 64)), 256, 0, s>>>(X, ldx, N, F, w.flag);
  count_launches();
  int32_t bad = 0;
  GBDT_CUDA(cudaMemcpyAsync(&bad, w.flag, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (bad) {
    set_error("gbdt_quantize: features contain NaN or Inf");
    return GBDT_ERR_NONFINITE;
  }
  const int fb = batch_columns(N, F);
  for (int j0 = 0; j0 < F; j0 += fb) {
    const int nb = std::min(fb, F - j0);
    distinct_batch(X, ldx, N, j0, nb, max_bins, edges, n_bins, w, s);
    const int rc = quantize_batch(X, ldx, N, j0, nb, max_bins, bins, ldb, edges, n_bins, w, s);
    if (rc != GBDT_OK) return rc;
  }
  return GBDT_OK;
}

extern "C" int gbdt_quantize_host(const float* X_host, int64_t ldx, int64_t N, int32_t F, int32_t max_bins,
                                  float* X_dev, uint8_t* bins, int64_t ldb, float* edges, int32_t* n_bins, void* ws,
                                  size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(X_host && X_dev && bins && edges && n_bins, "gbdt_quantize_host: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 65535, "gbdt_quantize_host: sizes out of range");
  GBDT_CHECK_ARG(max_bins >= 2 && max_bins <= GBDT_MAX_BINS, "gbdt_quantize_host: max_bins must be in 2..256");
  GBDT_CHECK_ARG(ldx >= N && ldb >= N && ldb % 16 == 0 && aligned(bins, 16),
                 "gbdt_quantize_host: need ldx >= N, ldb >= N, ldb %% 16 == 0 and 16-byte aligned bins");
  size_t need = 0;
  QuantWs w = carve_quant(ws, ws_bytes, N, F, &need);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_quantize_host: workspace needs %zu bytes", need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int fb = std::min(batch_columns(N, F), kHostBatchColumns);
  const int n_batches = ceil_div(F, fb);
  // the copies run on a stream of their own, after the work already queued on `stream` (which may still
  // read X_dev); each batch's sort waits for its own copy only
  struct Res {
    cudaStream_t cs = nullptr;
    std::vector<cudaEvent_t> ev;
    ~Res() {  // on an early return the copies from X_host still in flight finish first
      if (cs) cudaStreamSynchronize(cs);
      for (cudaEvent_t e : ev)
        if (e) cudaEventDestroy(e);
      if (cs) cudaStreamDestroy(cs);
    }
  } r;
  r.ev.assign(n_batches + 1, nullptr);
  for (cudaEvent_t& e : r.ev) GBDT_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  GBDT_CUDA(cudaStreamCreateWithFlags(&r.cs, cudaStreamNonBlocking));
  GBDT_CUDA(cudaEventRecord(r.ev[n_batches], s));
  GBDT_CUDA(cudaStreamWaitEvent(r.cs, r.ev[n_batches], 0));
  for (int b = 0; b < n_batches; ++b) {
    const int j0 = b * fb, nb = std::min(fb, F - j0);
    const size_t count = static_cast<size_t>(nb - 1) * static_cast<size_t>(ldx) + static_cast<size_t>(N);
    GBDT_CUDA(cudaMemcpyAsync(X_dev + static_cast<int64_t>(j0) * ldx, X_host + static_cast<int64_t>(j0) * ldx,
                              count * sizeof(float), cudaMemcpyHostToDevice, r.cs));
    GBDT_CUDA(cudaEventRecord(r.ev[b], r.cs));
  }
  GBDT_CUDA(cudaMemsetAsync(w.flag, 0, sizeof(int32_t), s));
  GBDT_CUDA(cudaMemsetAsync(w.cnt, 0, sizeof(uint32_t) * F, s));
  GBDT_CUDA(cudaMemsetAsync(w.more, 0, sizeof(int32_t) * F, s));
  for (int b = 0; b < n_batches; ++b) {
    const int j0 = b * fb, nb = std::min(fb, F - j0);
    GBDT_CUDA(cudaStreamWaitEvent(s, r.ev[b], 0));
    // finiteness (read once at the end: the outputs of a call that fails it are not to be used) and
    // distinct values of the batch, then its sort
    distinct_batch(X_dev, ldx, N, j0, nb, max_bins, edges, n_bins, w, s);
    const int rc = quantize_batch(X_dev, ldx, N, j0, nb, max_bins, bins, ldb, edges, n_bins, w, s);
    if (rc != GBDT_OK) return rc;
  }
  int32_t bad = 0;
  GBDT_CUDA(cudaMemcpyAsync(&bad, w.flag, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (bad) {
    set_error("gbdt_quantize_host: features contain NaN or Inf");
    return GBDT_ERR_NONFINITE;
  }
  return GBDT_OK;
}
