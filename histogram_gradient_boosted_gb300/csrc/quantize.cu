// Exact quantile binning of fp32 features into uint8 bins.
//
// The pages name the "Quantized" state ("Module Design: Training Core" s.5)
// without its rule; the rule used here is stated in gbdt.h.  It is made of
// order statistics and comparisons only, so it is reproducible bit for bit.
//
// Per batch of columns: map each value to an order-preserving uint32 key
// (-0.0 read as +0.0), sort every column with a stable 4-pass LSD radix sort
// (8-bit digits; tile counts, a per-column scan, and a stable scatter that
// ranks equal digits inside a warp with 8 ballots), read the edges off the
// sorted keys, then bin every value by binary search over its column's edges.
#include <algorithm>

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

__global__ void keys_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int j0, uint32_t* __restrict__ keys) {
  const int j = blockIdx.y;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x)
    keys[j * N + i] = f2key(X[(j0 + j) * ldx + i]);
}

// counts[j][digit][tile]
__global__ void __launch_bounds__(kQThreads)
    radix_count_kernel(const uint32_t* __restrict__ keys, int64_t N, int tiles, int shift,
                       uint32_t* __restrict__ counts) {
  __shared__ uint32_t h[256];
  const int j = blockIdx.y, t = blockIdx.x;
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

// In-place exclusive scan of one column's counts in (digit, tile) order.
__global__ void __launch_bounds__(1024) radix_scan_kernel(uint32_t* __restrict__ counts, int tiles) {
  __shared__ uint32_t s_warp[33];
  __shared__ uint32_t s_carry;
  const int64_t total = static_cast<int64_t>(256) * tiles;
  uint32_t* c = counts + blockIdx.x * total;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t c0 = 0; c0 < total; c0 += blockDim.x) {
    const int64_t i = c0 + threadIdx.x;
    const uint32_t v = i < total ? c[i] : 0u;
    uint32_t incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = s_warp[lane], wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      s_warp[lane] = wi - w;
      if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    if (i < total) c[i] = s_carry + s_warp[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_warp[32];
    __syncthreads();
  }
}

// Stable scatter: keys of a tile, taken in order 256 at a time; equal digits
// inside a warp are ranked with ballots, across warps and rounds with counters.
__global__ void __launch_bounds__(kQThreads)
    radix_scatter_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int64_t N, int tiles, int shift,
                         const uint32_t* __restrict__ offsets) {
  constexpr int kWarps = kQThreads / 32;
  __shared__ uint32_t s_base[256];       // running position of each digit in this tile
  __shared__ uint32_t s_wc[kWarps][256];  // per-warp count, then per-warp start, of each digit
  const int j = blockIdx.y, t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s_base[threadIdx.x] = offsets[(static_cast<int64_t>(j) * 256 + threadIdx.x) * tiles + t];
  const uint32_t* k = in + j * N;
  uint32_t* o = out + j * N;
  const int64_t b0 = static_cast<int64_t>(t) * kQTile;
  const uint32_t lt = (1u << lane) - 1u;
  for (int r = 0; r < kQRounds; ++r) {
    for (int w = 0; w < kWarps; ++w) s_wc[w][threadIdx.x] = 0;
    __syncthreads();
    const int64_t i = b0 + r * kQThreads + threadIdx.x;
    const bool valid = i < N;
    const uint32_t key = valid ? k[i] : 0u;
    const uint32_t dg = (key >> shift) & 0xff;
    uint32_t peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t bal = __ballot_sync(0xffffffffu, (dg >> b) & 1u);
      peers &= ((dg >> b) & 1u) ? bal : ~bal;
    }
    const uint32_t rank = __popc(peers & lt);
    if (valid && rank == 0) s_wc[warp][dg] = __popc(peers);
    __syncthreads();
    {  // thread d: exclusive prefix over warps of digit d, advance the running base
      const int d = threadIdx.x;
      uint32_t run = s_base[d];
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = s_wc[w][d];
        s_wc[w][d] = run;
        run += c;
      }
      s_base[d] = run;
    }
    __syncthreads();
    if (valid) o[s_wc[warp][dg] + rank] = key;
    __syncthreads();
  }
}

// One CTA per column: distinct count, edges, n_bins.
__global__ void __launch_bounds__(1024)
    edges_kernel(const uint32_t* __restrict__ sorted, int64_t N, int j0, int B, float* __restrict__ edges,
                 int32_t* __restrict__ n_bins) {
  const int j = blockIdx.x;
  const uint32_t* v = sorted + j * N;
  __shared__ uint32_t s_warp[33];
  __shared__ float s_e[256];
  __shared__ int s_ne;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // run starts per contiguous thread chunk
  const int64_t per = (N + blockDim.x - 1) / blockDim.x;
  const int64_t a = threadIdx.x * per, bnd = min(N, a + per);
  uint32_t c = 0;
  for (int64_t i = a; i < bnd; ++i) c += (i == 0 || v[i] != v[i - 1]) ? 1u : 0u;
  uint32_t incl = c;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = s_warp[lane], wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const uint32_t U = s_warp[32];
  float* e = edges + static_cast<int64_t>(j0 + j) * (B - 1);
  if (U <= static_cast<uint32_t>(B)) {
    uint32_t r = s_warp[warp] + incl - c;  // rank of this thread's first run start
    for (int64_t i = a; i < bnd; ++i) {
      if (i == 0 || v[i] != v[i - 1]) {
        if (r + 1 < U) e[r] = key2f(v[i]);
        ++r;
      }
    }
    for (int k = static_cast<int>(U) - 1 + threadIdx.x; k < B - 1; k += blockDim.x) e[k] = INFINITY;
    if (threadIdx.x == 0) n_bins[j0 + j] = static_cast<int32_t>(U);
    return;
  }
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

__global__ void bin_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int j0, int B,
                           const float* __restrict__ edges, const int32_t* __restrict__ n_bins,
                           uint8_t* __restrict__ bins, int64_t ldb) {
  __shared__ float s_e[256];
  const int j = j0 + blockIdx.y;
  const int ne = n_bins[j] - 1;
  for (int k = threadIdx.x; k < ne; k += blockDim.x) s_e[k] = edges[static_cast<int64_t>(j) * (B - 1) + k];
  __syncthreads();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    const float x = X[j * ldx + i];
    int lo = 0, hi = ne;  // number of edges strictly below x
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_e[mid] < x) lo = mid + 1;
      else hi = mid;
    }
    bins[j * ldb + i] = static_cast<uint8_t>(lo);
  }
}

int batch_columns(int64_t N, int32_t F) {
  const size_t per_col = static_cast<size_t>(N) * 8 + static_cast<size_t>(256) * ceil_div(N, kQTile) * 4;
  int fb = static_cast<int>(kQBatchBudget / (per_col ? per_col : 1));
  return std::max(1, std::min<int>(fb, F));
}

struct QuantWs {
  uint32_t* a;
  uint32_t* b;
  uint32_t* counts;
  int32_t* flag;
};
QuantWs carve_quant(void* ws, size_t bytes, int64_t N, int32_t F, size_t* need) {
  Carve c(ws, bytes);
  QuantWs w{};
  const int fb = batch_columns(N, F);
  w.a = c.take<uint32_t>(static_cast<size_t>(fb) * N);
  w.b = c.take<uint32_t>(static_cast<size_t>(fb) * N);
  w.counts = c.take<uint32_t>(static_cast<size_t>(fb) * 256 * ceil_div(N, kQTile));
  w.flag = c.take<int32_t>(1);
  *need = c.used;
  return w;
}

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
  const int tiles = ceil_div(N, kQTile);
  for (int j0 = 0; j0 < F; j0 += fb) {
    const int nb = std::min(fb, F - j0);
    keys_kernel<<<dim3(gx, nb), 256, 0, s>>>(X, ldx, N, j0, w.a);
    count_launches();
    uint32_t* src = w.a;
    uint32_t* dst = w.b;
    for (int pass = 0; pass < 4; ++pass) {
      radix_count_kernel<<<dim3(tiles, nb), kQThreads, 0, s>>>(src, N, tiles, 8 * pass, w.counts);
      count_launches();
      radix_scan_kernel<<<nb, 1024, 0, s>>>(w.counts, tiles);
      count_launches();
      radix_scatter_kernel<<<dim3(tiles, nb), kQThreads, 0, s>>>(src, dst, N, tiles, 8 * pass, w.counts);
      count_launches();
      std::swap(src, dst);
    }
    edges_kernel<<<nb, 1024, 0, s>>>(src, N, j0, max_bins, edges, n_bins);
    count_launches();
    bin_kernel<<<dim3(gx, nb), 256, 0, s>>>(X, ldx, N, j0, max_bins, edges, n_bins, bins, ldb);
    count_launches();
    GBDT_LAUNCH_CHECK();
  }
  return GBDT_OK;
}
