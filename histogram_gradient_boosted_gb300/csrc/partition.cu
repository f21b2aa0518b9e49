// Partition of a level's rows into children.
//
// "Module Design: Training Core" s.6 step 5 (partition samples) and s.3
// (bin <= threshold_bin goes left).  Two forms:
//  * route_rows: the per-row node id (sample -> node map) is advanced to the
//    child node, in row order; this is what the level scan of the next level
//    reads;
//  * gbdt_partition: additionally the stable partition of each node's segment
//    of a row-index array (left rows first, input order kept on both sides),
//    built as a tile count, a per-segment scan and a block-scan scatter.
#include <mutex>

#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRowsPerRouteThread = 8;
constexpr int kTile = 4096;          // positions per partition tile
constexpr int kPartThreads = 256;
constexpr int kItems = kTile / kPartThreads;  // 16 consecutive positions per thread

__global__ void __launch_bounds__(kRouteThreads)
    route_rows_kernel(const uint8_t* __restrict__ bins, int64_t ldb, int64_t N, const Route* __restrict__ route,
                      const gbdt_level* __restrict__ level, int32_t max_slots, uint16_t* __restrict__ node_of_row,
                      int32_t* __restrict__ err) {
  extern __shared__ Route s_route[];
  const int node_begin = level->node_begin;
  const int n_slots = min(level->n_slots, max_slots);
  for (int s = threadIdx.x; s < n_slots; s += blockDim.x) s_route[s] = route[s];
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * kRowsPerRouteThread;
  for (int64_t r0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * kRowsPerRouteThread; r0 < N; r0 += stride) {
    uint16_t v[kRowsPerRouteThread];
    const bool full = r0 + kRowsPerRouteThread <= N;
    if (full) {
      uint4 w = *reinterpret_cast<const uint4*>(node_of_row + r0);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = static_cast<uint16_t>(ws[i] & 0xffffu);
        v[2 * i + 1] = static_cast<uint16_t>(ws[i] >> 16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerRouteThread; ++i) v[i] = (r0 + i < N) ? node_of_row[r0 + i] : 0xffffu;
    }
    bool changed = false;
#pragma unroll
    for (int i = 0; i < kRowsPerRouteThread; ++i) {
      const int slot = static_cast<int>(v[i]) - node_begin;
      if (slot < 0 || slot >= n_slots || r0 + i >= N) continue;
      const Route rt = s_route[slot];
      if (rt.feature < 0) continue;
      const int b = bins[static_cast<int64_t>(rt.feature) * ldb + r0 + i];
      v[i] = static_cast<uint16_t>(rt.left_node + (b > rt.bin ? 1 : 0));
      changed = true;
    }
    if (!changed) continue;
    if (full) {
      uint4 w;
      w.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
      w.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
      w.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
      w.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
      *reinterpret_cast<uint4*>(node_of_row + r0) = w;
    } else {
      for (int i = 0; i < kRowsPerRouteThread; ++i)
        if (r0 + i < N) node_of_row[r0 + i] = v[i];
    }
  }
  (void)err;
}

// ---- gbdt_partition ----------------------------------------------------------------------
struct PartState {
  int32_t total_tiles;
  int32_t n_splits;
};

// One CTA: child numbering (route table), tile offsets per slot, next level descriptor.
__global__ void part_setup_kernel(const gbdt_split* __restrict__ splits, const gbdt_level* __restrict__ level,
                                  int32_t max_slots, const gbdt_segment* __restrict__ seg_in, Route* __restrict__ route,
                                  int32_t* __restrict__ tile_start /*[max_slots+1]*/, PartState* __restrict__ st,
                                  gbdt_level* __restrict__ next_level) {
  __shared__ int s_split_pre, s_tile_pre;
  if (threadIdx.x == 0) s_split_pre = s_tile_pre = 0;
  __syncthreads();
  const int node_begin = level->node_begin;
  const int n_slots = min(level->n_slots, max_slots);
  const int next_begin = node_begin + level->n_slots;
  // sequential chunks of blockDim slots, block-scanned in order
  __shared__ int s_a[1024], s_b[1024];
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool in = s < n_slots;
    const int is_split = (in && splits[s].feature >= 0) ? 1 : 0;
    const int tiles = in ? static_cast<int>((seg_in[s].count + kTile - 1) / kTile) : 0;
    s_a[threadIdx.x] = is_split;
    s_b[threadIdx.x] = tiles;
    __syncthreads();
    for (int o = 1; o < blockDim.x; o <<= 1) {  // inclusive Hillis-Steele scan
      int a = threadIdx.x >= o ? s_a[threadIdx.x - o] : 0;
      int b = threadIdx.x >= o ? s_b[threadIdx.x - o] : 0;
      __syncthreads();
      s_a[threadIdx.x] += a;
      s_b[threadIdx.x] += b;
      __syncthreads();
    }
    if (in) {
      const int k = s_split_pre + s_a[threadIdx.x] - is_split;
      Route r;
      r.feature = is_split ? splits[s].feature : -1;
      r.bin = is_split ? splits[s].bin : -1;
      r.left_node = is_split ? next_begin + 2 * k : -1;
      r.pad = k;
      route[s] = r;
      tile_start[s] = s_tile_pre + s_b[threadIdx.x] - tiles;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      s_split_pre += s_a[threadIdx.x];
      s_tile_pre += s_b[threadIdx.x];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    tile_start[n_slots] = s_tile_pre;
    st->total_tiles = s_tile_pre;
    st->n_splits = s_split_pre;
    next_level->node_begin = next_begin;
    next_level->n_slots = 2 * s_split_pre;
  }
}

__device__ __forceinline__ int find_slot(const int32_t* __restrict__ tile_start, int n_slots, int t) {
  int lo = 0, hi = n_slots - 1;  // last slot with tile_start <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + incl - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPartThreads)
    part_count_kernel(const uint8_t* __restrict__ bins, int64_t ldb, const gbdt_level* __restrict__ level,
                      int32_t max_slots, const gbdt_segment* __restrict__ seg_in, const uint32_t* __restrict__ idx_in,
                      const Route* __restrict__ route, const int32_t* __restrict__ tile_start,
                      const PartState* __restrict__ st, int32_t* __restrict__ tile_left) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int n_slots = min(level->n_slots, max_slots);
  const int s = find_slot(tile_start, n_slots, t);
  const Route rt = route[s];
  __shared__ int s_warp[33];
  if (rt.feature < 0) {
    if (threadIdx.x == 0) tile_left[t] = 0;
    return;
  }
  const int64_t p0 = seg_in[s].start + static_cast<int64_t>(t - tile_start[s]) * kTile;
  const int64_t p1 = min(seg_in[s].start + seg_in[s].count, p0 + kTile);
  const uint8_t* col = bins + static_cast<int64_t>(rt.feature) * ldb;
  int c = 0;
  for (int i = 0; i < kItems; ++i) {
    const int64_t p = p0 + threadIdx.x * kItems + i;
    if (p < p1 && col[idx_in[p]] <= rt.bin) ++c;
  }
  int total;
  block_excl_scan(c, s_warp, &total);
  if (threadIdx.x == 0) tile_left[t] = total;
}

// One CTA: exclusive scan of the tile left counts over all tiles (tiles of a
// segment are contiguous, so a segment's offsets are differences of this
// scan); left totals and child segments per slot.
__global__ void part_scan_kernel(const gbdt_split* __restrict__ splits, const gbdt_level* __restrict__ level,
                                 int32_t max_slots, const gbdt_segment* __restrict__ seg_in,
                                 const Route* __restrict__ route, const int32_t* __restrict__ tile_start,
                                 const PartState* __restrict__ st, const int32_t* __restrict__ tile_left,
                                 int64_t* __restrict__ tile_excl /*[tiles+1]*/, int64_t* __restrict__ seg_left,
                                 gbdt_segment* __restrict__ seg_out, int32_t* __restrict__ err) {
  __shared__ int s_warp[33];
  __shared__ long long s_carry;
  const int total = st->total_tiles;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < total; c0 += blockDim.x) {
    const int t = c0 + threadIdx.x;
    const int v = t < total ? tile_left[t] : 0;
    int chunk_total;
    const int e = block_excl_scan(v, s_warp, &chunk_total);
    if (t < total) tile_excl[t] = s_carry + e;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) tile_excl[total] = s_carry;
  __syncthreads();
  const int n_slots = min(level->n_slots, max_slots);
  for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
    const Route rt = route[s];
    if (rt.feature < 0) continue;
    const int64_t left = tile_excl[tile_start[s + 1]] - tile_excl[tile_start[s]];
    seg_left[s] = left;
    if (left != static_cast<int64_t>(splits[s].cnt_left)) raise_error(err, kErrPartitionCount);
    const int k = rt.pad;
    seg_out[2 * k] = gbdt_segment{seg_in[s].start, left};
    seg_out[2 * k + 1] = gbdt_segment{seg_in[s].start + left, seg_in[s].count - left};
  }
}

__global__ void __launch_bounds__(kPartThreads)
    part_scatter_kernel(const uint8_t* __restrict__ bins, int64_t ldb, const gbdt_level* __restrict__ level,
                        int32_t max_slots, const gbdt_segment* __restrict__ seg_in, const uint32_t* __restrict__ idx_in,
                        const Route* __restrict__ route, const int32_t* __restrict__ tile_start,
                        const PartState* __restrict__ st, const int64_t* __restrict__ tile_excl,
                        const int64_t* __restrict__ seg_left, uint16_t* __restrict__ node_of_row,
                        uint32_t* __restrict__ idx_out) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int n_slots = min(level->n_slots, max_slots);
  const int s = find_slot(tile_start, n_slots, t);
  const Route rt = route[s];
  __shared__ int s_warp[33];
  const int64_t seg0 = seg_in[s].start;
  const int64_t tile_off = static_cast<int64_t>(t - tile_start[s]) * kTile;
  const int64_t p0 = seg0 + tile_off;
  const int64_t p1 = min(seg0 + seg_in[s].count, p0 + kTile);
  const int64_t pb = p0 + threadIdx.x * kItems;
  if (rt.feature < 0) {
    for (int i = 0; i < kItems; ++i)
      if (pb + i < p1) idx_out[pb + i] = idx_in[pb + i];
    return;
  }
  const uint8_t* col = bins + static_cast<int64_t>(rt.feature) * ldb;
  uint32_t rows[kItems];
  uint32_t left_mask = 0;
  int c = 0, n = 0;
  for (int i = 0; i < kItems; ++i) {
    const int64_t p = pb + i;
    if (p < p1) {
      rows[i] = idx_in[p];
      ++n;
      if (col[rows[i]] <= rt.bin) {
        left_mask |= 1u << i;
        ++c;
      }
    }
  }
  int total_left;
  const int lrank = block_excl_scan(c, s_warp, &total_left);
  const int64_t tile_left_off = tile_excl[t] - tile_excl[tile_start[s]];
  const int64_t left_base = seg0 + tile_left_off + lrank;
  // right rows before this thread: positions before it in the tile minus lefts before it
  const int64_t right_base = seg0 + seg_left[s] + (tile_off - tile_left_off) +
                             (static_cast<int64_t>(threadIdx.x) * kItems - lrank);
  int li = 0, ri = 0;
  for (int i = 0; i < n; ++i) {
    const uint32_t r = rows[i];
    if (left_mask & (1u << i)) {
      idx_out[left_base + li++] = r;
      node_of_row[r] = static_cast<uint16_t>(rt.left_node);
    } else {
      idx_out[right_base + ri++] = r;
      node_of_row[r] = static_cast<uint16_t>(rt.left_node + 1);
    }
  }
}

}  // namespace

void launch_route_rows(const uint8_t* bins, int64_t ldb, int64_t N, const Route* route, const gbdt_level* level,
                       int32_t max_slots, uint16_t* node_of_row, int32_t* err, cudaStream_t s) {
  const int64_t want = (N + kRouteThreads * kRowsPerRouteThread - 1) / (kRouteThreads * kRowsPerRouteThread);
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  const size_t smem = sizeof(Route) * static_cast<size_t>(max_slots);
  static bool once = (cudaFuncSetAttribute(route_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sizeof(Route) * kMaxSlots)),
                      true);
  (void)once;
  route_rows_kernel<<<grid, kRouteThreads, smem, s>>>(bins, ldb, N, route, level, max_slots, node_of_row, err);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

namespace {
struct PartWs {
  int32_t* err;
  PartState* st;
  Route* route;
  int32_t* tile_start;
  int32_t* tile_left;
  int64_t* tile_excl;
  int64_t* seg_left;
};
PartWs carve_partition(void* ws, size_t bytes, int64_t N, int32_t max_slots, size_t* need) {
  Carve c(ws, bytes);
  PartWs w{};
  w.err = c.take<int32_t>(1);
  w.st = c.take<PartState>(1);
  w.route = c.take<Route>(max_slots);
  w.tile_start = c.take<int32_t>(max_slots + 1);
  w.tile_left = c.take<int32_t>(static_cast<size_t>(ceil_div(N, kTile)) + max_slots);
  w.tile_excl = c.take<int64_t>(static_cast<size_t>(ceil_div(N, kTile)) + max_slots + 1);
  w.seg_left = c.take<int64_t>(max_slots);
  *need = c.used;
  return w;
}
}  // namespace

extern "C" size_t gbdt_partition_workspace_size(int64_t N, int32_t max_slots) {
  size_t need = 0;
  carve_partition(nullptr, 0, N, max_slots, &need);
  return need;
}

extern "C" int gbdt_partition(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const gbdt_split* splits,
                              const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg_in,
                              const uint32_t* idx_in, uint16_t* node_of_row, uint32_t* idx_out,
                              gbdt_segment* seg_out, gbdt_level* next_level, void* ws, size_t ws_bytes,
                              void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && splits && level && seg_in && idx_in && node_of_row && idx_out && seg_out && next_level,
                 "gbdt_partition: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && ldb >= N, "gbdt_partition: sizes out of range");
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kMaxSlots, "gbdt_partition: max_slots out of range");
  GBDT_CHECK_ARG(idx_in != idx_out, "gbdt_partition: idx_in and idx_out must differ");
  size_t need = 0;
  PartWs w = carve_partition(ws, ws_bytes, N, max_slots, &need);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_partition: workspace needs %zu bytes", need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GBDT_CUDA(cudaMemsetAsync(w.err, 0, sizeof(int32_t), s));
  part_setup_kernel<<<1, 1024, 0, s>>>(splits, level, max_slots, seg_in, w.route, w.tile_start, w.st, next_level);
  count_launches();
  const int max_tiles = ceil_div(N, kTile) + max_slots;
  part_count_kernel<<<max_tiles, kPartThreads, 0, s>>>(bins, ldb, level, max_slots, seg_in, idx_in, w.route,
                                                       w.tile_start, w.st, w.tile_left);
  count_launches();
  part_scan_kernel<<<1, 1024, 0, s>>>(splits, level, max_slots, seg_in, w.route, w.tile_start, w.st, w.tile_left,
                                      w.tile_excl, w.seg_left, seg_out, w.err);
  count_launches();
  part_scatter_kernel<<<max_tiles, kPartThreads, 0, s>>>(bins, ldb, level, max_slots, seg_in, idx_in, w.route,
                                                         w.tile_start, w.st, w.tile_excl, w.seg_left, node_of_row,
                                                         idx_out);
  count_launches();
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

// ---- gbdt_partition_noalloc: the same partition with library-owned scratch -------------------
// For callers that cannot allocate device memory: the scratch lives in one
// file-scope device array, sized for at most kNoAllocMaxRows rows and
// kNoAllocMaxSlots slots.  Every call on a device shares that array.
namespace {

constexpr int64_t kNoAllocMaxRows = int64_t(1) << 24;  // 16,777,216 rows
constexpr int32_t kNoAllocMaxSlots = 1024;
constexpr size_t kNoAllocScratchBytes = 128 * 1024;  // >= the carve for the limits above (about 90 KB)
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_partition_scratch[kNoAllocScratchBytes];

// The array's device address is looked up once per device and context: a cached address is reused
// only while the context it was taken in is the current one (a device reset, or a primary context
// released and created again, gives a new context and a new lookup).  Contexts are told apart by
// the driver's context id, which is never reused within a process.
using CtxGetCurrent = CUresult (*)(CUcontext*);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);

struct NoAllocEntry {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_noalloc_mu;
NoAllocEntry g_noalloc[kNoAllocMaxDevices] = {};

// Id of the current context (0 when there is none yet or the driver entry points are unavailable:
// then the address is looked up, which also creates the device's primary context).
unsigned long long current_context_id() {
  static CtxGetCurrent get_ctx = nullptr;
  static CtxGetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<CtxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetId>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context.
int noalloc_scratch(void** out) {
  int dev = -1;
  GBDT_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    set_error("gbdt_partition_noalloc: device %d outside the supported range", dev);
    return GBDT_ERR_INVALID_ARG;
  }
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocEntry& e = g_noalloc[dev];
  if (!e.ptr || id == 0 || e.ctx_id != id) {
    void* p = nullptr;
    GBDT_CUDA(cudaGetSymbolAddress(&p, g_partition_scratch));
    e.ptr = p;
    e.ctx_id = id;
  }
  *out = e.ptr;
  return GBDT_OK;
}

}  // namespace

extern "C" int gbdt_partition_noalloc(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F,
                                      const gbdt_split* splits, const gbdt_level* level, int32_t max_slots,
                                      const gbdt_segment* seg_in, const uint32_t* idx_in, uint16_t* node_of_row,
                                      uint32_t* idx_out, gbdt_segment* seg_out, gbdt_level* next_level,
                                      void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && splits && level && seg_in && idx_in && node_of_row && idx_out && seg_out && next_level,
                 "gbdt_partition_noalloc: null pointer");
  GBDT_CHECK_ARG(N >= 1 && F >= 1 && ldb >= N, "gbdt_partition_noalloc: sizes out of range");
  GBDT_CHECK_ARG(N <= kNoAllocMaxRows, "gbdt_partition_noalloc: N = %lld exceeds the limit of %lld rows of its "
                 "built-in scratch; use gbdt_partition with a workspace", (long long)N, (long long)kNoAllocMaxRows);
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kNoAllocMaxSlots, "gbdt_partition_noalloc: max_slots = %d outside "
                 "1..%d supported by its built-in scratch", max_slots, kNoAllocMaxSlots);
  GBDT_CHECK_ARG(idx_in != idx_out, "gbdt_partition_noalloc: idx_in and idx_out must differ");
  size_t need = 0;
  carve_partition(nullptr, 0, N, max_slots, &need);
  if (need > kNoAllocScratchBytes) {
    set_error("gbdt_partition_noalloc: needs %zu bytes of scratch, has %zu", need, kNoAllocScratchBytes);
    return GBDT_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != GBDT_OK) return rc;
  PartWs w = carve_partition(scratch, kNoAllocScratchBytes, N, max_slots, &need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word is the only scratch that must start at zero; the rest is rewritten by each call
  GBDT_CUDA(cudaMemsetAsync(w.err, 0, sizeof(int32_t), s));
  part_setup_kernel<<<1, 1024, 0, s>>>(splits, level, max_slots, seg_in, w.route, w.tile_start, w.st, next_level);
  count_launches();
  const int max_tiles = ceil_div(N, kTile) + max_slots;
  part_count_kernel<<<max_tiles, kPartThreads, 0, s>>>(bins, ldb, level, max_slots, seg_in, idx_in, w.route,
                                                       w.tile_start, w.st, w.tile_left);
  count_launches();
  part_scan_kernel<<<1, 1024, 0, s>>>(splits, level, max_slots, seg_in, w.route, w.tile_start, w.st, w.tile_left,
                                      w.tile_excl, w.seg_left, seg_out, w.err);
  count_launches();
  part_scatter_kernel<<<max_tiles, kPartThreads, 0, s>>>(bins, ldb, level, max_slots, seg_in, idx_in, w.route,
                                                         w.tile_start, w.st, w.tile_excl, w.seg_left, node_of_row,
                                                         idx_out);
  count_launches();
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" int gbdt_partition_noalloc_status(int32_t* bits, void* stream) {
  clear_error();
  if (bits) *bits = 0;
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != GBDT_OK) return rc;
  size_t need = 0;
  const PartWs w = carve_partition(scratch, kNoAllocScratchBytes, 1, 1, &need);  // the error word leads the carve
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  GBDT_CUDA(cudaMemcpyAsync(&h, w.err, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (bits) *bits = h;
  return report_error_bits("gbdt_partition_noalloc_status", h);
}
