// Level pass over node-contiguous rows.
//
// "Module Design: Training Core" s.6 steps 2 and 5: build the histograms of a
// level's nodes, and partition the samples into the children.  Here the
// partition moves the per-position data itself (every bin column, the
// gradient and the original row id), stably, so that each node's rows are one
// contiguous range of positions in every column.  Then:
//  * the histogram of a node reads only that node's range: one node per CTA,
//    up to 64 features per CTA in shared memory, no per-row node lookups, the
//    gradient of a row read once per CTA and reused for all its features;
//  * only the smaller child of each sibling pair is read (the larger comes by
//    subtraction), so a level reads at most half of the rows.
// The shared-memory accumulation is the exact fixed-point scheme of
// histogram.cu: 32-bit atomics only (count, low word with carry from the
// returned value, high word when needed), merged into global memory once.
//
// The partition is a tile count, a scan over tiles, and a move in which each
// CTA ranks its tile once and then streams several columns through shared
// memory, writing the left and right runs with aligned 16-byte stores.
#include <type_traits>

#include "kernels.cuh"

namespace gbdt {

namespace {

// ---------------------------------------------------------------------------------------- histograms
constexpr int kSegThreads = 1024;
constexpr int kSegMaxFeats = 64;  // features per CTA (64 x 256 x 12 B = 192 KB of shared memory)

struct SegWork {
  int64_t total_rows;  // rows over all built slots
  int32_t n_built;     // built slots
  int32_t ctas;        // CTAs per feature group that have rows
};

// One CTA: compact list of built slots, the prefix of their row counts, and
// how many CTAs per feature group share the rows (at most max_ctas, and no
// fewer than min_rows rows each).
__global__ void seg_work_setup_kernel(const gbdt_level* __restrict__ level, int32_t max_slots,
                                      const uint8_t* __restrict__ build_flag, const gbdt_segment* __restrict__ seg,
                                      int32_t max_ctas, int64_t min_rows, int32_t* __restrict__ build_slot,
                                      int64_t* __restrict__ row_start /*[max_slots+1]*/, SegWork* __restrict__ st) {
  __shared__ int s_a[1024];
  __shared__ long long s_b[1024];
  __shared__ int s_pre_slots;
  __shared__ long long s_pre_rows;
  if (threadIdx.x == 0) s_pre_slots = 0, s_pre_rows = 0;
  __syncthreads();
  const int n_slots = min(level->n_slots, max_slots);
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool in = s < n_slots && build_flag[s] && seg[s].count > 0;
    const long long rows = in ? seg[s].count : 0;
    s_a[threadIdx.x] = in ? 1 : 0;
    s_b[threadIdx.x] = rows;
    __syncthreads();
    for (int o = 1; o < blockDim.x; o <<= 1) {
      const int a = threadIdx.x >= o ? s_a[threadIdx.x - o] : 0;
      const long long b = threadIdx.x >= o ? s_b[threadIdx.x - o] : 0;
      __syncthreads();
      s_a[threadIdx.x] += a;
      s_b[threadIdx.x] += b;
      __syncthreads();
    }
    if (in) {
      const int k = s_pre_slots + s_a[threadIdx.x] - 1;
      build_slot[k] = s;
      row_start[k] = s_pre_rows + s_b[threadIdx.x] - rows;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      s_pre_slots += s_a[threadIdx.x];
      s_pre_rows += s_b[threadIdx.x];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    row_start[s_pre_slots] = s_pre_rows;
    st->total_rows = s_pre_rows;
    st->n_built = s_pre_slots;
    const long long by_size = (s_pre_rows + min_rows - 1) / min_rows;
    st->ctas = static_cast<int32_t>(by_size < max_ctas ? by_size : max_ctas);
  }
}

// Lane = feature: a warp takes 32 consecutive rows at a time and each lane adds
// those rows of one feature per group half (features j and j + 32), so the 32
// lanes of one atomic instruction update 32 different features' histograms.
// The shared histograms are stored bin-major with the lane innermost (word
// (half * 256 + bin) * 32 + lane for feature half * 32 + lane): every word a
// lane touches lies in the lane's own bank, so an atomic instruction is one
// shared-memory wavefront whatever the bins are.  Lanes with no feature in a
// half add to that half's unused entries (bin 0 of a feature past the group),
// which are never flushed: this keeps the update branch-free and costs no
// extra wavefront.  The fixed-point gradients of a 32-row block are staged
// per warp in shared memory and read back two rows per broadcast load.
constexpr int kHalfWords = kBins * 32;
constexpr uint32_t kHalfBytes = kHalfWords * 4;

// One exact fixed-point update, in two halves so that a warp can have several
// updates' atomics in flight: entry_lo adds the count and the low word and
// returns the low word's old value; entry_hi adds high part + carry (the carry
// out of old + low) to the high word.  The high-word add is unconditional:
// with the fixed-point scale the high part is non-zero for almost every row,
// and a skipped add would cost a branch, not a wavefront.  addr is the
// shared-memory byte address of the entry's count word; the low and high
// words sit kLo and kHi bytes above it.
template <uint32_t kLo>
__device__ __forceinline__ uint32_t entry_lo(uint32_t addr, uint32_t ql) {
  uint32_t old;
  asm volatile(
      "red.shared.add.u32 [%1], 1;\n\t"
      "atom.shared.add.u32 %0, [%1+%3], %2;"
      : "=r"(old)
      : "r"(addr), "r"(ql), "n"(kLo)
      : "memory");
  return old;
}

template <uint32_t kHi>
__device__ __forceinline__ void entry_hi(uint32_t addr, uint32_t ql, int32_t qh, uint32_t old) {
  asm volatile(
      "{\n\t.reg .u32 t;\n\t"
      "add.cc.u32 t, %2, %1;\n\t"
      "addc.s32 t, %3, 0;\n\t"
      "red.shared.add.s32 [%0+%4], t;\n\t}" ::"r"(addr),
      "r"(ql), "r"(old), "r"(qh), "n"(kHi)
      : "memory");
}

// Byte k of w times 128 (the byte stride between bins) plus base.
__device__ __forceinline__ uint32_t bin_addr(uint32_t w, int k, uint32_t base) {
  return base + (__byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(k)) << 7);
}

// Rows i and i + 1 of the block, every half: the low-word atomics of all of
// them are issued before the first carry is needed.
template <int NH, bool kFull>
__device__ __forceinline__ void seg_rows32(uint32_t base, const uint32_t (&w)[NH][8], const uint4* s_q,
                                           uint32_t valid) {
  constexpr uint32_t kLo = NH * kHalfBytes, kHi = 2 * NH * kHalfBytes;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    if (!kFull && !(valid >> i & 3u)) continue;  // warp-uniform
    const uint4 qq = s_q[i >> 1];  // rows i and i + 1: (low, high, low, high)
    const bool use1 = kFull || (valid >> (i + 1) & 1u);
    const bool use0 = kFull || (valid >> i & 1u);
    uint32_t a[2][NH], old[2][NH];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int h = 0; h < NH; ++h) a[r][h] = bin_addr(w[h][(i + r) >> 2], (i + r) & 3, base + h * kHalfBytes);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (use0) old[0][h] = entry_lo<kLo>(a[0][h], qq.x);
      if (use1) old[1][h] = entry_lo<kLo>(a[1][h], qq.z);
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (use0) entry_hi<kHi>(a[0][h], qq.x, static_cast<int32_t>(qq.y), old[0][h]);
      if (use1) entry_hi<kHi>(a[1][h], qq.z, static_cast<int32_t>(qq.w), old[1][h]);
    }
  }
}

// 32 bytes of a column (rows r0 .. r0 + 31 of one feature).  With kV8 the
// column starts are 32-byte aligned and one 256-bit load reads them all.
template <bool kV8>
__device__ __forceinline__ void load_rows32(const uint8_t* p, bool second, uint32_t (&w)[8]) {
  if (kV8 && second) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
    return;
  }
  const uint4 x0 = __ldg(reinterpret_cast<const uint4*>(p));
  const uint4 x1 = second ? __ldg(reinterpret_cast<const uint4*>(p + 16)) : make_uint4(0, 0, 0, 0);
  w[0] = x0.x, w[1] = x0.y, w[2] = x0.z, w[3] = x0.w;
  w[4] = x1.x, w[5] = x1.y, w[6] = x1.z, w[7] = x1.w;
}

// Add the rows at positions [p0, p1) of one slot to the CTA's shared histograms.
template <typename GT, int NH, bool kV8>
__device__ __forceinline__ void seg_hist_rows(uint32_t base, const uint8_t* const (&col)[NH], const bool (&has)[NH],
                                              const GT* __restrict__ g, double scale, int64_t p0, int64_t p1,
                                              uint4* s_q) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  // aligned 32-position blocks covering [p0, p1); positions outside are masked
  for (int64_t b = (p0 >> 5) + warp; (b << 5) < p1; b += n_warps) {
    const int64_t r0 = b << 5;
    const int64_t pr = r0 + lane;
    const bool v = pr >= p0 && pr < p1;
    const uint32_t valid = __ballot_sync(0xffffffffu, v);
    const int64_t q = v ? to_fixed(static_cast<double>(g[pr]), scale) : 0;
    const bool second = r0 + 16 < p1;  // any row of the block's upper half is in range
    uint32_t w[NH][8];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (has[h]) {
        load_rows32<kV8>(col[h] + r0, second, w[h]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[h][k] = 0;
      }
    }
    __syncwarp();
    reinterpret_cast<uint2*>(s_q)[lane] =
        make_uint2(static_cast<uint32_t>(static_cast<uint64_t>(q)), static_cast<uint32_t>(q >> 32));
    __syncwarp();
    if (valid == 0xffffffffu) seg_rows32<NH, true>(base, w, s_q, valid);
    else seg_rows32<NH, false>(base, w, s_q, valid);
  }
}

// Merge the CTA's shared histograms into slot's global histograms and leave
// the shared ones zeroed for the next slot.
template <int NH>
__device__ __forceinline__ void seg_hist_flush(uint32_t* s_cnt, uint32_t* s_lo, int32_t* s_hi, int slot, int32_t F,
                                               int f_lo, int nf, uint32_t* __restrict__ hist_cnt,
                                               int64_t* __restrict__ hist_q) {
  constexpr int entries = NH * kHalfWords;
  for (int e = threadIdx.x; e < entries; e += blockDim.x) {
    const uint32_t cn = s_cnt[e];
    if (cn == 0) continue;
    const int j = ((e / kHalfWords) << 5) + (e & 31);  // feature within the group
    const int64_t v = static_cast<int64_t>(s_hi[e]) * 4294967296ll + static_cast<int64_t>(s_lo[e]);
    s_cnt[e] = 0;
    s_lo[e] = 0;
    s_hi[e] = 0;
    if (j >= nf) continue;  // unused entries of lanes without a feature
    const int bin = (e >> 5) & (kBins - 1);
    const int64_t o = (static_cast<int64_t>(slot) * F + f_lo + j) * kBins + bin;
    atomicAdd(hist_cnt + o, cn);
    atomicAdd(reinterpret_cast<unsigned long long*>(hist_q + o), static_cast<unsigned long long>(v));
  }
}

// One CTA per (share of the level's built rows, feature group): the built
// slots' rows are concatenated in slot order and cut into equal shares, one
// per CTA, so the level runs as one balanced wave.  A share that crosses
// slot boundaries flushes its histograms at each crossing.
template <typename GT, bool kV8>
__global__ void __launch_bounds__(kSegThreads, 1)
    seg_hist_kernel(const uint8_t* __restrict__ bins, int64_t ldb, int32_t F, const GT* __restrict__ g,
                    const int32_t* __restrict__ fixed_exp, const gbdt_segment* __restrict__ seg,
                    const int32_t* __restrict__ build_slot, const int64_t* __restrict__ row_start,
                    const SegWork* __restrict__ st, int32_t group_feats, uint32_t* __restrict__ hist_cnt,
                    int64_t* __restrict__ hist_q) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int ctas = st->ctas;
  if (static_cast<int>(blockIdx.x) >= ctas) return;
  const int f_lo = blockIdx.y * group_feats;
  const int nf = min(group_feats, F - f_lo);
  if (nf <= 0) return;
  const int64_t total = st->total_rows;
  const int64_t lo = total * blockIdx.x / ctas, hi = total * (blockIdx.x + 1) / ctas;
  if (lo >= hi) return;
  const int n_built = st->n_built;
  int k = 0, kh = n_built - 1;  // last built slot whose first row <= lo
  while (k < kh) {
    const int mid = (k + kh + 1) >> 1;
    if (row_start[mid] <= lo) k = mid;
    else kh = mid - 1;
  }
  const double scale = ldexp(1.0, *fixed_exp);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto run = [&](auto nh_tag) {
    constexpr int NH = decltype(nh_tag)::value;
    constexpr int entries = NH * kHalfWords;
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(smem);
    uint32_t* s_lo = s_cnt + entries;
    int32_t* s_hi = reinterpret_cast<int32_t*>(s_lo + entries);
    uint4* s_q = reinterpret_cast<uint4*>(s_hi + entries) + warp * 16;  // 32 rows x (low, high)
    for (int e = threadIdx.x * 4; e < entries; e += blockDim.x * 4) {
      *reinterpret_cast<uint4*>(s_cnt + e) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(s_lo + e) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(s_hi + e) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const uint32_t base = smem_u32(s_cnt) + lane * 4;
    bool has[NH];
    const uint8_t* col[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      has[h] = h * 32 + lane < nf;
      col[h] = bins + static_cast<int64_t>(f_lo + (has[h] ? h * 32 + lane : 0)) * ldb;
    }
    for (int64_t r = lo; r < hi; ++k) {
      const int64_t r_end = min(hi, row_start[k + 1]);
      const int slot = build_slot[k];
      const int64_t p0 = seg[slot].start + (r - row_start[k]);
      seg_hist_rows<GT, NH, kV8>(base, col, has, g, scale, p0, p0 + (r_end - r), s_q);
      __syncthreads();
      seg_hist_flush<NH>(s_cnt, s_lo, s_hi, slot, F, f_lo, nf, hist_cnt, hist_q);
      __syncthreads();
      r = r_end;
    }
  };
  if (group_feats > 32) run(std::integral_constant<int, 2>{});
  else run(std::integral_constant<int, 1>{});
}

// ---------------------------------------------------------------------------------------- partition
constexpr int kMvThreads = 256;
constexpr int kMvTile = 4096;  // positions per tile

struct MvState {
  int32_t total_tiles;
  int32_t pad;
};

// One CTA: tiles per slot (every slot of the level: split slots are moved,
// the others have their rows recorded as leaves).
__global__ void mv_setup_kernel(const gbdt_level* __restrict__ level, int32_t max_slots,
                                const gbdt_segment* __restrict__ seg, int32_t* __restrict__ tile_start,
                                MvState* __restrict__ st) {
  __shared__ int s_b[1024];
  __shared__ int s_pre;
  if (threadIdx.x == 0) s_pre = 0;
  __syncthreads();
  const int n_slots = min(level->n_slots, max_slots);
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const int tiles = s < n_slots ? static_cast<int>((seg[s].count + kMvTile - 1) / kMvTile) : 0;
    s_b[threadIdx.x] = tiles;
    __syncthreads();
    for (int o = 1; o < blockDim.x; o <<= 1) {
      const int b = threadIdx.x >= o ? s_b[threadIdx.x - o] : 0;
      __syncthreads();
      s_b[threadIdx.x] += b;
      __syncthreads();
    }
    if (s < n_slots) tile_start[s] = s_pre + s_b[threadIdx.x] - tiles;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_pre += s_b[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    tile_start[n_slots] = s_pre;
    st->total_tiles = s_pre;
  }
}

__device__ __forceinline__ int slot_of_tile(const int32_t* __restrict__ tile_start, int n_slots, int t) {
  int lo = 0, hi = n_slots - 1;  // last slot whose first tile <= t (skips empty slots)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int block_scan_excl(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
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

// Decision of position p of a split slot: 1 = goes right.
__device__ __forceinline__ int goes_right(const uint8_t* __restrict__ col, int bin, const uint8_t* __restrict__ go_right,
                                          int64_t p) {
  return go_right ? (go_right[p] != 0) : (col[p] > bin);
}

__global__ void __launch_bounds__(kMvThreads)
    mv_count_kernel(const uint8_t* __restrict__ bins, int64_t ldb, const uint8_t* __restrict__ go_right,
                    const gbdt_level* __restrict__ level, int32_t max_slots, const gbdt_segment* __restrict__ seg,
                    const Route* __restrict__ route, const int32_t* __restrict__ tile_start,
                    const MvState* __restrict__ st, int32_t* __restrict__ tile_left) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  __shared__ int s_warp[33];
  const int n_slots = min(level->n_slots, max_slots);
  const int s = slot_of_tile(tile_start, n_slots, t);
  const Route rt = route[s];
  if (rt.feature < 0) {
    if (threadIdx.x == 0) tile_left[t] = 0;
    return;
  }
  const int64_t p0 = seg[s].start + static_cast<int64_t>(t - tile_start[s]) * kMvTile;
  const int n = static_cast<int>(min(seg[s].start + seg[s].count - p0, static_cast<int64_t>(kMvTile)));
  const uint8_t* col = bins + static_cast<int64_t>(rt.feature) * ldb;
  int c = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) c += 1 - goes_right(col, rt.bin, go_right, p0 + j);
  int total;
  block_scan_excl(c, s_warp, &total);
  if (threadIdx.x == 0) tile_left[t] = total;
}

// One CTA: exclusive scan of tile left counts over all tiles; left totals per slot.
__global__ void __launch_bounds__(1024)
    mv_scan_kernel(const gbdt_level* __restrict__ level, int32_t max_slots, const Route* __restrict__ route,
                   const int32_t* __restrict__ tile_start, const MvState* __restrict__ st,
                   const int32_t* __restrict__ tile_left, int64_t* __restrict__ tile_excl,
                   int64_t* __restrict__ seg_left, const gbdt_segment* __restrict__ seg, gbdt_segment* __restrict__ seg_out,
                   const gbdt_split* __restrict__ splits, int32_t* __restrict__ err) {
  __shared__ int s_warp[33];
  __shared__ long long s_carry;
  const int total = st->total_tiles;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < total; c0 += blockDim.x) {
    const int t = c0 + threadIdx.x;
    const int v = t < total ? tile_left[t] : 0;
    int chunk_total;
    const int e = block_scan_excl(v, s_warp, &chunk_total);
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
    if (splits && left != static_cast<int64_t>(splits[s].cnt_left)) raise_error(err, kErrPartitionCount);
    if (seg_out) {
      const int k = rt.pad;
      seg_out[2 * k] = gbdt_segment{seg[s].start, left};
      seg_out[2 * k + 1] = gbdt_segment{seg[s].start + left, seg[s].count - left};
    }
  }
}

// Column c < F: bins column c; c == F: gradient (4 or 8 B); c == F + 1: original row id (4 B).
// Output-centric move.  Once per tile: the rows' decisions (lane = row,
// ballots), their ranks, and the inverse permutation inv[o] = tile position of
// the o-th output row (left rows first, then right rows) in shared memory.
// The gradient and the row id move one output position per thread, in
// batches of independent loads.  For the bin columns each thread owns up to
// kMvWordsPerThread aligned 4-byte words of the tile's two output runs and
// keeps, in registers, the source positions of their bytes; every output word
// is gathered from the column's tile in shared memory and written with one
// aligned 4-byte store (byte stores only where a run starts or ends inside a
// word), so stores fill whole sectors.  The column tiles arrive by bulk
// asynchronous copies, kMvStages columns ahead of the one being gathered, so
// the loads of later columns overlap the gathers and stores of earlier ones.
constexpr int kMvChunks = kMvTile / 32;
constexpr int kMvChunksPerWarp = kMvChunks / (kMvThreads / 32);
constexpr int kMvWordsPerThread = (kMvTile / 4 + 4 + kMvThreads - 1) / kMvThreads;  // 5: both runs, edges included
constexpr int kMvStages = 4;
constexpr int kMvStageBytes = kMvTile + 16;  // a tile plus its 16-byte alignment slack
constexpr uint32_t kMvWaitPolls = 1u << 20;

template <typename T>
__device__ __forceinline__ void move_positions(const T* __restrict__ in, T* __restrict__ out, int64_t p0, int n,
                                               int nl, int64_t dst_l, int64_t dst_r, const uint16_t* s_inv) {
  constexpr int U = 8;
  for (int o0 = threadIdx.x; o0 < n; o0 += U * kMvThreads) {
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int o = o0 + u * kMvThreads;
      if (o < n) v[u] = in[p0 + s_inv[o]];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int o = o0 + u * kMvThreads;
      if (o < n) out[o < nl ? dst_l + o : dst_r + (o - nl)] = v[u];
    }
  }
}

__global__ void __launch_bounds__(kMvThreads, 4)
    mv_move_kernel(const uint8_t* __restrict__ bins_in, uint8_t* __restrict__ bins_out, int64_t ldb, int32_t F,
                   const void* __restrict__ g_in, void* __restrict__ g_out, int g_size,
                   const uint32_t* __restrict__ orig_in, uint32_t* __restrict__ orig_out,
                   const uint8_t* __restrict__ go_right, const gbdt_level* __restrict__ level, int32_t max_slots,
                   const gbdt_segment* __restrict__ seg, const Route* __restrict__ route,
                   const int32_t* __restrict__ tile_start, const MvState* __restrict__ st,
                   const int64_t* __restrict__ tile_excl, const int64_t* __restrict__ seg_left,
                   uint16_t* __restrict__ leaf_of_row, int32_t* __restrict__ err) {
  __shared__ uint32_t s_right[kMvChunks];
  __shared__ uint32_t s_valid[kMvChunks];
  __shared__ int s_lbase[kMvChunks];
  __shared__ uint16_t s_inv[kMvTile];
  __shared__ __align__(128) uint8_t s_stage[kMvStages][kMvStageBytes];
  __shared__ __align__(8) uint64_t s_full[kMvStages];
  __shared__ int s_warp[33];
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int n_slots = min(level->n_slots, max_slots);
  const int s = slot_of_tile(tile_start, n_slots, t);
  const Route rt = route[s];
  const int64_t tile_off = static_cast<int64_t>(t - tile_start[s]) * kMvTile;
  const int64_t p0 = seg[s].start + tile_off;
  const int n = static_cast<int>(min(seg[s].start + seg[s].count - p0, static_cast<int64_t>(kMvTile)));
  if (rt.feature < 0) {  // a leaf: remember each row's leaf, nothing moves
    if (leaf_of_row) {
      const uint16_t node = static_cast<uint16_t>(level->node_begin + s);
      for (int i = threadIdx.x; i < n; i += blockDim.x) leaf_of_row[orig_in[p0 + i]] = node;
    }
    return;
  }
  // ---- start the first column copies: the tile's 16-byte-aligned span of each column
  const int64_t a0 = p0 & ~int64_t(15);
  const uint32_t span = static_cast<uint32_t>(((p0 + n + 15) & ~int64_t(15)) - a0);
  const int a_off = static_cast<int>(p0 & 15);  // stage index of tile position 0
  if (threadIdx.x == 0) {
    for (int k = 0; k < kMvStages; ++k) mbar_init(&s_full[k], 1);
    mbar_init_fence();
    for (int c = 0; c < F && c < kMvStages; ++c) bulk_load(s_stage[c], bins_in + c * ldb + a0, span, &s_full[c]);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint8_t* col = bins_in + static_cast<int64_t>(rt.feature) * ldb;
  // ---- rank the tile (lane = row) and build the inverse permutation
#pragma unroll 1
  for (int k = 0; k < kMvChunksPerWarp; ++k) {
    const int ch = warp * kMvChunksPerWarp + k;
    const int j = ch * 32 + lane;
    const bool v = j < n;
    const int r = v ? goes_right(col, rt.bin, go_right, p0 + j) : 0;
    const uint32_t rm = __ballot_sync(0xffffffffu, r);
    const uint32_t vm = __ballot_sync(0xffffffffu, v);
    if (lane == 0) {
      s_right[ch] = rm;
      s_valid[ch] = vm;
    }
  }
  __syncthreads();
  const int lc = threadIdx.x < kMvChunks ? __popc(s_valid[threadIdx.x] & ~s_right[threadIdx.x]) : 0;
  int nl;
  const int lex = block_scan_excl(lc, s_warp, &nl);
  if (threadIdx.x < kMvChunks) s_lbase[threadIdx.x] = lex;
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll 1
  for (int k = 0; k < kMvChunksPerWarp; ++k) {
    const int ch = warp * kMvChunksPerWarp + k;
    const uint32_t vm = s_valid[ch], rm = s_right[ch];
    if (vm >> lane & 1u) {
      const int lb = s_lbase[ch];
      const int o = (rm >> lane & 1u) ? nl + (ch * 32 - lb) + __popc(rm & lt) : lb + __popc(vm & ~rm & lt);
      s_inv[o] = static_cast<uint16_t>(ch * 32 + lane);
    }
  }
  __syncthreads();
  const int nr = n - nl;
  const int64_t left_before = tile_excl[t] - tile_excl[tile_start[s]];
  const int64_t dst_l = seg[s].start + left_before;                             // this tile's left run
  const int64_t dst_r = seg[s].start + seg_left[s] + (tile_off - left_before);  // this tile's right run
  // ---- gradient and row id, while the first column copies are in flight
  if (g_size == 8)
    move_positions(static_cast<const uint64_t*>(g_in), static_cast<uint64_t*>(g_out), p0, n, nl, dst_l, dst_r, s_inv);
  else
    move_positions(static_cast<const uint32_t*>(g_in), static_cast<uint32_t*>(g_out), p0, n, nl, dst_l, dst_r, s_inv);
  move_positions(orig_in, orig_out, p0, n, nl, dst_l, dst_r, s_inv);
  // ---- the output words this thread owns: left run words, then right run words
  const int64_t wl0 = dst_l >> 2, wr0 = dst_r >> 2;
  const int nwl = nl > 0 ? static_cast<int>(((dst_l + nl + 3) >> 2) - wl0) : 0;
  const int nwr = nr > 0 ? static_cast<int>(((dst_r + nr + 3) >> 2) - wr0) : 0;
  const int ol = static_cast<int>(dst_l & 3), orr = static_cast<int>(dst_r & 3);  // run start inside its first word
  int wrel[kMvWordsPerThread];       // word offset within its run's words; bit 30: right run; -1: none
  uint32_t srcl[kMvWordsPerThread];  // stage positions of bytes 0,1 (16 bits each; 0xffff: not written)
  uint32_t srch[kMvWordsPerThread];  // stage positions of bytes 2,3
#pragma unroll
  for (int m = 0; m < kMvWordsPerThread; ++m) {
    const int vw = threadIdx.x + m * kMvThreads;
    uint32_t sp[4] = {0xffffu, 0xffffu, 0xffffu, 0xffffu};
    int wr = -1;
    if (vw < nwl + nwr) {
      const bool left = vw < nwl;
      const int rel = left ? vw : vw - nwl;
      const int len = left ? nl : nr, base = left ? 0 : nl, first = left ? ol : orr;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int o = 4 * rel + i - first;  // offset in the run
        if (o >= 0 && o < len) sp[i] = s_inv[base + o] + a_off;
      }
      wr = left ? rel : (rel | 0x40000000);
    }
    wrel[m] = wr;
    srcl[m] = sp[0] | (sp[1] << 16);
    srch[m] = sp[2] | (sp[3] << 16);
  }
  // ---- bin columns, each from its stage
  int c_fail = -1;
#pragma unroll 1
  for (int c = 0; c < F; ++c) {
    const int k = c % kMvStages;
    const uint8_t* stage = s_stage[k];
    const bool ok = mbar_wait(&s_full[k], static_cast<uint32_t>((c / kMvStages) & 1), kMvWaitPolls);
    if (ok) {
      uint32_t* out = reinterpret_cast<uint32_t*>(bins_out + static_cast<int64_t>(c) * ldb);
#pragma unroll
      for (int m = 0; m < kMvWordsPerThread; ++m) {
        const int wr = wrel[m];
        if (wr < 0) continue;
        const int64_t wa = (wr & 0x40000000) ? wr0 + (wr & 0x3fffffff) : wl0 + wr;
        const uint32_t s0 = srcl[m] & 0xffffu, s1 = srcl[m] >> 16, s2 = srch[m] & 0xffffu, s3 = srch[m] >> 16;
        if (s0 != 0xffffu && s1 != 0xffffu && s2 != 0xffffu && s3 != 0xffffu) {
          out[wa] = static_cast<uint32_t>(stage[s0]) | (static_cast<uint32_t>(stage[s1]) << 8) |
                    (static_cast<uint32_t>(stage[s2]) << 16) | (static_cast<uint32_t>(stage[s3]) << 24);
        } else {  // a run starts or ends inside this word: write only its own bytes
          uint8_t* ob = reinterpret_cast<uint8_t*>(out + wa);
          if (s0 != 0xffffu) ob[0] = stage[s0];
          if (s1 != 0xffffu) ob[1] = stage[s1];
          if (s2 != 0xffffu) ob[2] = stage[s2];
          if (s3 != 0xffffu) ob[3] = stage[s3];
        }
      }
    }
    if (__syncthreads_or(!ok)) {  // every thread is done with this stage (or a copy timed out)
      c_fail = c;
      break;
    }
    if (threadIdx.x == 0 && c + kMvStages < F)
      bulk_load(s_stage[k], bins_in + static_cast<int64_t>(c + kMvStages) * ldb + a0, span, &s_full[k]);
  }
  if (c_fail >= 0 && threadIdx.x == 0) {
    raise_error(err, kErrWaitTimeout);
    // let the copies still in flight (columns c_fail .. issued - 1) land before the CTA's shared memory is
    // released; each stage completes in order, so waiting for its last issued column suffices
    const int issued = min(F, c_fail + kMvStages);
    for (int c = c_fail; c < issued; ++c) {
      if (c + kMvStages < issued) continue;  // a later column of the same stage is waited for instead
      mbar_wait(&s_full[c % kMvStages], static_cast<uint32_t>((c / kMvStages) & 1), kMvWaitPolls);
    }
  }
}

// Last split level: the children are leaves, so nothing moves.  Every row
// records its leaf: the child its split sends it to, or the slot's own node
// when the slot did not split.
__global__ void __launch_bounds__(kMvThreads)
    mv_leaves_kernel(const uint8_t* __restrict__ bins_in, int64_t ldb, const uint32_t* __restrict__ orig_in,
                     const uint8_t* __restrict__ go_right, const gbdt_level* __restrict__ level, int32_t max_slots,
                     const gbdt_segment* __restrict__ seg, const Route* __restrict__ route,
                     const int32_t* __restrict__ tile_start, const MvState* __restrict__ st,
                     uint16_t* __restrict__ leaf_of_row) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int n_slots = min(level->n_slots, max_slots);
  const int s = slot_of_tile(tile_start, n_slots, t);
  const Route rt = route[s];
  const int64_t p0 = seg[s].start + static_cast<int64_t>(t - tile_start[s]) * kMvTile;
  const int n = static_cast<int>(min(seg[s].start + seg[s].count - p0, static_cast<int64_t>(kMvTile)));
  if (rt.feature < 0) {
    const uint16_t node = static_cast<uint16_t>(level->node_begin + s);
    for (int i = threadIdx.x; i < n; i += blockDim.x) leaf_of_row[orig_in[p0 + i]] = node;
    return;
  }
  const uint8_t* col = bins_in + static_cast<int64_t>(rt.feature) * ldb;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    leaf_of_row[orig_in[p0 + i]] = static_cast<uint16_t>(rt.left_node + goes_right(col, rt.bin, go_right, p0 + i));
}

// One CTA: routing of every slot from its split record; the k-th splitting slot
// (in slot order) gets child slots 2k, 2k+1 of the next level.
__global__ void routes_from_splits_kernel(const gbdt_split* __restrict__ splits, const gbdt_level* __restrict__ level,
                                          int32_t max_slots, Route* __restrict__ route,
                                          gbdt_level* __restrict__ next_level) {
  __shared__ int s_a[1024];
  __shared__ int s_pre;
  if (threadIdx.x == 0) s_pre = 0;
  __syncthreads();
  const int n_slots = min(level->n_slots, max_slots);
  const int next_begin = level->node_begin + level->n_slots;
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const int sp = (s < n_slots && splits[s].feature >= 0) ? 1 : 0;
    s_a[threadIdx.x] = sp;
    __syncthreads();
    for (int o = 1; o < blockDim.x; o <<= 1) {
      const int a = threadIdx.x >= o ? s_a[threadIdx.x - o] : 0;
      __syncthreads();
      s_a[threadIdx.x] += a;
      __syncthreads();
    }
    if (s < n_slots) {
      const int k = s_pre + s_a[threadIdx.x] - sp;
      route[s] = sp ? Route{splits[s].feature, splits[s].bin, next_begin + 2 * k, k} : Route{-1, -1, -1, k};
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_pre += s_a[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0 && next_level) {
    next_level->node_begin = next_begin;
    next_level->n_slots = 2 * s_pre;
  }
}

template <typename K>
cudaError_t smem_attr(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

}  // namespace

// ---- plans and launchers ------------------------------------------------------------------------
SegHistPlan plan_seg_histograms(int64_t N, int32_t F, int32_t max_slots, int32_t max_build) {
  (void)N, (void)max_slots, (void)max_build;
  SegHistPlan p{};
  p.n_fgroups = ceil_div(F, kSegMaxFeats);
  p.group_feats = ceil_div(F, p.n_fgroups);
  p.max_ctas = sm_count() / p.n_fgroups;  // one wave: a CTA per SM
  if (p.max_ctas < 1) p.max_ctas = 1;
  p.min_rows = 4096;
  p.smem = static_cast<size_t>(ceil_div(p.group_feats, 32)) * kHalfWords * 12 + (kSegThreads / 32) * 256;
  return p;
}

size_t seg_hist_scratch_bytes(int32_t max_slots) {
  return sizeof(SegWork) + sizeof(int32_t) * (static_cast<size_t>(max_slots) + 1) +
         sizeof(int64_t) * (static_cast<size_t>(max_slots) + 1) + 3 * kWsAlign;
}

int launch_seg_histograms(const SegHistPlan& plan, const uint8_t* bins, int64_t ldb, int64_t N, int32_t F,
                          const void* g, int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                          int32_t max_slots, const uint8_t* build_flag, const gbdt_segment* seg, void* scratch,
                          uint32_t* hist_cnt, int64_t* hist_q, cudaStream_t s) {
  (void)N;
  Carve c(scratch, seg_hist_scratch_bytes(max_slots));
  SegWork* st = c.take<SegWork>(1);
  int32_t* build_slot = c.take<int32_t>(max_slots + 1);
  int64_t* row_start = c.take<int64_t>(max_slots + 1);
  launch_hist_zero(level, max_slots, build_flag, F, hist_cnt, hist_q, s);
  seg_work_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, build_flag, seg, plan.max_ctas, plan.min_rows,
                                           build_slot, row_start, st);
  count_launches();
  dim3 grid(static_cast<unsigned>(plan.max_ctas), static_cast<unsigned>(plan.n_fgroups));
  // 256-bit column loads need every column start 32-byte aligned
  const bool v8 = aligned(bins, 32) && ldb % 32 == 0;
  auto launch = [&](auto kernel, const auto* gp) -> int {
    GBDT_CUDA(smem_attr(kernel, plan.smem));
    kernel<<<grid, kSegThreads, plan.smem, s>>>(bins, ldb, F, gp, fixed_exp, seg, build_slot, row_start, st,
                                                plan.group_feats, hist_cnt, hist_q);
    return GBDT_OK;
  };
  int rc;
  if (g_dtype == GBDT_DTYPE_F32) {
    const float* gp = static_cast<const float*>(g);
    rc = v8 ? launch(seg_hist_kernel<float, true>, gp) : launch(seg_hist_kernel<float, false>, gp);
  } else {
    const double* gp = static_cast<const double*>(g);
    rc = v8 ? launch(seg_hist_kernel<double, true>, gp) : launch(seg_hist_kernel<double, false>, gp);
  }
  if (rc != GBDT_OK) return rc;
  count_launches();
  return GBDT_OK;
}

size_t move_scratch_bytes(int64_t N, int32_t max_slots) {
  const size_t tiles = static_cast<size_t>(ceil_div(N, kMvTile)) + max_slots;
  return sizeof(MvState) + sizeof(int32_t) * (max_slots + 1) + sizeof(int32_t) * tiles +
         sizeof(int64_t) * (tiles + 1) + sizeof(int64_t) * max_slots + 6 * kWsAlign;
}

void launch_move_rows(const uint8_t* bins_in, uint8_t* bins_out, int64_t ldb, int64_t N, int32_t F,
                      const void* g_in, void* g_out, int g_size, const uint32_t* orig_in, uint32_t* orig_out,
                      const uint8_t* go_right, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, const gbdt_split* splits, gbdt_segment* seg_out,
                      uint16_t* leaf_of_row, void* scratch, int32_t* err, cudaStream_t s) {
  Carve c(scratch, move_scratch_bytes(N, max_slots));
  MvState* st = c.take<MvState>(1);
  int32_t* tile_start = c.take<int32_t>(max_slots + 1);
  const int max_tiles = ceil_div(N, kMvTile) + max_slots;
  int32_t* tile_left = c.take<int32_t>(max_tiles);
  int64_t* tile_excl = c.take<int64_t>(max_tiles + 1);
  int64_t* seg_left = c.take<int64_t>(max_slots);
  mv_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, seg, tile_start, st);
  count_launches();
  mv_count_kernel<<<max_tiles, kMvThreads, 0, s>>>(bins_in, ldb, go_right, level, max_slots, seg, route, tile_start,
                                                   st, tile_left);
  count_launches();
  mv_scan_kernel<<<1, 1024, 0, s>>>(level, max_slots, route, tile_start, st, tile_left, tile_excl, seg_left, seg,
                                    seg_out, splits, err);
  count_launches();
  mv_move_kernel<<<max_tiles, kMvThreads, 0, s>>>(bins_in, bins_out, ldb, F, g_in, g_out, g_size, orig_in, orig_out,
                                             go_right,
                                             level, max_slots, seg, route, tile_start, st, tile_excl, seg_left,
                                             leaf_of_row, err);
  count_launches();
}

void launch_leaf_rows(const uint8_t* bins_in, int64_t ldb, int64_t N, const uint32_t* orig_in,
                      const uint8_t* go_right, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, uint16_t* leaf_of_row, void* scratch, cudaStream_t s) {
  Carve c(scratch, move_scratch_bytes(N, max_slots));
  MvState* st = c.take<MvState>(1);
  int32_t* tile_start = c.take<int32_t>(max_slots + 1);
  const int max_tiles = ceil_div(N, kMvTile) + max_slots;
  mv_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, seg, tile_start, st);
  count_launches();
  mv_leaves_kernel<<<max_tiles, kMvThreads, 0, s>>>(bins_in, ldb, orig_in, go_right, level, max_slots, seg, route,
                                                    tile_start, st, leaf_of_row);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

extern "C" size_t gbdt_histograms_segmented_workspace_size(int32_t max_slots) {
  return seg_hist_scratch_bytes(max_slots);
}

extern "C" int gbdt_build_histograms_segmented(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g,
                                               int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                                               int32_t max_slots, const uint8_t* build_flag, int32_t max_build,
                                               const gbdt_segment* segments, uint32_t* hist_cnt, int64_t* hist_q,
                                               void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && g && fixed_exp && level && build_flag && segments && hist_cnt && hist_q,
                 "gbdt_build_histograms_segmented: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 4096,
                 "gbdt_build_histograms_segmented: sizes out of range");
  GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins, 16) && aligned(g, 16),
                 "gbdt_build_histograms_segmented: need ldb >= N, ldb %% 16 == 0, 16-byte aligned bins and g");
  GBDT_CHECK_ARG(g_dtype == GBDT_DTYPE_F32 || g_dtype == GBDT_DTYPE_F64, "gbdt_build_histograms_segmented: bad dtype");
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kMaxSlots && max_build >= 1 && max_build <= max_slots,
                 "gbdt_build_histograms_segmented: slot bounds out of range");
  if (!ws || ws_bytes < seg_hist_scratch_bytes(max_slots) || !aligned(ws, kWsAlign)) {
    set_error("gbdt_build_histograms_segmented: workspace needs %zu bytes", seg_hist_scratch_bytes(max_slots));
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SegHistPlan plan = plan_seg_histograms(N, F, max_slots, max_build);
  int rc = launch_seg_histograms(plan, bins, ldb, N, F, g, g_dtype, fixed_exp, level, max_slots, build_flag, segments,
                                 ws, hist_cnt, hist_q, s);
  if (rc != GBDT_OK) return rc;
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

namespace {
struct RowsWs {
  int32_t* err;
  Route* route;
  void* move;
};
RowsWs carve_rows(void* ws, size_t bytes, int64_t N, int32_t max_slots, size_t* need) {
  Carve c(ws, bytes);
  RowsWs w{};
  w.err = c.take<int32_t>(1);
  w.route = c.take<Route>(max_slots);
  w.move = c.take<unsigned char>(move_scratch_bytes(N, max_slots));
  *need = c.used;
  return w;
}
}  // namespace

extern "C" size_t gbdt_partition_rows_workspace_size(int64_t N, int32_t max_slots) {
  size_t need = 0;
  carve_rows(nullptr, 0, N, max_slots, &need);
  return need;
}

extern "C" int gbdt_partition_rows(const uint8_t* bins_in, uint8_t* bins_out, int64_t ldb, int64_t N, int32_t F,
                                   const void* g_in, void* g_out, int32_t g_dtype, const uint32_t* orig_in,
                                   uint32_t* orig_out, const uint8_t* go_right, const gbdt_split* splits,
                                   const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg_in,
                                   gbdt_segment* seg_out, gbdt_level* next_level, uint16_t* leaf_of_row, void* ws,
                                   size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins_in && bins_out && g_in && g_out && orig_in && orig_out && splits && level && seg_in && seg_out,
                 "gbdt_partition_rows: null pointer");
  GBDT_CHECK_ARG(bins_in != bins_out && g_in != g_out && orig_in != orig_out,
                 "gbdt_partition_rows: inputs and outputs must not alias");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 4096, "gbdt_partition_rows: sizes out of range");
  GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins_in, 16) && aligned(bins_out, 16),
                 "gbdt_partition_rows: need ldb >= N, ldb %% 16 == 0 and 16-byte aligned bins");
  GBDT_CHECK_ARG(g_dtype == GBDT_DTYPE_F32 || g_dtype == GBDT_DTYPE_F64, "gbdt_partition_rows: bad g dtype");
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kMaxSlots, "gbdt_partition_rows: max_slots out of range");
  size_t need = 0;
  RowsWs w = carve_rows(ws, ws_bytes, N, max_slots, &need);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_partition_rows: workspace needs %zu bytes", need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GBDT_CUDA(cudaMemsetAsync(w.err, 0, sizeof(int32_t), s));
  routes_from_splits_kernel<<<1, 1024, 0, s>>>(splits, level, max_slots, w.route, next_level);
  count_launches();
  launch_move_rows(bins_in, bins_out, ldb, N, F, g_in, g_out, g_dtype == GBDT_DTYPE_F64 ? 8 : 4, orig_in, orig_out,
                   go_right, level, max_slots, seg_in, w.route, splits, seg_out, leaf_of_row, w.move, w.err, s);
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}
