// Grouping of a level's rows by node, for gbdt_build_histograms on rows in any order.
//
// "Module Design: Training Core" s.6 step 2 builds the histograms of all active
// nodes of a level; s.7 fixes what they hold (count and G per bin), not how the
// rows are visited.  When each row only carries its node id (the per-level
// sample_to_node pass of "New tree builder classes") and the nodes are mixed
// along the rows, a shared-memory histogram per CTA cannot hold every node's
// bins, and a scan that filters by node reads every row once per node group.
// Instead the rows of the built slots are first copied, grouped by slot, into
// a row-block buffer (every column read once, with bulk copies), and the
// histograms are then built from that buffer by the node-contiguous kernel.
// Histogram sums are exact integers, so the order of the rows inside a group
// (set here by shared-memory atomics) does not change any result.
//
// Passes: (1) rows per built slot; (2) each slot's range of the buffer, its
// start rounded up to a row block; (3) one CTA per tile of rows ranks the
// tile's rows by slot, claims each slot's run from a per-slot cursor, and
// writes the gradient and every column of its rows to their runs.
#include <type_traits>

#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kGrpThreads = 256;
constexpr int kGrpTile = 4096;                             // rows per tile (one CTA)
constexpr int kGrpRowsPerThread = kGrpTile / kGrpThreads;  // 16
constexpr int kGrpStages = 4;                              // column copies in flight
constexpr int kGrpMinBlocks = 3;                           // resident CTAs per SM the registers are sized for
constexpr uint32_t kGrpWaitPolls = 1u << 20;

// (1) Rows of every built slot: shared counters per CTA, one global atomic per slot per CTA.
__global__ void __launch_bounds__(kGrpThreads)
    grp_count_kernel(const uint16_t* __restrict__ node, int64_t N, const gbdt_level* __restrict__ level,
                     int32_t max_slots, const uint8_t* __restrict__ build_flag, uint32_t* __restrict__ count,
                     int32_t* __restrict__ err) {
  extern __shared__ uint32_t s_cnt[];  // [max_slots], then the flags as bytes
  uint8_t* s_flag = reinterpret_cast<uint8_t*>(s_cnt + max_slots);
  const int node_begin = level->node_begin;
  int n_slots = level->n_slots;
  if (n_slots > max_slots) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, kErrLevelSize);
    n_slots = max_slots;
  }
  for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
    s_cnt[s] = 0;
    s_flag[s] = build_flag[s];
  }
  __syncthreads();
  auto add = [&](uint32_t id) {
    const int slot = static_cast<int>(id) - node_begin;
    if (slot >= 0 && slot < n_slots && s_flag[slot]) atomicAdd(&s_cnt[slot], 1u);
  };
  const int64_t n8 = N / 8;  // eight node ids per 16-byte load (node_of_row is 16-byte aligned)
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(node) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      add(w[k] & 0xffffu);
      add(w[k] >> 16);
    }
  }
  if (blockIdx.x == 0)
    for (int64_t r = n8 * 8 + threadIdx.x; r < N; r += blockDim.x) add(node[r]);
  __syncthreads();
  for (int s = threadIdx.x; s < n_slots; s += blockDim.x)
    if (s_cnt[s]) atomicAdd(&count[s], s_cnt[s]);
}

// (2) One CTA: each built slot's range of the grouped buffer (start rounded up to a row block, so
// no two slots share a row block), its cursor, and its segment for the histogram pass.
__global__ void __launch_bounds__(1024)
    grp_setup_kernel(const gbdt_level* __restrict__ level, int32_t max_slots, const uint8_t* __restrict__ build_flag,
                     const uint32_t* __restrict__ count, uint32_t* __restrict__ cursor,
                     gbdt_segment* __restrict__ seg) {
  __shared__ long long s_w[33];
  long long pre = 0;  // block-uniform running total
  const int n_slots = min(level->n_slots, max_slots);
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const long long c = (s < n_slots && build_flag[s]) ? count[s] : 0;
    const long long padded = (c + kRowBlock - 1) / kRowBlock * kRowBlock;
    long long tot;
    const long long e = block_scan_excl(padded, s_w, &tot);
    if (s < n_slots) {
      seg[s] = gbdt_segment{pre + e, c};
      cursor[s] = static_cast<uint32_t>(pre + e);
    }
    pre += tot;
  }
}

// (3) One CTA per tile of kGrpTile rows.  Ranks: a row's rank among the tile's rows of its slot comes
// from a shared-memory counter; the tile's output order lists its slots' runs one after another
// (exclusive scan of the counts); each run's place in the buffer is claimed from the slot's cursor.
// Every thread then owns output positions o = threadIdx.x + k * kGrpThreads: it moves the gradient and,
// column by column from the staged copies, the bin byte of the row at o.  Consecutive output positions
// of a run are consecutive bytes of a row block, so a warp's byte stores cover a few sectors.
template <int GS>
__global__ void __launch_bounds__(kGrpThreads, kGrpMinBlocks)
    grp_scatter_kernel(const uint8_t* __restrict__ bins, int64_t ldb, int64_t N, int32_t F,
                       const void* __restrict__ g_in, void* __restrict__ g_out, const uint16_t* __restrict__ node,
                       const gbdt_level* __restrict__ level, int32_t max_slots, const uint8_t* __restrict__ build_flag,
                       uint32_t* __restrict__ cursor, uint8_t* __restrict__ rb, int64_t pitch,
                       int32_t* __restrict__ err) {
  using GW = typename std::conditional<GS == 8, unsigned long long, uint32_t>::type;
  extern __shared__ __align__(128) unsigned char smem[];
  uint8_t(*s_stage)[kGrpTile] = reinterpret_cast<uint8_t(*)[kGrpTile]>(smem);
  uint32_t* s_inv = reinterpret_cast<uint32_t*>(smem + kGrpStages * kGrpTile);  // row | slot << 16
  uint32_t* s_cnt = s_inv + kGrpTile;                                           // [max_slots]
  uint32_t* s_off = s_cnt + max_slots;                                          // [max_slots]
  uint32_t* s_base = s_off + max_slots;                                         // [max_slots]
  uint8_t* s_flag = reinterpret_cast<uint8_t*>(s_base + max_slots);             // [max_slots]
  __shared__ __align__(8) uint64_t s_full[kGrpStages];
  __shared__ uint32_t s_w[33];

  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kGrpTile;
  const int n = static_cast<int>(min(static_cast<int64_t>(kGrpTile), N - p0));
  const uint32_t span = static_cast<uint32_t>((n + 15) & ~15);  // p0 is 16-byte aligned, ldb % 16 == 0
  if (threadIdx.x == 0) {
    for (int k = 0; k < kGrpStages; ++k) mbar_init(&s_full[k], 1);
    mbar_init_fence();
    for (int c = 0; c < F && c < kGrpStages; ++c) bulk_load(s_stage[c], bins + c * ldb + p0, span, &s_full[c]);
  }
  const int node_begin = level->node_begin;
  const int n_slots = min(level->n_slots, max_slots);
  for (int s = threadIdx.x; s < n_slots; s += blockDim.x) {
    s_cnt[s] = 0;
    s_flag[s] = build_flag[s];
  }
  __syncthreads();
  // ---- ranks of the tile's rows within their slots
  uint32_t rk[kGrpRowsPerThread];  // rank | slot << 16, or ~0u for a row that is not grouped
#pragma unroll
  for (int k = 0; k < kGrpRowsPerThread; ++k) {
    const int r = threadIdx.x + k * kGrpThreads;
    rk[k] = ~0u;
    if (r < n) {
      const int slot = static_cast<int>(node[p0 + r]) - node_begin;
      if (slot >= 0 && slot < n_slots && s_flag[slot])
        rk[k] = atomicAdd(&s_cnt[slot], 1u) | (static_cast<uint32_t>(slot) << 16);
    }
  }
  __syncthreads();
  // ---- the tile's runs: exclusive scan of the counts in slot order (consecutive slots per thread)
  const int per = (n_slots + kGrpThreads - 1) / kGrpThreads;
  const int s0 = threadIdx.x * per, s1 = min(n_slots, s0 + per);
  uint32_t mine = 0;
  for (int s = s0; s < s1; ++s) mine += s_cnt[s];
  uint32_t n_out;
  uint32_t off = block_scan_excl(mine, s_w, &n_out);
  for (int s = s0; s < s1; ++s) {
    const uint32_t c = s_cnt[s];
    s_off[s] = off;
    if (c) s_base[s] = atomicAdd(&cursor[s], c);  // this tile's run in the slot's range
    off += c;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kGrpRowsPerThread; ++k) {
    if (rk[k] == ~0u) continue;
    const uint32_t slot = rk[k] >> 16;
    s_inv[s_off[slot] + (rk[k] & 0xffffu)] = static_cast<uint32_t>(threadIdx.x + k * kGrpThreads) | (slot << 16);
  }
  __syncthreads();
  // ---- gradient: each output position's row, read in the tile (cached lines), written to its run
  const GW* gi = static_cast<const GW*>(g_in) + p0;
  GW* go = static_cast<GW*>(g_out);
  for (uint32_t o = threadIdx.x; o < n_out; o += kGrpThreads) {
    const uint32_t e = s_inv[o];
    const uint32_t slot = e >> 16;
    go[s_base[slot] + (o - s_off[slot])] = gi[e & 0xffffu];
  }
  // ---- columns through the stages: a thread owns output positions o = threadIdx.x + k * kGrpThreads and
  // stores each one's byte (a warp's 32 consecutive positions cover one or two runs: a few sectors).  Storing
  // whole aligned words instead (four gathered bytes each) was measured slower: a run holds about 16 rows
  // when 128 nodes share a 4096-row tile, so a warp's words spread over many more sectors than its bytes.
  uint32_t src[kGrpRowsPerThread], dst[kGrpRowsPerThread];
  const int n_own = n_out > threadIdx.x ? static_cast<int>((n_out - 1 - threadIdx.x) / kGrpThreads) + 1 : 0;
#pragma unroll
  for (int k = 0; k < kGrpRowsPerThread; ++k) {
    const uint32_t o = threadIdx.x + k * kGrpThreads;
    src[k] = 0;
    dst[k] = 0;
    if (k < n_own) {
      const uint32_t e = s_inv[o];
      const uint32_t slot = e >> 16;
      src[k] = e & 0xffffu;
      dst[k] = s_base[slot] + (o - s_off[slot]);
    }
  }
  int c_fail = -1;
#pragma unroll 1
  for (int c = 0; c < F; ++c) {
    const int st = c % kGrpStages;
    const bool ok = mbar_wait(&s_full[st], static_cast<uint32_t>((c / kGrpStages) & 1), kGrpWaitPolls);
    if (ok) {
      const uint8_t* stage = s_stage[st];
      uint8_t* out = rb + static_cast<int64_t>(c) * kRowBlock;
#pragma unroll
      for (int k = 0; k < kGrpRowsPerThread; ++k)
        if (k < n_own) out[static_cast<int64_t>(dst[k] >> 5) * pitch + (dst[k] & 31)] = stage[src[k]];
    }
    if (__syncthreads_or(!ok)) {  // every thread is done with this stage (or a copy timed out)
      c_fail = c;
      break;
    }
    if (threadIdx.x == 0 && c + kGrpStages < F)
      bulk_load(s_stage[st], bins + static_cast<int64_t>(c + kGrpStages) * ldb + p0, span, &s_full[st]);
  }
  if (c_fail >= 0 && threadIdx.x == 0) {
    raise_error(err, kErrWaitTimeout);
    // let the copies still in flight land before the CTA's shared memory is released
    const int issued = min(F, c_fail + kGrpStages);
    for (int c = c_fail; c < issued; ++c) {
      if (c + kGrpStages < issued) continue;
      mbar_wait(&s_full[c % kGrpStages], static_cast<uint32_t>((c / kGrpStages) & 1), kGrpWaitPolls);
    }
  }
}

}  // namespace

size_t group_rows_capacity(int64_t N, int32_t max_slots) {
  return static_cast<size_t>(N) + static_cast<size_t>(kRowBlock) * static_cast<size_t>(max_slots);
}

void launch_group_rows(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, const void* g, int g_size,
                       const uint16_t* node, const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag,
                       uint32_t* count, uint32_t* cursor, gbdt_segment* seg, uint8_t* rb, void* g_out,
                       int32_t* err, cudaStream_t s) {
  cudaMemsetAsync(count, 0, sizeof(uint32_t) * max_slots, s);
  const int count_grid = sm_count() * 4;
  grp_count_kernel<<<count_grid, kGrpThreads, static_cast<size_t>(max_slots) * 5, s>>>(node, N, level, max_slots,
                                                                                        build_flag, count, err);
  count_launches();
  grp_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, build_flag, count, cursor, seg);
  count_launches();
  const size_t smem = group_rows_smem_bytes(max_slots);
  const int tiles = ceil_div(N, kGrpTile);
  const int64_t pitch = rb_pitch(F);
  if (g_size == 8) {
    static bool once = (cudaFuncSetAttribute(grp_scatter_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(group_rows_smem_bytes(kMaxSlots))),
                        true);
    (void)once;
    grp_scatter_kernel<8><<<tiles, kGrpThreads, smem, s>>>(bins, ldb, N, F, g, g_out, node, level, max_slots,
                                                           build_flag, cursor, rb, pitch, err);
  } else {
    static bool once = (cudaFuncSetAttribute(grp_scatter_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(group_rows_smem_bytes(kMaxSlots))),
                        true);
    (void)once;
    grp_scatter_kernel<4><<<tiles, kGrpThreads, smem, s>>>(bins, ldb, N, F, g, g_out, node, level, max_slots,
                                                           build_flag, cursor, rb, pitch, err);
  }
  count_launches();
}

size_t group_rows_smem_bytes(int32_t max_slots) {
  return static_cast<size_t>(kGrpStages) * kGrpTile + sizeof(uint32_t) * kGrpTile +
         static_cast<size_t>(max_slots) * (3 * sizeof(uint32_t) + 1);
}

}  // namespace gbdt
