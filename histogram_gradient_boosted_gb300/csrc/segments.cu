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
// The one-level partition is a tile count, a scan over tiles, and a move in
// which each CTA ranks its tile once and then streams several columns through
// shared memory, writing the left and right runs with aligned 16-byte stores.
// The training's pair move (two levels at once, four runs) needs no count or
// scan launch: each tile finds its place by a look-back over its pair's
// earlier tiles.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "rows.cuh"

namespace gbdt {

namespace {

// ---------------------------------------------------------------------------------------- histograms
constexpr int kSegThreads = 768;  // 24 warps: registers for two blocks' loads per warp
constexpr int kSegMaxFeats = 64;  // features per CTA (64 x 256 x 12 B = 192 KB of shared memory)

// The work of a level is cut by cost (kSlotCost, SegWork: kernels.cuh).

// One CTA: compact list of built slots, the prefix of their row counts, and
// how many CTAs per feature group share the work (at most max_ctas, and no
// less than min_rows of cost each).
__global__ void seg_work_setup_kernel(const gbdt_level* __restrict__ level, int32_t max_slots,
                                      const uint8_t* __restrict__ build_flag, const gbdt_segment* __restrict__ seg,
                                      int32_t max_ctas, int64_t min_rows, int32_t* __restrict__ build_slot,
                                      int64_t* __restrict__ row_start /*[max_slots+1]*/, SegWork* __restrict__ st) {
  // (a slot's rows are its segment's positions, narrowed by its filter inside the histogram kernel)
  __shared__ int s_wa[33];
  __shared__ long long s_wb[33];
  int s_pre_slots = 0;        // block-uniform running totals
  long long s_pre_rows = 0;
  const int n_slots = min(level->n_slots, max_slots);
  for (int c0 = 0; c0 < n_slots; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool in = s < n_slots && build_flag[s] && seg[s].count > 0;
    const long long rows = in ? seg[s].count : 0;
    int n_in;
    long long n_rows;
    const int ea = block_scan_excl(in ? 1 : 0, s_wa, &n_in);
    const long long eb = block_scan_excl(rows, s_wb, &n_rows);
    if (in) {
      const int k = s_pre_slots + ea;
      build_slot[k] = s;
      row_start[k] = s_pre_rows + eb;
    }
    s_pre_slots += n_in;
    s_pre_rows += n_rows;
  }
  if (threadIdx.x == 0) {
    row_start[s_pre_slots] = s_pre_rows;
    const long long cost = s_pre_rows + kSlotCost * s_pre_slots;
    st->total_rows = s_pre_rows;
    st->total_cost = cost;
    st->n_built = s_pre_slots;
    const long long by_size = (cost + min_rows - 1) / min_rows;
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
// kCnt false: the counts are known (the root level after the first tree: a row set's counts do not
// depend on the gradients), only the low word is added.
template <uint32_t kLo, bool kCnt = true>
__device__ __forceinline__ uint32_t entry_lo(uint32_t addr, uint32_t ql) {
  uint32_t old;
  if constexpr (kCnt) {
    asm volatile(
        "red.shared.add.u32 [%1], 1;\n\t"
        "atom.shared.add.u32 %0, [%1+%3], %2;"
        : "=r"(old)
        : "r"(addr), "r"(ql), "n"(kLo)
        : "memory");
  } else {
    asm volatile("atom.shared.add.u32 %0, [%1+%2], %3;" : "=r"(old) : "r"(addr), "n"(kLo), "r"(ql) : "memory");
  }
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

// Low word of the H entry (logistic): add and return the old value, like entry_lo's G word.
template <uint32_t kLo>
__device__ __forceinline__ uint32_t atom_lo(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared.add.u32 %0, [%1+%3], %2;" : "=r"(old) : "r"(addr), "r"(v), "n"(kLo) : "memory");
  return old;
}

// Byte k of w times 128 (the byte stride between bins) plus base.
__device__ __forceinline__ uint32_t bin_addr(uint32_t w, int k, uint32_t base) {
  return base + (__byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(k)) << 7);
}

// Rows i and i + 1 of the block, every half: the low-word atomics of all of
// them are issued before the first carry is needed.
template <int NH, bool kFull, bool kCnt>
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
      if (use0) old[0][h] = entry_lo<kLo, kCnt>(a[0][h], qq.x);
      if (use1) old[1][h] = entry_lo<kLo, kCnt>(a[1][h], qq.z);
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      if (use0) entry_hi<kHi>(a[0][h], qq.x, static_cast<int32_t>(qq.y), old[0][h]);
      if (use1) entry_hi<kHi>(a[1][h], qq.z, static_cast<int32_t>(qq.w), old[1][h]);
    }
  }
}

// Partial block (some rows outside the slot or filtered out): only the valid
// rows are visited, a loaded word (four rows) at a time, so a row that does
// not belong to the slot costs a uniform branch.  The low-word atomics of the
// valid rows of each pair of a word's rows are issued before the first carry is
// needed (pairs: a batch of four rows spills registers and runs slower).
constexpr int kSparseBatch = 2;
template <int NH, bool kCnt>
__device__ __forceinline__ void seg_rows_sparse(uint32_t base, const uint32_t (&w)[NH][8], const uint4* s_q,
                                                uint32_t valid) {
  constexpr uint32_t kLo = NH * kHalfBytes, kHi = 2 * NH * kHalfBytes;
  const uint2* s_q2 = reinterpret_cast<const uint2*>(s_q);
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    const uint32_t m = (valid >> (4 * wi)) & 0xfu;  // warp-uniform
    if (m == 0) continue;
#pragma unroll
    for (int k0 = 0; k0 < 4; k0 += kSparseBatch) {
      uint2 q[kSparseBatch];
      uint32_t a[kSparseBatch][NH], old[kSparseBatch][NH];
#pragma unroll
      for (int j = 0; j < kSparseBatch; ++j) {
        const int k = k0 + j;
        if (!(m >> k & 1u)) continue;
        q[j] = s_q2[4 * wi + k];
#pragma unroll
        for (int h = 0; h < NH; ++h) a[j][h] = bin_addr(w[h][wi], k, base + h * kHalfBytes);
#pragma unroll
        for (int h = 0; h < NH; ++h) old[j][h] = entry_lo<kLo, kCnt>(a[j][h], q[j].x);
      }
#pragma unroll
      for (int j = 0; j < kSparseBatch; ++j) {
        if (!(m >> (k0 + j) & 1u)) continue;
#pragma unroll
        for (int h = 0; h < NH; ++h) entry_hi<kHi>(a[j][h], q[j].x, static_cast<int32_t>(q[j].y), old[j][h]);
      }
    }
  }
}

// With H (logistic objective): one group half of up to 32 features, five words per entry (count,
// G low and high, H low and high, one half size apart) and a staged record per row of (G low,
// G high, H low, H high).  Full block: two rows at a time, their four returning atomics first.
constexpr uint32_t kHLo = 3 * kHalfBytes, kHHi = 4 * kHalfBytes;

template <bool kCnt>
__device__ __forceinline__ void seg_rows32_h(uint32_t base, const uint32_t (&w)[8], const uint4* s_q) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint4 q0 = s_q[i], q1 = s_q[i + 1];
    const uint32_t a0 = bin_addr(w[i >> 2], i & 3, base), a1 = bin_addr(w[(i + 1) >> 2], (i + 1) & 3, base);
    const uint32_t og0 = entry_lo<kHalfBytes, kCnt>(a0, q0.x), oh0 = atom_lo<kHLo>(a0, q0.z);
    const uint32_t og1 = entry_lo<kHalfBytes, kCnt>(a1, q1.x), oh1 = atom_lo<kHLo>(a1, q1.z);
    entry_hi<2 * kHalfBytes>(a0, q0.x, static_cast<int32_t>(q0.y), og0);
    entry_hi<kHHi>(a0, q0.z, static_cast<int32_t>(q0.w), oh0);
    entry_hi<2 * kHalfBytes>(a1, q1.x, static_cast<int32_t>(q1.y), og1);
    entry_hi<kHHi>(a1, q1.z, static_cast<int32_t>(q1.w), oh1);
  }
}

// Partial block with H: the valid rows only, as seg_rows_sparse.
template <bool kCnt>
__device__ __forceinline__ void seg_rows_sparse_h(uint32_t base, const uint32_t (&w)[8], const uint4* s_q,
                                                  uint32_t valid) {
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    uint32_t m = (valid >> (4 * wi)) & 0xfu;  // warp-uniform
    while (m != 0) {
      const uint32_t k = __ffs(m) - 1;
      m &= m - 1;
      const uint4 q = s_q[4 * wi + k];
      const uint32_t a = base + (__byte_perm(w[wi], 0u, 0x4440u | k) << 7);
      const uint32_t og = entry_lo<kHalfBytes, kCnt>(a, q.x), oh = atom_lo<kHLo>(a, q.z);
      entry_hi<2 * kHalfBytes>(a, q.x, static_cast<int32_t>(q.y), og);
      entry_hi<kHHi>(a, q.z, static_cast<int32_t>(q.w), oh);
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

// The loads of one 32-position block: the lane's bytes of every half, its row's gradient and, with a
// filter, its row's decision byte.
template <int NH>
struct SegBlock {
  uint32_t w[NH][8];
  double gv;
  int fb;
};

// Issue the loads of block b (positions outside [p0, p1) read nothing).  kRB: bins in the row-block
// layout (ldb is then the row-block pitch and col[h] points at the column's 32 bytes of row block 0).
template <typename GT, int NH, bool kV8, bool kRB>
__device__ __forceinline__ void seg_load_block(SegBlock<NH>& x, int64_t b, const uint8_t* const (&col)[NH],
                                               const bool (&has)[NH], int64_t ldb, const GT* __restrict__ g,
                                               int64_t p0, int64_t p1, const uint8_t* __restrict__ fcol, uint32_t fsh,
                                               uint32_t fmk) {
  const int lane = threadIdx.x & 31;
  const int64_t r0 = b << 5, pr = r0 + lane;
  const bool in = pr >= p0 && pr < p1;
  const bool second = r0 + 16 < p1;  // any row of the block's upper half is in range
  const int64_t boff = kRB ? b * ldb : r0;  // the block's bytes of a column, from col[h]
  x.fb = (fcol && in) ? static_cast<int>((fcol[boff + lane] >> fsh) & fmk) : 0;
  x.gv = in ? static_cast<double>(g[pr]) : 0.0;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    if (has[h]) {
      load_rows32<kV8>(col[h] + boff, second, x.w[h]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x.w[h][k] = 0;
    }
  }
}

// Add the rows at positions [p0, p1) of one slot to the CTA's shared histograms.
// With a filter (fcol != nullptr) only the rows whose decision fcol[p] > fbin
// equals fside are added.
// kH: also the logistic hessian h = |g| (1 - |g|) of each row, in fixed point with scale_h.
// A lane's byte is its slot's code: a feature's bin, or for a 4-bit slot the joint code of its two
// features (first | second << 4), whose histogram the flush splits into the two.  The filter's
// feature may sit in a 4-bit slot: its decision is (byte >> fsh) & fmk.
// A warp takes every n_warps-th block and loads its next block before it counts the current one,
// so the loads' latency is spent on the current block's atomics.
template <typename GT, int NH, bool kV8, bool kRB, bool kH, bool kCnt>
__device__ __forceinline__ void seg_hist_rows(uint32_t base, const uint8_t* const (&col)[NH], const bool (&has)[NH],
                                              int64_t ldb, const GT* __restrict__ g, double scale, double scale_h,
                                              int64_t p0, int64_t p1, const uint8_t* __restrict__ fcol, int fbin,
                                              int fside, uint4* s_q, uint32_t fsh, uint32_t fmk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  // aligned 32-position blocks covering [p0, p1); positions outside are masked
  int64_t b = (p0 >> 5) + warp;
  if ((b << 5) >= p1) return;  // warp-uniform
  SegBlock<NH> cur, nxt;
  seg_load_block<GT, NH, kV8, kRB>(cur, b, col, has, ldb, g, p0, p1, fcol, fsh, fmk);
  while (true) {
    const int64_t bn = b + n_warps;
    const bool more = (bn << 5) < p1;  // warp-uniform
    if (more) seg_load_block<GT, NH, kV8, kRB>(nxt, bn, col, has, ldb, g, p0, p1, fcol, fsh, fmk);
    const int64_t pr = (b << 5) + lane;
    const bool in = pr >= p0 && pr < p1;
    const bool v = in && (!fcol || (cur.fb > fbin) == (fside != 0));
    const uint32_t valid = __ballot_sync(0xffffffffu, v);
    if (valid != 0) {  // warp-uniform: some row of this block belongs to the slot
      const int64_t q = v ? to_fixed(cur.gv, scale) : 0;
      __syncwarp();
      if constexpr (kH) {
        const int64_t qh = v ? to_fixed(logistic_hess(cur.gv), scale_h) : 0;
        s_q[lane] = make_uint4(static_cast<uint32_t>(static_cast<uint64_t>(q)), static_cast<uint32_t>(q >> 32),
                               static_cast<uint32_t>(static_cast<uint64_t>(qh)), static_cast<uint32_t>(qh >> 32));
      } else {
        reinterpret_cast<uint2*>(s_q)[lane] =
            make_uint2(static_cast<uint32_t>(static_cast<uint64_t>(q)), static_cast<uint32_t>(q >> 32));
      }
      __syncwarp();
      if constexpr (kH) {
        if (valid == 0xffffffffu) seg_rows32_h<kCnt>(base, cur.w[0], s_q);
        else seg_rows_sparse_h<kCnt>(base, cur.w[0], s_q, valid);
      } else {
        if (valid == 0xffffffffu) seg_rows32<NH, true, kCnt>(base, cur.w, s_q, valid);
        else seg_rows_sparse<NH, kCnt>(base, cur.w, s_q, valid);
      }
    }
    if (!more) break;
    b = bn;
    cur = nxt;
  }
}

// ---- register histograms (slots of at most kRegMaxCodes codes: a feature with at most 8 bins, or two whose
// bin counts multiply to at most 8, in one 4-bit slot).  A lane's code of a row is (byte & 15) + na *
// (byte >> 4) (na: the first feature's bins; a single feature's byte is below 8, so its code is the byte),
// and the lane keeps each code's count and fixed-point G in registers: no shared atomics, and a flush of
// kCodes entries per lane instead of 256.
template <int kCodes, bool kFull, bool kCnt>
__device__ __forceinline__ void reg_rows32(const uint32_t (&w)[8], const uint2* s_q2, uint32_t valid, int na,
                                           uint32_t (&rc)[kCodes], long long (&rq)[kCodes]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (!kFull && !(valid >> i & 1u)) continue;  // warp-uniform
    const uint2 qq = s_q2[i];
    const long long q = static_cast<long long>((static_cast<unsigned long long>(qq.y) << 32) | qq.x);
    const uint32_t byte = __byte_perm(w[i >> 2], 0u, 0x4440u | static_cast<uint32_t>(i & 3));
    const int code = static_cast<int>(byte & 15u) + na * static_cast<int>(byte >> 4);
#pragma unroll
    for (int c = 0; c < kCodes; ++c) {
      const bool m = code == c;
      if (kCnt) rc[c] += m ? 1u : 0u;
      rq[c] += m ? q : 0ll;
    }
  }
}

// The rows at positions [p0, p1) of one slot added to this lane's registers (a warp takes every n_warps-th
// row block, loading the next before counting the current, as seg_hist_rows); fp64 g, row-block layout.
template <int kCodes, bool kCnt>
__device__ __forceinline__ void seg_reg_rows(const uint8_t* col, bool has, int64_t pitch, const double* __restrict__ g,
                                             double scale, int64_t p0, int64_t p1, const uint8_t* __restrict__ fcol,
                                             int fbin, int fside, uint2* s_q2, uint32_t fsh, uint32_t fmk, int na,
                                             uint32_t (&rc)[kCodes], long long (&rq)[kCodes]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  int64_t b = (p0 >> 5) + warp;
  if ((b << 5) >= p1) return;  // warp-uniform
  const uint8_t* const cols[1] = {col};
  const bool hs[1] = {has};
  SegBlock<1> cur, nxt;
  seg_load_block<double, 1, true, true>(cur, b, cols, hs, pitch, g, p0, p1, fcol, fsh, fmk);
  while (true) {
    const int64_t bn = b + n_warps;
    const bool more = (bn << 5) < p1;  // warp-uniform
    if (more) seg_load_block<double, 1, true, true>(nxt, bn, cols, hs, pitch, g, p0, p1, fcol, fsh, fmk);
    const int64_t pr = (b << 5) + lane;
    const bool in = pr >= p0 && pr < p1;
    const bool v = in && (!fcol || (cur.fb > fbin) == (fside != 0));
    const uint32_t valid = __ballot_sync(0xffffffffu, v);
    if (valid != 0) {
      const int64_t q = v ? to_fixed(cur.gv, scale) : 0;
      __syncwarp();
      s_q2[lane] = make_uint2(static_cast<uint32_t>(static_cast<uint64_t>(q)), static_cast<uint32_t>(q >> 32));
      __syncwarp();
      if (valid == 0xffffffffu) reg_rows32<kCodes, true, kCnt>(cur.w[0], s_q2, valid, na, rc, rq);
      else reg_rows32<kCodes, false, kCnt>(cur.w[0], s_q2, valid, na, rc, rq);
    }
    if (!more) break;
    b = bn;
    cur = nxt;
  }
}

// Merge the CTA's shared histograms into slot's global histograms and leave
// the shared ones zeroed for the next slot.  kH: the H words (s_hlo, s_hhi, the
// two arrays after s_hi) go to hist_h.  Lane j of the group holds column s_lo + j
// of the bins (a slot): src (the slot's features: first | second << 16, second
// 0xffff for a whole-byte slot; null: slot s is feature s) sends a 4-bit slot's
// joint entry to both features' bins.
template <bool kCnt>
__device__ __forceinline__ void flush_add(uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q,
                                          int64_t* __restrict__ hist_h, int64_t o, uint32_t cn, int64_t v,
                                          int64_t vh) {
  if (kCnt) atomicAdd(hist_cnt + o, cn);
  atomicAdd(reinterpret_cast<unsigned long long*>(hist_q + o), static_cast<unsigned long long>(v));
  if (hist_h) atomicAdd(reinterpret_cast<unsigned long long*>(hist_h + o), static_cast<unsigned long long>(vh));
}

template <int NH, bool kH, bool kCnt>
__device__ __forceinline__ void seg_hist_flush(uint32_t* s_cnt, uint32_t* s_lo, int32_t* s_hi, int slot, int32_t F,
                                               int c_lo, int ns, const uint32_t* __restrict__ src,
                                               uint32_t* __restrict__ hist_cnt, int64_t* __restrict__ hist_q,
                                               int64_t* __restrict__ hist_h) {
  constexpr int entries = NH * kHalfWords;
  uint32_t* s_hlo = reinterpret_cast<uint32_t*>(s_hi + entries);
  int32_t* s_hhi = reinterpret_cast<int32_t*>(s_hlo + entries);
  // a thread's entries all sit in one lane (blockDim.x is a multiple of 32): its slot per half
  uint32_t sv[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const int j = (h << 5) + (threadIdx.x & 31);
    const int col = c_lo + (j < ns ? j : 0);
    sv[h] = src ? src[col] : (static_cast<uint32_t>(col) | 0xffff0000u);
  }
  // CTAs that flush the same slot at about the same time (every CTA at the root) start at different
  // entries, so that their global atomics do not queue on the same addresses; the rotation is a
  // multiple of 32, which keeps each entry in its lane
  static_assert((entries & (entries - 1)) == 0, "entries is a power of two");
  const int rot = (static_cast<int>(blockIdx.x) * 32 * 37) & (entries - 1);
  for (int i = threadIdx.x; i < entries; i += blockDim.x) {
    const int e = (i + rot) & (entries - 1);
    const uint32_t cn = s_cnt[e];
    if (kCnt ? cn == 0 : (s_lo[e] | static_cast<uint32_t>(s_hi[e]) |
                          (kH ? s_hlo[e] | static_cast<uint32_t>(s_hhi[e]) : 0u)) == 0u)
      continue;  // nothing to add (without counts: every word of the entry is zero)
    const int hh = e / kHalfWords;
    const int j = (hh << 5) + (e & 31);  // column within the group
    const int64_t v = static_cast<int64_t>(s_hi[e]) * 4294967296ll + static_cast<int64_t>(s_lo[e]);
    s_cnt[e] = 0;
    s_lo[e] = 0;
    s_hi[e] = 0;
    int64_t vh = 0;
    if constexpr (kH) {
      vh = static_cast<int64_t>(s_hhi[e]) * 4294967296ll + static_cast<int64_t>(s_hlo[e]);
      s_hlo[e] = 0;
      s_hhi[e] = 0;
    }
    if (j >= ns) continue;  // unused entries of lanes without a column
    const int code = (e >> 5) & (kBins - 1);
    uint32_t svh = sv[0];
#pragma unroll
    for (int h = 1; h < NH; ++h)
      if (hh == h) svh = sv[h];
    const int64_t fa = static_cast<int64_t>(svh & 0xffffu), fb = static_cast<int64_t>(svh >> 16);
    const int64_t row = static_cast<int64_t>(slot) * F;
    if (fb == 0xffff) {
      flush_add<kCnt>(hist_cnt, hist_q, kH ? hist_h : nullptr, (row + fa) * kBins + code, cn, v, vh);
    } else {  // a 4-bit slot: the joint entry adds to each feature's own bin
      flush_add<kCnt>(hist_cnt, hist_q, kH ? hist_h : nullptr, (row + fa) * kBins + (code & 15), cn, v, vh);
      flush_add<kCnt>(hist_cnt, hist_q, kH ? hist_h : nullptr, (row + fb) * kBins + (code >> 4), cn, v, vh);
    }
  }
}

// One CTA per (share of the level's built rows, feature group): the built
// slots' rows are concatenated in slot order and cut into equal shares, one
// per CTA, so the level runs as one balanced wave.  A share that crosses
// slot boundaries flushes its histograms at each crossing.  kH (logistic):
// also the H histograms, up to 32 features per CTA, fixed_exp[1] their exponent.
// kCnt false: the counts are already in place (copied by the zeroing launch), only G (and H) add.
template <typename GT, bool kV8, bool kRB, bool kH, bool kCnt = true, bool kReg = false>
__global__ void __launch_bounds__(kSegThreads, 1)
    seg_hist_kernel(const uint8_t* __restrict__ bins, int64_t ldb, int32_t F, int32_t S, const GT* __restrict__ g,
                    const int32_t* __restrict__ fixed_exp, const gbdt_segment* __restrict__ seg,
                    const gbdt_filter* __restrict__ filters, const int32_t* __restrict__ build_slot,
                    const int64_t* __restrict__ row_start, const SegWork* __restrict__ st, int32_t group_cols,
                    int32_t sm_budget, int32_t total_weight, int32_t row_weight, uint32_t* __restrict__ hist_cnt,
                    int64_t* __restrict__ hist_q, int64_t* __restrict__ hist_h, const uint32_t* __restrict__ floc,
                    const uint32_t* __restrict__ slot_src, RegGroups rg) {
  extern __shared__ __align__(16) unsigned char smem[];
  // this CTA's group: columns (slots) [c_lo, c_lo + ns) of the bins.  Groups get CTAs in proportion
  // to their 32-lane halves + row_weight: where every scanned row is counted a CTA's time per row is
  // about its halves' atomics (row_weight 0); where a filter skips about half of the scanned rows
  // the row's own work (loads, ballots, the returned values' latency) adds about one half (1).
  // Register groups (rg: slots from rg.reg_begin on, 32 per group) weigh rg.weight.
  const bool reg = static_cast<int>(blockIdx.y) >= rg.n_norm_groups;
  const int c_lo = reg ? rg.reg_begin + (static_cast<int>(blockIdx.y) - rg.n_norm_groups) * 32
                       : static_cast<int>(blockIdx.y) * group_cols;
  const int ns = reg ? min(32, S - c_lo) : min(group_cols, rg.reg_begin - c_lo);
  if (ns <= 0) return;
  const int weight = reg ? rg.weight : ((ns + 31) >> 5) + row_weight;
  const int cap = max(1, static_cast<int>(static_cast<int64_t>(sm_budget) * weight / total_weight));
  const int ctas = min(st->ctas, cap);
  if (static_cast<int>(blockIdx.x) >= ctas) return;
  // this CTA's share [xlo, xhi) of the cost line: built slot j covers [row_start[j] + kSlotCost * j,
  // row_start[j + 1] + kSlotCost * (j + 1)), its rows first, its fixed cost after them
  const int64_t total = st->total_cost;
  const int64_t xlo = total * blockIdx.x / ctas, xhi = total * (blockIdx.x + 1) / ctas;
  if (xlo >= xhi) return;
  const int n_built = st->n_built;
  int k = 0, kh = n_built - 1;  // last built slot whose cost range starts at or before xlo
  while (k < kh) {
    const int mid = (k + kh + 1) >> 1;
    if (row_start[mid] + kSlotCost * mid <= xlo) k = mid;
    else kh = mid - 1;
  }
  const double scale = ldexp(1.0, fixed_exp[0]);
  const double scale_h = kH ? ldexp(1.0, fixed_exp[1]) : 0.0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto run = [&](auto nh_tag) {
    constexpr int NH = decltype(nh_tag)::value;
    constexpr int entries = NH * kHalfWords;
    constexpr int words = kH ? 5 : 3;  // shared words per entry
    constexpr int stage = kH ? 32 : 16;  // uint4 of staged row records per warp
    uint32_t* s_cnt = reinterpret_cast<uint32_t*>(smem);
    uint32_t* s_lo = s_cnt + entries;
    int32_t* s_hi = reinterpret_cast<int32_t*>(s_lo + entries);
    uint4* s_q = reinterpret_cast<uint4*>(s_cnt + words * entries) + warp * stage;
    for (int e = threadIdx.x * 4; e < words * entries; e += blockDim.x * 4)
      *reinterpret_cast<uint4*>(s_cnt + e) = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const uint32_t base = smem_u32(s_cnt) + lane * 4;
    // a lane's column: a slot of the row blocks (one feature, or two in 4 bits each), or in the
    // column layout a feature
    bool has[NH];
    const uint8_t* col[NH];
    const bool unpack = kRB && floc != nullptr;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      has[h] = h * 32 + lane < ns;
      const int c = c_lo + (has[h] ? h * 32 + lane : 0);
      col[h] = bins + static_cast<int64_t>(c) * (kRB ? kRowBlock : ldb);
    }
    for (; k < n_built && row_start[k] + kSlotCost * k < xhi; ++k) {
      // the share's rows of slot k: offsets [o0, o1) of its rows
      const int64_t c0 = row_start[k] + kSlotCost * k, n_k = row_start[k + 1] - row_start[k];
      const int64_t o0 = min(max(xlo - c0, int64_t(0)), n_k), o1 = min(xhi - c0, n_k);
      if (o0 >= o1) continue;  // CTA-uniform: only the slot's fixed cost falls in this share
      const int slot = build_slot[k];
      const int64_t p0 = seg[slot].start + o0;
      const int64_t r = 0, r_end = o1 - o0;
      const gbdt_filter fl = filters ? filters[slot] : gbdt_filter{-1, 0, 0, 0};
      const uint32_t floc_f = fl.feature < 0 ? 0u : unpack ? floc[fl.feature] : static_cast<uint32_t>(fl.feature);
      const uint8_t* fcol =
          fl.feature >= 0 ? bins + static_cast<int64_t>(loc_slot(floc_f)) * (kRB ? kRowBlock : ldb) : nullptr;
      seg_hist_rows<GT, NH, kV8, kRB, kH, kCnt>(base, col, has, ldb, g, scale, scale_h, p0, p0 + (r_end - r), fcol, fl.bin,
                                          fl.side, s_q, loc_shift(floc_f), loc_mask(floc_f));
      __syncthreads();
      seg_hist_flush<NH, kH, kCnt>(s_cnt, s_lo, s_hi, slot, F, c_lo, ns, kRB ? slot_src : nullptr, hist_cnt, hist_q,
                             hist_h);
      __syncthreads();
    }
  };
  if constexpr (kReg && kRB && !kH && std::is_same<GT, double>::value) {  // only launches with register groups
    if (reg) {
      // register groups: per lane kCodes counts and fixed-point sums; per slot a reduction over the warps in
      // shared memory and one global add per (lane, code)
      auto run_reg = [&](auto codes_tag) {
        constexpr int kCodes = decltype(codes_tag)::value;
        constexpr int kW = kSegThreads / 32;
        uint32_t* s_rc = reinterpret_cast<uint32_t*>(smem);                              // [kW][32][kCodes]
        long long* s_rq = reinterpret_cast<long long*>(smem + kW * 32 * kCodes * 4);    // [kW][32][kCodes]
        uint2* s_q2 = reinterpret_cast<uint2*>(smem + kW * 32 * kCodes * 12) + warp * 32;
        const bool has = lane < ns;
        const int c = c_lo + (has ? lane : 0);
        const uint8_t* col = bins + static_cast<int64_t>(c) * kRowBlock;
        const uint32_t sv = slot_src[c];
        const int fa = static_cast<int>(sv & 0xffffu), fb = static_cast<int>(sv >> 16);
        const int na = rg.n_bins[fa];
        for (; k < n_built && row_start[k] + kSlotCost * k < xhi; ++k) {
          const int64_t c0 = row_start[k] + kSlotCost * k, n_k = row_start[k + 1] - row_start[k];
          const int64_t o0 = min(max(xlo - c0, int64_t(0)), n_k), o1 = min(xhi - c0, n_k);
          if (o0 >= o1) continue;  // CTA-uniform
          const int slot = build_slot[k];
          const int64_t p0 = seg[slot].start + o0;
          const gbdt_filter fl = filters ? filters[slot] : gbdt_filter{-1, 0, 0, 0};
          const uint32_t floc_f = fl.feature < 0 ? 0u : floc[fl.feature];
          const uint8_t* fcol = fl.feature >= 0 ? bins + static_cast<int64_t>(loc_slot(floc_f)) * kRowBlock : nullptr;
          uint32_t rc[kCodes];
          long long rq[kCodes];
#pragma unroll
          for (int i = 0; i < kCodes; ++i) rc[i] = 0, rq[i] = 0;
          seg_reg_rows<kCodes, kCnt>(col, has, ldb, reinterpret_cast<const double*>(g), scale, p0, p0 + (o1 - o0),
                                     fcol, fl.bin, fl.side, s_q2, loc_shift(floc_f), loc_mask(floc_f), na, rc, rq);
#pragma unroll
          for (int i = 0; i < kCodes; ++i) {
            s_rc[(warp * 32 + lane) * kCodes + i] = rc[i];
            s_rq[(warp * 32 + lane) * kCodes + i] = rq[i];
          }
          __syncthreads();
          for (int e = threadIdx.x; e < 32 * kCodes; e += blockDim.x) {
            const int l = e / kCodes, code = e % kCodes;
            if (l >= ns) continue;
            uint32_t cn = 0;
            long long v = 0;
            for (int ww = 0; ww < kW; ++ww) {
              cn += s_rc[(ww * 32 + l) * kCodes + code];
              v += s_rq[(ww * 32 + l) * kCodes + code];
            }
            if (kCnt ? cn == 0 : v == 0) continue;
            const uint32_t svl = slot_src[c_lo + l];
            const int la = static_cast<int>(svl & 0xffffu), lb = static_cast<int>(svl >> 16);
            const int nal = rg.n_bins[la];
            const int64_t row = static_cast<int64_t>(slot) * F;
            flush_add<kCnt>(hist_cnt, hist_q, nullptr, (row + la) * kBins + code % nal, cn, v, 0);
            if (lb != 0xffff) flush_add<kCnt>(hist_cnt, hist_q, nullptr, (row + lb) * kBins + code / nal, cn, v, 0);
          }
          __syncthreads();
        }
        (void)fb;
      };
      if (rg.codes <= 4) run_reg(std::integral_constant<int, 4>{});
      else run_reg(std::integral_constant<int, 8>{});
      return;
    }
  }
  if constexpr (kH) {
    run(std::integral_constant<int, 1>{});
  } else {
    if (ns > 32) run(std::integral_constant<int, 2>{});
    else run(std::integral_constant<int, 1>{});
  }
}

// ---------------------------------------------------------------------------------------- partition
constexpr int kMvThreads = 256;
// One CTA: tiles per slot (every slot of the level: split slots are moved,
// the others have their rows recorded as leaves).
__global__ void mv_setup_kernel(const gbdt_level* __restrict__ level, int32_t max_slots,
                                const gbdt_segment* __restrict__ seg, int32_t* __restrict__ tile_start,
                                MvState* __restrict__ st) {
  rows_slot_tiles(level, max_slots, seg, tile_start, st);
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

// Output-centric move.  Once per tile: the rows' decisions (lane = row,
// ballots), their ranks, and the inverse permutation inv[o] = tile position of
// the o-th output row (the rows of each output run in order, the runs one
// after another) in shared memory.  The gradient and the row id move one
// output position per thread, in batches of independent loads.  For the bin
// columns each thread owns up to kMvWordsPerThread aligned 4-byte words of the
// tile's output runs and keeps, in registers, the source positions of their
// bytes; every output word is gathered from the column's tile in shared
// memory and written with one aligned 4-byte store (byte stores only where a
// run starts or ends inside a word), so stores fill whole sectors.  The column
// tiles arrive by bulk asynchronous copies, kMvStages columns ahead of the one
// being gathered, so the loads of later columns overlap the gathers and stores
// of earlier ones.
constexpr int kMvChunks = kMvTile / 32;
constexpr int kMvChunksPerWarp = kMvChunks / (kMvThreads / 32);
constexpr int kMvWordsPerThread = (kMvTile / 4 + 8 + kMvThreads - 1) / kMvThreads;  // 5: up to 4 runs, edges included
constexpr int kMvStages = 4;
// A stage holds a tile's span of one column: in the column layout up to kMvTile + 15 bytes from a
// 16-byte boundary; in the row-block layout kMvBoxBlocks row blocks of 32 bytes (a tile plus its
// offset inside its first row block), the box of one tensor copy.  128-byte aligned stages.
constexpr int kMvBoxBlocks = kMvTile / kRowBlock + 1;
constexpr uint32_t kMvBoxBytes = kMvBoxBlocks * kRowBlock;
constexpr int kMvStageBytes = (kMvBoxBytes + 127) / 128 * 128;
constexpr uint32_t kMvWaitPolls = 1u << 20;

// The output runs of one tile: run r's rows are inv[base[r] .. base[r] + len[r])
// and go to positions dst[r] ...
template <int R>
struct MvRuns {
  int64_t dst[R];
  int len[R];
  int base[R];
};

template <typename T, int R>
__device__ __forceinline__ void move_positions(const T* __restrict__ in, T* __restrict__ out, int64_t p0,
                                               const MvRuns<R>& ru, const uint16_t* s_inv) {
  constexpr int U = 8;
  const int n = ru.base[R - 1] + ru.len[R - 1];
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
      if (o < n) {
        int r = 0;
#pragma unroll
        for (int k = 1; k < R; ++k) r = o >= ru.base[k] ? k : r;
        out[ru.dst[r] + (o - ru.base[r])] = v[u];
      }
    }
  }
}

// Thread 0: arm the stage barriers and start the first column copies: in the
// column layout the tile's 16-byte-aligned span [a0, a0 + span) of each
// column, in the row-block layout the box of row blocks z0 .. of each feature.
template <bool kRB>
__device__ __forceinline__ void mv_start_copies(uint8_t (*s_stage)[kMvStageBytes], uint64_t* s_full,
                                                const uint8_t* __restrict__ bins_in, int64_t ldb, int F, int64_t a0,
                                                uint32_t span, const CUtensorMap* map, int z0) {
  if (threadIdx.x != 0) return;
  for (int k = 0; k < kMvStages; ++k) mbar_init(&s_full[k], 1);
  mbar_init_fence();
  for (int c = 0; c < F && c < kMvStages; ++c) {
    if (kRB) tma_load_3d(s_stage[c], map, 0, c, z0, kMvBoxBytes, &s_full[c]);
    else bulk_load(s_stage[c], bins_in + c * ldb + a0, span, &s_full[c]);
  }
}

// The output words this thread owns: the runs' words listed one run after
// another; off = the word's byte offset from the column's (or in the
// row-block layout the feature's) first byte, -1: none; src = stage positions
// of its four bytes (16 bits each, 0xffff: byte not written).
template <int R, bool kRB>
__device__ __forceinline__ void mv_own_words(const MvRuns<R>& ru, const uint16_t* s_inv, int a_off, int64_t pitch,
                                             int64_t (&off)[kMvWordsPerThread], uint32_t (&srcl)[kMvWordsPerThread],
                                             uint32_t (&srch)[kMvWordsPerThread]) {
  int nw[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    nw[r] = ru.len[r] > 0 ? static_cast<int>(((ru.dst[r] + ru.len[r] + 3) >> 2) - (ru.dst[r] >> 2)) : 0;
#pragma unroll
  for (int m = 0; m < kMvWordsPerThread; ++m) {
    int vw = threadIdx.x + m * kMvThreads;
    uint32_t sp[4] = {0xffffu, 0xffffu, 0xffffu, 0xffffu};
    int64_t w = -1;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (w < 0 && vw >= 0 && vw < nw[r]) {
        const int first = static_cast<int>(ru.dst[r] & 3);  // run start inside its first word
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int o = 4 * vw + i - first;  // offset in the run
          if (o >= 0 && o < ru.len[r]) sp[i] = s_inv[ru.base[r] + o] + a_off;
        }
        w = (ru.dst[r] >> 2) + vw;  // word index
      }
      vw -= nw[r];
    }
    off[m] = w < 0 ? -1 : (kRB ? (w >> 3) * pitch + ((w & 7) << 2) : w << 2);
    srcl[m] = sp[0] | (sp[1] << 16);
    srch[m] = sp[2] | (sp[3] << 16);
  }
}

// The pair move's output words, owned by units: a unit is kMvUnit aligned positions of one grandchild
// run's output (a 32-position unit is one row block of a slot, 8 words; the first and last unit of a
// run may be partial), and the units of the four runs are ordered by the tile position of their first
// row (an exact merge of four lists that are each in that order already, the runs being stable).  A
// warp takes 32 / (kMvUnit / 4) consecutive units, one word per lane, so that the rows a gather
// instruction reads lie close together in the staged column (consecutive units of the merged order
// come from the same stretch of the tile) and spread over more banks than 32 consecutive words of one
// run would.
constexpr int kMvUnit = 32;                        // positions per unit
constexpr int kMvUnitWords = kMvUnit / 4;          // lanes per unit
constexpr int kMvMaxUnits = 32 / kMvUnitWords * kMvThreads / 32 * kMvWordsPerThread;
static_assert(kMvMaxUnits >= kMvTile / kMvUnit + 8, "every unit of a tile has an owner");

// The four runs of a tile in shared memory (read by the unit functions with a run index).
struct MvRunTable {
  long long dst[4];
  int len[4], base[4], a[4], nu[4];  // a: dst % kMvUnit; nu: the run's units
};

// Merge position of every unit: its rank in its own run plus, for each other run, how many of that
// run's units start at an earlier tile position.  mask/cbase: per run and 32-row chunk, the run's
// rows in the chunk and before it.
__device__ __forceinline__ void mv_order_units(const MvRunTable& rt, const uint16_t* s_inv,
                                               const uint32_t (*mask)[kMvChunks], const int (*cbase)[kMvChunks],
                                               uint16_t* s_unit) {
  const int n_units = rt.nu[0] + rt.nu[1] + rt.nu[2] + rt.nu[3];
  for (int k = threadIdx.x; k < n_units; k += blockDim.x) {
    int i = k, q = 0;
    while (i >= rt.nu[q]) i -= rt.nu[q++];                    // unit k of the concatenated runs -> run q, unit i
    const int o_first = i == 0 ? 0 : kMvUnit * i - rt.a[q];  // the unit's first offset in its run
    const int src = s_inv[rt.base[q] + o_first];             // its tile position
    int pos = i;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (r == q || rt.nu[r] == 0) continue;
      const int c = src >> 5;
      const int rows = cbase[r][c] + __popc(mask[r][c] & ((1u << (src & 31)) - 1u));  // run r rows before src
      pos += rows == 0 ? 0 : min(rt.nu[r], (rows + rt.a[r] + kMvUnit - 1) / kMvUnit);
    }
    s_unit[pos] = static_cast<uint16_t>((q << 14) | i);
  }
}

// This thread's words in unit order (off, srcl, srch as mv_own_words; row-block layout).
__device__ __forceinline__ void mv_own_units(const MvRunTable& rt, const uint16_t* s_inv, const uint16_t* s_unit,
                                             int n_units, int a_off, int64_t pitch,
                                             int64_t (&off)[kMvWordsPerThread], uint32_t (&srcl)[kMvWordsPerThread],
                                             uint32_t (&srch)[kMvWordsPerThread]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 0; m < kMvWordsPerThread; ++m) {
    const int k = 32 / kMvUnitWords * (warp + (kMvThreads / 32) * m) + lane / kMvUnitWords;
    uint32_t sp[4] = {0xffffu, 0xffffu, 0xffffu, 0xffffu};
    off[m] = -1;
    if (k < n_units) {
      const int e = s_unit[k], q = e >> 14, u = e & 0x3fff;
      const int64_t dst = rt.dst[q];
      const int len = rt.len[q], base = rt.base[q];
      const int64_t p0 = (dst / kMvUnit + u) * kMvUnit + 4 * (lane % kMvUnitWords);  // the word's first position
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t o = p0 + j - dst;  // offset in the run
        if (o >= 0 && o < len) sp[j] = s_inv[base + o] + a_off;
      }
      if ((sp[0] & sp[1] & sp[2] & sp[3]) != 0xffffu) off[m] = (p0 >> 5) * pitch + (p0 & 31);
    }
    srcl[m] = sp[0] | (sp[1] << 16);
    srch[m] = sp[2] | (sp[3] << 16);
  }
}

// Move every bin column of the tile through the stages.  Returns false when
// a copy did not complete within its wait limit (the error bit is raised and
// the copies still in flight have landed).
template <bool kRB>
__device__ __forceinline__ bool mv_columns(const uint8_t* __restrict__ bins_in, uint8_t* __restrict__ bins_out,
                                           int64_t ldb, int F, int64_t a0, uint32_t span, const CUtensorMap* map,
                                           int z0, uint8_t (*s_stage)[kMvStageBytes], uint64_t* s_full,
                                           const int64_t (&off)[kMvWordsPerThread],
                                           const uint32_t (&srcl)[kMvWordsPerThread],
                                           const uint32_t (&srch)[kMvWordsPerThread], int32_t* err) {
  int c_fail = -1;
#pragma unroll 1
  for (int c = 0; c < F; ++c) {
    const int k = c % kMvStages;
    const uint8_t* stage = s_stage[k];
    const bool ok = mbar_wait(&s_full[k], static_cast<uint32_t>((c / kMvStages) & 1), kMvWaitPolls);
    if (ok) {
      uint8_t* out = bins_out + static_cast<int64_t>(c) * (kRB ? kRowBlock : ldb);
#pragma unroll
      for (int m = 0; m < kMvWordsPerThread; ++m) {
        if (off[m] < 0) continue;
        const uint32_t s0 = srcl[m] & 0xffffu, s1 = srcl[m] >> 16, s2 = srch[m] & 0xffffu, s3 = srch[m] >> 16;
        if (s0 != 0xffffu && s1 != 0xffffu && s2 != 0xffffu && s3 != 0xffffu) {
          *reinterpret_cast<uint32_t*>(out + off[m]) =
              static_cast<uint32_t>(stage[s0]) | (static_cast<uint32_t>(stage[s1]) << 8) |
              (static_cast<uint32_t>(stage[s2]) << 16) | (static_cast<uint32_t>(stage[s3]) << 24);
        } else {  // a run starts or ends inside this word: write only its own bytes
          uint8_t* ob = out + off[m];
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
    if (threadIdx.x == 0 && c + kMvStages < F) {
      if (kRB) tma_load_3d(s_stage[k], map, 0, c + kMvStages, z0, kMvBoxBytes, &s_full[k]);
      else bulk_load(s_stage[k], bins_in + static_cast<int64_t>(c + kMvStages) * ldb + a0, span, &s_full[k]);
    }
  }
  if (c_fail < 0) return true;
  if (threadIdx.x == 0) {
    raise_error(err, kErrWaitTimeout);
    // let the copies still in flight (columns c_fail .. issued - 1) land before the CTA's shared memory is
    // released; each stage completes in order, so waiting for its last issued column suffices
    const int issued = min(F, c_fail + kMvStages);
    for (int c = c_fail; c < issued; ++c) {
      if (c + kMvStages < issued) continue;  // a later column of the same stage is waited for instead
      mbar_wait(&s_full[c % kMvStages], static_cast<uint32_t>((c / kMvStages) & 1), kMvWaitPolls);
    }
  }
  return false;
}

// Move of one level: two runs (left, right) per split slot.
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
  const int64_t a0 = p0 & ~int64_t(15);
  const uint32_t span = static_cast<uint32_t>(((p0 + n + 15) & ~int64_t(15)) - a0);
  const int a_off = static_cast<int>(p0 & 15);  // stage index of tile position 0
  mv_start_copies<false>(s_stage, s_full, bins_in, ldb, F, a0, span, nullptr, 0);
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
  const int64_t left_before = tile_excl[t] - tile_excl[tile_start[s]];
  MvRuns<2> ru;
  ru.dst[0] = seg[s].start + left_before;                             // this tile's left run
  ru.dst[1] = seg[s].start + seg_left[s] + (tile_off - left_before);  // this tile's right run
  ru.len[0] = nl, ru.len[1] = n - nl;
  ru.base[0] = 0, ru.base[1] = nl;
  // ---- gradient and row id, while the first column copies are in flight
  if (g_size == 8)
    move_positions(static_cast<const uint64_t*>(g_in), static_cast<uint64_t*>(g_out), p0, ru, s_inv);
  else
    move_positions(static_cast<const uint32_t*>(g_in), static_cast<uint32_t*>(g_out), p0, ru, s_inv);
  move_positions(orig_in, orig_out, p0, ru, s_inv);
  int64_t wa[kMvWordsPerThread];
  uint32_t srcl[kMvWordsPerThread], srch[kMvWordsPerThread];
  mv_own_words<2, false>(ru, s_inv, a_off, ldb, wa, srcl, srch);
  mv_columns<false>(bins_in, bins_out, ldb, F, a0, span, nullptr, 0, s_stage, s_full, wa, srcl, srch, err);
}

// Last split level: the children are leaves, so nothing moves.  Every row
// records its leaf: the child its split sends it to, or the slot's own node
// when the slot did not split.  With frozen_only, only the slots that did not
// split record their rows (the others are handled at a later level).  Bins in
// the row-block layout (pitch); floc: feature locators (null: feature f in slot f).
__global__ void __launch_bounds__(kMvThreads)
    mv_leaves_kernel(const uint8_t* __restrict__ bins_in, int64_t pitch, const uint32_t* __restrict__ floc,
                     const uint32_t* __restrict__ orig_in, const gbdt_level* __restrict__ level, int32_t max_slots,
                     const gbdt_segment* __restrict__ seg, const Route* __restrict__ route,
                     const int32_t* __restrict__ tile_start, const MvState* __restrict__ st, bool frozen_only,
                     uint16_t* __restrict__ leaf_of_row) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int n_slots = min(level->n_slots, max_slots);
  const int s = slot_of_tile(tile_start, n_slots, t);
  const Route rt = route[s];
  if (frozen_only && rt.feature >= 0) return;
  const int64_t p0 = seg[s].start + static_cast<int64_t>(t - tile_start[s]) * kMvTile;
  const int n = static_cast<int>(min(seg[s].start + seg[s].count - p0, static_cast<int64_t>(kMvTile)));
  if (rt.feature < 0) {
    const uint16_t node = static_cast<uint16_t>(level->node_begin + s);
    for (int i = threadIdx.x; i < n; i += blockDim.x) leaf_of_row[orig_in[p0 + i]] = node;
    return;
  }
  const uint32_t loc = floc ? floc[rt.feature] : static_cast<uint32_t>(rt.feature);
  for (int i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {  // four rows in flight per thread
    int d[4];
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      d[u] = i < n ? rb_bin(bins_in, loc, p0 + i, pitch) : -1;
      o[u] = i < n ? orig_in[p0 + i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (d[u] >= 0) leaf_of_row[o[u]] = static_cast<uint16_t>(rt.left_node + (d[u] > rt.bin ? 1 : 0));
  }
}

// Column layout [F][ldb] -> row-block layout: one thread per (slot, row block) piece of 32 bytes;
// consecutive threads take consecutive row blocks of one slot, so the reads are coalesced and
// every write is one whole 32-byte sector.  Bytes of the last block past N are copied as they are.
// src (null: slot s is feature s) gives each slot's features: first | second << 16, second 0xffff
// for a whole-byte slot; a 4-bit slot's byte is first | second << 4 (both bins below 16).
__device__ __forceinline__ void load_piece(const uint8_t* __restrict__ cols, int64_t ldb, int f, int64_t blk,
                                           uint4& a, uint4& b) {
  const uint8_t* p = cols + static_cast<int64_t>(f) * ldb + blk * kRowBlock;
  a = *reinterpret_cast<const uint4*>(p);  // blk * 32 < N <= ldb, ldb % 16 == 0
  b = blk * kRowBlock + 32 <= ldb ? *reinterpret_cast<const uint4*>(p + 16) : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ uint4 nibbles(uint4 lo, uint4 hi) {
  return make_uint4(lo.x | (hi.x << 4), lo.y | (hi.y << 4), lo.z | (hi.z << 4), lo.w | (hi.w << 4));
}

// Any byte of rows below `rows` (0..32) in the 32-byte piece (a, b) at or above nb (1..256)?
__device__ __forceinline__ bool piece_out_of_range(uint4 a, uint4 b, int rows, int nb) {
  if (nb >= 256) return false;
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const uint32_t lim = static_cast<uint32_t>(nb) * 0x01010101u;
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int v = min(max(rows - 4 * k, 0), 4);  // valid bytes of word k
    const uint32_t keep = v >= 4 ? 0xffffffffu : (1u << (8 * v)) - 1u;
    bad |= (__vcmpgeu4(w[k], lim) & keep) != 0;
  }
  return bad;
}

// n_bins (may be null): every bin of rows below N is checked against its feature's n_bins;
// a bin out of range raises kErrBinRange.
__global__ void cols_to_row_blocks_kernel(const uint8_t* __restrict__ cols, int64_t ldb, int64_t N,
                                          int64_t n_blocks, int32_t S, const uint32_t* __restrict__ src,
                                          const int32_t* __restrict__ n_bins, uint8_t* __restrict__ rb,
                                          int64_t pitch, int32_t* __restrict__ err) {
  const int64_t pieces = n_blocks * S;
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < pieces;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int sl = static_cast<int>(i / n_blocks);
    const int64_t blk = i - static_cast<int64_t>(sl) * n_blocks;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kRowBlock), N - blk * kRowBlock));
    const uint32_t sv = src ? src[sl] : static_cast<uint32_t>(sl) | 0xffff0000u;
    const int fa = static_cast<int>(sv & 0xffffu);
    uint4 a, b;
    load_piece(cols, ldb, fa, blk, a, b);
    if (n_bins) bad |= piece_out_of_range(a, b, rows, n_bins[fa]);
    if ((sv >> 16) != 0xffffu) {
      const int fb = static_cast<int>(sv >> 16);
      uint4 c, d;
      load_piece(cols, ldb, fb, blk, c, d);
      if (n_bins) bad |= piece_out_of_range(c, d, rows, n_bins[fb]);
      a = nibbles(a, c);
      b = nibbles(b, d);
    }
    uint4* dst = reinterpret_cast<uint4*>(rb + blk * pitch + static_cast<int64_t>(sl) * kRowBlock);
    dst[0] = a;
    dst[1] = b;
  }
  if (bad) raise_error(err, kErrBinRange);
}

// ------------------------------------------------------------------------- two levels at once
// At an odd level the rows of each sibling pair still sit, unpartitioned, in
// their parent's segment.  After the level's splits are known they move once,
// straight into the four grandchildren's runs (child 0 left, child 0 right,
// child 1 left, child 1 right); rows of a child that does not split record
// that child as their leaf instead.  The grandchildren's segments are the
// next level's (virtual) segments computed from the split records.

// One CTA: the pair records of a level and the tiles per pair.  level, seg and
// route_cur describe the level (slots in sibling pairs); route_prev and
// pair_parent the level above; seg_next the next level.
__global__ void pair_routes_kernel(const gbdt_level* __restrict__ level, int32_t max_slots,
                                   const gbdt_segment* __restrict__ seg, const Route* __restrict__ route_cur,
                                   const Route* __restrict__ route_prev, const int32_t* __restrict__ pair_parent,
                                   const gbdt_segment* __restrict__ seg_next, const uint32_t* __restrict__ floc,
                                   PairRoute* __restrict__ pairs, int32_t* __restrict__ tile_start,
                                   PairState* __restrict__ st, unsigned long long* __restrict__ tile_status,
                                   int32_t n_status) {
  rows_pair_routes(level, max_slots, seg, route_cur, route_prev, pair_parent, seg_next, floc, pairs, tile_start, st,
                   tile_status, n_status);
}

// Run of position p of pair pr: 0..3, or -1 when its child is a leaf (*child is set either way).
// (bins in the row-block layout).  The parent's decision and both children's
// are loaded together (independent loads), then the child's is selected.
__device__ __forceinline__ int pair_run(const PairRoute& pr, const uint8_t* __restrict__ bins, int64_t pitch,
                                        int64_t p, int* child) {
  const int d1 = rb_bin(bins, static_cast<uint32_t>(pr.f1), p, pitch);
  const int d20 = pr.f2[0] >= 0 ? rb_bin(bins, static_cast<uint32_t>(pr.f2[0]), p, pitch) : 0;
  const int d21 = pr.f2[1] >= 0 ? rb_bin(bins, static_cast<uint32_t>(pr.f2[1]), p, pitch) : 0;
  const int c = d1 > pr.b1 ? 1 : 0;
  *child = c;
  const int f2 = c ? pr.f2[1] : pr.f2[0];
  if (f2 < 0) return -1;
  return 2 * c + ((c ? d21 > pr.b2[1] : d20 > pr.b2[0]) ? 1 : 0);
}

// Threads of the leaf pass (pair_leaves_kernel): a thread per row of a tile and four rows in flight;
// consecutive lanes take consecutive rows, whose row ids (stable moves from the identity) are close
// together, so the leaf writes of a warp fall on few sectors.  (Whole-word decision loads, four rows
// per thread, spread a warp's writes over more sectors and were slower.)
constexpr int kPairLeafThreads = 1024;

// Decoupled look-back over the tiles of one pair (tiles first .. t-1, consecutive CTAs of this launch;
// each waits only for earlier ones).  Warp 0 of tile t: publishes its run counts (status[t] = AGG |
// counts, 13 bits each), sums the counts of the tiles before it - from the nearest tile that has
// published its inclusive prefix (incl[], status PREFIX) or from the pair's first tile - into
// s_pref, then publishes its own inclusive prefix.  status[] is zeroed with the pair records (rows_pair_routes).  Every wait
// is bounded: a tile that gives up raises kErrWaitTimeout (its prefix is then incomplete; the writes
// stay clamped to the runs' records).  The pair's last tile checks the four totals against the split
// records (kErrPartitionCount).
constexpr unsigned long long kTileAgg = 1ull << 62, kTilePrefix = 2ull << 62;

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

struct Want4 {
  long long v[4];  // each grandchild's rows from the split records (-1: its child does not split)
};

__device__ __forceinline__ void mv_tile_prefix(int t, int first, int end, int4 len4, Want4 want,
                                               unsigned long long* __restrict__ status, int4* __restrict__ incl,
                                               long long* s_pref, int32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int len[4] = {len4.x, len4.y, len4.z, len4.w};
  const unsigned long long agg = static_cast<unsigned long long>(len[0]) |
                                 static_cast<unsigned long long>(len[1]) << 13 |
                                 static_cast<unsigned long long>(len[2]) << 26 |
                                 static_cast<unsigned long long>(len[3]) << 39;
  if (lane == 0) st_release_u64(&status[t], kTileAgg | agg);
  long long pref[4] = {0, 0, 0, 0};
  bool gave_up = false;
  for (int top = t - 1; top >= first; top -= 32) {  // window of predecessors top, top - 1, ...
    const int p = top - lane;
    unsigned long long v = 0;
    if (p >= first) {
      for (uint32_t i = 0; i < kMvWaitPolls; ++i) {
        v = ld_acquire_u64(&status[p]);
        if (v >> 62) break;
      }
      if (!(v >> 62)) gave_up = true;
    }
    const uint32_t has_prefix = __ballot_sync(0xffffffffu, p >= first && (v >> 62) == 2);
    const int stop = has_prefix ? __ffs(has_prefix) - 1 : 32;  // the nearest predecessor with a prefix
    long long c[4] = {0, 0, 0, 0};
    if (p >= first && lane < stop) {
      c[0] = v & 0x1fff, c[1] = (v >> 13) & 0x1fff, c[2] = (v >> 26) & 0x1fff, c[3] = (v >> 39) & 0x1fff;
    } else if (lane == stop) {
      const int4 x = incl[p];  // written before its PREFIX status (acquired above)
      c[0] = x.x, c[1] = x.y, c[2] = x.z, c[3] = x.w;
    }
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int q = 0; q < 4; ++q) c[q] += __shfl_xor_sync(0xffffffffu, c[q], o);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) pref[q] += c[q];
    if (stop < 32) break;
  }
  if (__any_sync(0xffffffffu, gave_up) && lane == 0) raise_error(err, kErrWaitTimeout);
  if (lane == 0) {
    incl[t] = make_int4(static_cast<int>(pref[0] + len[0]), static_cast<int>(pref[1] + len[1]),
                        static_cast<int>(pref[2] + len[2]), static_cast<int>(pref[3] + len[3]));
    __threadfence();
    st_release_u64(&status[t], kTilePrefix | agg);
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long tot = pref[q] + len[q];
      if (want.v[q] < 0 ? len[q] != 0 : (tot > want.v[q] || (t == end - 1 && tot != want.v[q]))) bad = true;
    }
    if (bad) raise_error(err, kErrPartitionCount);
  }
  if (lane < 4) s_pref[lane] = pref[lane];
}

__global__ void __launch_bounds__(kMvThreads, 5)
    pair_move_kernel(const __grid_constant__ CUtensorMap map_in, uint8_t* __restrict__ bins_out, int64_t pitch,
                     const uint8_t* __restrict__ bins_in, int32_t F,
                     const uint64_t* __restrict__ g_in, uint64_t* __restrict__ g_out,
                     const uint32_t* __restrict__ orig_in, uint32_t* __restrict__ orig_out,
                     const PairRoute* __restrict__ pairs, const int32_t* __restrict__ tile_start,
                     const PairState* __restrict__ st, unsigned long long* __restrict__ status,
                     int4* __restrict__ incl, uint16_t* __restrict__ leaf_of_row, int32_t* __restrict__ err) {
  __shared__ uint32_t s_mask[4][kMvChunks];  // per run, per 32-row chunk: rows of the run
  __shared__ int s_cbase[4][kMvChunks];      // per run, per chunk: the run's rows before the chunk
  __shared__ uint16_t s_inv[kMvTile];
  __shared__ __align__(128) uint8_t s_stage[kMvStages][kMvStageBytes];
  __shared__ __align__(8) uint64_t s_full[kMvStages];
  __shared__ int s_wtot[kMvThreads / 32][4];
  __shared__ uint16_t s_unit[kMvMaxUnits];
  __shared__ MvRunTable s_rt;
  __shared__ long long s_pref[4];
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  // Every tile of the launch publishes its run counts (see mv_tile_prefix), so none returns early; a
  // run whose rows disagree with its split record is clamped to the record's range and the error
  // raised, so no write leaves the grandchild's range.
  const int k = slot_of_tile(tile_start, st->n_pairs, t);
  const PairRoute pr = pairs[k];
  const int64_t tile_off = static_cast<int64_t>(t - tile_start[k]) * kMvTile;
  const int64_t p0 = pr.start + tile_off;
  const int n = static_cast<int>(min(pr.start + pr.count - p0, static_cast<int64_t>(kMvTile)));
  const int z0 = static_cast<int>(p0 >> 5);     // first row block of the tile
  const int a_off = static_cast<int>(p0 & 31);  // stage index of tile position 0
  mv_start_copies<true>(s_stage, s_full, bins_in, 0, F, 0, 0, &map_in, z0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // ---- rank the tile (lane = row) into four runs; rows of a leaf child record their leaf
  static_assert(kMvChunksPerWarp % 4 == 0, "chunks are ranked four at a time");
#pragma unroll 1
  for (int k0 = 0; k0 < kMvChunksPerWarp; k0 += 4) {
    int r[4], child[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // four chunks' decisions in flight
      const int j = (warp * kMvChunksPerWarp + k0 + u) * 32 + lane;
      r[u] = j < n ? pair_run(pr, bins_in, pitch, p0 + j, &child[u]) : -2;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ch = warp * kMvChunksPerWarp + k0 + u;
      const int j = ch * 32 + lane;
      if (r[u] == -1 && leaf_of_row)
        leaf_of_row[orig_in[p0 + j]] = static_cast<uint16_t>(child[u] ? pr.node[1] : pr.node[0]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t m = __ballot_sync(0xffffffffu, r[u] == q);
        if (lane == 0) s_mask[q][ch] = m;
      }
    }
  }
  __syncthreads();
  // each run's rows before each chunk: the four exclusive scans over the chunks in one pass (a warp
  // per 32 chunks: shuffles; then the warps' totals)
  int len[4];
  {
    int c[4], e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      c[q] = threadIdx.x < kMvChunks ? __popc(s_mask[q][threadIdx.x]) : 0;
      e[q] = c[q];
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, e[q], o);
        if (lane >= o) e[q] += v;
      }
    }
    if (lane == 31) {
#pragma unroll
      for (int q = 0; q < 4; ++q) s_wtot[warp][q] = e[q];
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int before = 0, all = 0;
      for (int w = 0; w < kMvThreads / 32; ++w) {
        const int v = s_wtot[w][q];
        before += w < warp ? v : 0;
        all += v;
      }
      len[q] = all;
      if (threadIdx.x < kMvChunks) s_cbase[q][threadIdx.x] = before + e[q] - c[q];
    }
  }
  __syncthreads();
  if (warp == 0)
    mv_tile_prefix(t, tile_start[k], tile_start[k + 1], make_int4(len[0], len[1], len[2], len[3]),
                   Want4{{pr.want[0], pr.want[1], pr.want[2], pr.want[3]}},
                   status, incl, s_pref, err);
  __syncthreads();
  MvRuns<4> ru;
  int lim[4];  // rows of each run this tile may write: clamped to the run's record
  int acc = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const long long pref = s_pref[q];
    ru.dst[q] = pr.dst[q] + pref;
    ru.len[q] = len[q];
    ru.base[q] = acc;
    acc += len[q];
    const long long room = pr.want[q] < 0 ? 0 : pr.want[q] - pref;
    lim[q] = static_cast<int>(room < 0 ? 0 : (room < len[q] ? room : len[q]));
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      s_rt.dst[q] = ru.dst[q];
      s_rt.len[q] = lim[q];
      s_rt.base[q] = ru.base[q];
      s_rt.a[q] = static_cast<int>(ru.dst[q] % kMvUnit);
      s_rt.nu[q] = lim[q] > 0 ? (s_rt.a[q] + lim[q] + kMvUnit - 1) / kMvUnit : 0;
    }
  }
  // ---- the inverse permutation; the gradient and the row id of every moved row go straight to its
  // output position (read in the tile's order, one coalesced load per chunk, written to at most four
  // runs), four chunks' loads in flight, while the first column copies are in flight
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll 1
  for (int k0 = 0; k0 < kMvChunksPerWarp; k0 += 4) {
    uint64_t gv[4];
    uint32_t ov[4];
    int64_t dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int ch = warp * kMvChunksPerWarp + k0 + u;
      dst[u] = -1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t m = s_mask[q][ch];
        if (m >> lane & 1u) {
          const int o = s_cbase[q][ch] + __popc(m & lt);  // the row's rank in its run
          s_inv[ru.base[q] + o] = static_cast<uint16_t>(ch * 32 + lane);
          if (o < lim[q]) dst[u] = ru.dst[q] + o;
        }
      }
      if (dst[u] >= 0) {
        gv[u] = g_in[p0 + ch * 32 + lane];
        ov[u] = orig_in[p0 + ch * 32 + lane];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (dst[u] >= 0) {
        g_out[dst[u]] = gv[u];
        orig_out[dst[u]] = ov[u];
      }
    }
  }
  __syncthreads();
  mv_order_units(s_rt, s_inv, s_mask, s_cbase, s_unit);
  __syncthreads();
  const int n_units = s_rt.nu[0] + s_rt.nu[1] + s_rt.nu[2] + s_rt.nu[3];
  int64_t wa[kMvWordsPerThread];
  uint32_t srcl[kMvWordsPerThread], srch[kMvWordsPerThread];
  mv_own_units(s_rt, s_inv, s_unit, n_units, a_off, pitch, wa, srcl, srch);
  mv_columns<true>(bins_in, bins_out, pitch, F, 0, 0, &map_in, z0, s_stage, s_full, wa, srcl, srch, err);
}

// Last split level when it is an odd level: every row of a pair records its
// leaf (a grandchild when its child splits, else the child), nothing moves.
__global__ void __launch_bounds__(kPairLeafThreads)
    pair_leaves_kernel(const uint8_t* __restrict__ bins_in, int64_t pitch, const uint32_t* __restrict__ orig_in,
                       const PairRoute* __restrict__ pairs, const int32_t* __restrict__ tile_start,
                       const PairState* __restrict__ st, uint16_t* __restrict__ leaf_of_row) {
  const int t = blockIdx.x;
  if (t >= st->total_tiles) return;
  const int k = slot_of_tile(tile_start, st->n_pairs, t);
  const PairRoute pr = pairs[k];
  const int64_t p0 = pr.start + static_cast<int64_t>(t - tile_start[k]) * kMvTile;
  const int n = static_cast<int>(min(pr.start + pr.count - p0, static_cast<int64_t>(kMvTile)));
  for (int i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {  // four rows in flight per thread
    int r[4], ch[4];
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      r[u] = i < n ? pair_run(pr, bins_in, pitch, p0 + i, &ch[u]) : -2;
      o[u] = i < n ? orig_in[p0 + i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (r[u] == -2) continue;
      const int node = ch[u] ? pr.node[1] : pr.node[0], left = ch[u] ? pr.left[1] : pr.left[0];
      leaf_of_row[o[u]] = static_cast<uint16_t>(r[u] < 0 ? node : left + (r[u] & 1));
    }
  }
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
SegHistPlan plan_seg_histograms(int64_t N, int32_t S, int32_t max_slots, int32_t max_build, bool with_h,
                                bool filtered, int32_t reg_begin, int32_t reg_codes) {
  (void)N, (void)max_slots, (void)max_build;
  SegHistPlan p{};
  const int max_feats = with_h ? 32 : kSegMaxFeats;  // five shared words per entry with H, three without
  const int Sn = (reg_begin >= 0 && !with_h) ? reg_begin : S;  // ordinary slots
  // groups of whole 32-lane halves (an atomic instruction costs the same with idle lanes): full
  // groups of max_feats columns and the remainder; then register groups of 32 slots
  p.n_cols = S;
  p.n_norm_groups = Sn > 0 ? ceil_div(Sn, max_feats) : 0;
  p.group_feats = p.n_norm_groups == 1 ? Sn : max_feats;
  const int rem = Sn - (p.n_norm_groups - 1) * p.group_feats;
  const int n_reg = Sn < S ? ceil_div(S - Sn, 32) : 0;
  p.reg_begin = Sn;
  p.reg_codes = reg_codes <= 4 ? 4 : kRegMaxCodes;
  p.n_fgroups = p.n_norm_groups + n_reg;
  // a group's weight: its halves + row_weight (see seg_hist_kernel; measured on the 10M x 100 levels,
  // 64 + 26 slots: 2 : 1 fastest where every scanned row counts, 3 : 2 at the filtered levels); a register
  // group weighs as much as one half
  p.row_weight = filtered ? 1 : 0;
  p.reg_weight = 1 + p.row_weight;
  p.total_weight = n_reg * p.reg_weight;
  if (p.n_norm_groups > 0)
    p.total_weight += (p.n_norm_groups - 1) * (ceil_div(p.group_feats, 32) + p.row_weight) + ceil_div(rem, 32) +
                      p.row_weight;
  p.sm_budget = sm_count();  // one wave: a CTA per SM, shared by the groups in proportion to their weights
  const int full_weight = p.n_norm_groups > 0 ? ceil_div(p.group_feats, 32) + p.row_weight : p.reg_weight;
  p.max_ctas = std::max(1, static_cast<int>(static_cast<int64_t>(p.sm_budget) * full_weight / p.total_weight));
  p.min_rows = 1024;  // least cost (rows + kSlotCost per slot) per CTA
  p.with_h = with_h;
  const size_t words = with_h ? 5 : 3, stage = with_h ? 512 : 256;  // staged row records per warp
  p.smem = p.n_norm_groups > 0
               ? static_cast<size_t>(ceil_div(p.group_feats, 32)) * kHalfWords * 4 * words + (kSegThreads / 32) * stage
               : 0;
  if (n_reg > 0)  // per warp and lane each code's count and sum, then the staged row records
    p.smem = std::max(p.smem, static_cast<size_t>(kSegThreads / 32) * 32 * p.reg_codes * 12 + (kSegThreads / 32) * 256);
  return p;
}

size_t seg_hist_scratch_bytes(int32_t max_slots) {
  return sizeof(SegWork) + sizeof(int32_t) * (static_cast<size_t>(max_slots) + 1) +
         sizeof(int64_t) * (static_cast<size_t>(max_slots) + 1) + 3 * kWsAlign;
}

SegWorkView seg_work_view(void* scratch, int32_t max_slots) {
  Carve c(scratch, seg_hist_scratch_bytes(max_slots));
  SegWorkView v;
  v.st = c.take<SegWork>(1);
  v.build_slot = c.take<int32_t>(max_slots + 1);
  v.row_start = c.take<int64_t>(max_slots + 1);
  return v;
}

int launch_seg_histograms(const SegHistPlan& plan, const uint8_t* bins, int64_t ldb, int64_t N, int32_t F,
                          const void* g, int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                          int32_t max_slots, const uint8_t* build_flag, const gbdt_segment* seg,
                          const gbdt_filter* filters, void* scratch, uint32_t* hist_cnt, int64_t* hist_q,
                          int64_t* hist_h, cudaStream_t s, bool row_blocks, const uint32_t* floc,
                          const uint32_t* slot_src, const uint32_t* root_cnt, const int32_t* n_bins,
                          bool work_ready) {
  (void)N;
  if (root_cnt && !(row_blocks && g_dtype == GBDT_DTYPE_F64 && max_slots == 1)) {
    set_error("known root counts need the row-block layout, fp64 gradients and a one-slot level");
    return GBDT_ERR_INTERNAL;
  }
  if (plan.reg_begin < plan.n_cols && !(row_blocks && g_dtype == GBDT_DTYPE_F64 && !plan.with_h && n_bins && slot_src)) {
    set_error("register histograms need the row-block layout, fp64 gradients, squared error, n_bins and slot sources");
    return GBDT_ERR_INTERNAL;
  }
  const SegWorkView wv = seg_work_view(scratch, max_slots);
  SegWork* st = wv.st;
  int32_t* build_slot = wv.build_slot;
  int64_t* row_start = wv.row_start;
  if (work_ready)  // the work list (written by the level above) names the built slots: at most half the
                   // slots past the root, one of each sibling pair
    launch_hist_zero_built(st, build_slot, max_slots > 1 ? max_slots / 2 : 1, F, hist_cnt, hist_q,
                           plan.with_h ? hist_h : nullptr, s, root_cnt, n_bins);
  else
    launch_hist_zero(level, max_slots, build_flag, F, hist_cnt, hist_q, plan.with_h ? hist_h : nullptr, s, root_cnt,
                     n_bins);
  if (!work_ready) {  // else the work list is already in the scratch (written by the level above)
    seg_work_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, build_flag, seg, plan.max_ctas, plan.min_rows,
                                             build_slot, row_start, st);
    count_launches();
  }
  dim3 grid(static_cast<unsigned>(plan.max_ctas), static_cast<unsigned>(plan.n_fgroups));
  // 256-bit column loads need every column start 32-byte aligned
  const bool v8 = aligned(bins, 32) && ldb % 32 == 0;
  auto launch = [&](auto kernel, const auto* gp) -> int {
    GBDT_CUDA(smem_attr(kernel, plan.smem));
    const RegGroups rg{plan.reg_begin, plan.n_norm_groups, plan.reg_weight, plan.reg_codes, n_bins};
    kernel<<<grid, kSegThreads, plan.smem, s>>>(bins, ldb, F, plan.n_cols, gp, fixed_exp, seg, filters, build_slot,
                                                row_start, st, plan.group_feats, plan.sm_budget, plan.total_weight,
                                                plan.row_weight,
                                                hist_cnt, hist_q, hist_h, row_blocks ? floc : nullptr,
                                                row_blocks ? slot_src : nullptr, rg);
    return GBDT_OK;
  };
  auto pick = [&](const auto* gp, auto h_tag) -> int {
    using GT = std::remove_const_t<std::remove_pointer_t<decltype(gp)>>;
    constexpr bool kH = decltype(h_tag)::value;
    return row_blocks ? launch(seg_hist_kernel<GT, true, true, kH>, gp)
           : v8       ? launch(seg_hist_kernel<GT, true, false, kH>, gp)
                      : launch(seg_hist_kernel<GT, false, false, kH>, gp);
  };
  int rc;
  if (plan.reg_begin < plan.n_cols) {  // register groups (row blocks, fp64 g, squared error: checked above)
    const double* gp = static_cast<const double*>(g);
    rc = root_cnt ? launch(seg_hist_kernel<double, true, true, false, false, true>, gp)
                  : launch(seg_hist_kernel<double, true, true, false, true, true>, gp);
  } else if (root_cnt) {  // the root's counts are known: G (and H) only
    const double* gp = static_cast<const double*>(g);
    rc = plan.with_h ? launch(seg_hist_kernel<double, true, true, true, false>, gp)
                     : launch(seg_hist_kernel<double, true, true, false, false>, gp);
  } else if (g_dtype == GBDT_DTYPE_F32) {
    const float* gp = static_cast<const float*>(g);
    rc = plan.with_h ? pick(gp, std::true_type{}) : pick(gp, std::false_type{});
  } else {
    const double* gp = static_cast<const double*>(g);
    rc = plan.with_h ? pick(gp, std::true_type{}) : pick(gp, std::false_type{});
  }
  if (rc != GBDT_OK) return rc;
  count_launches();
  return GBDT_OK;
}

namespace {
size_t two_way_scratch_bytes(int64_t N, int32_t max_slots) {
  const size_t tiles = static_cast<size_t>(ceil_div(N, kMvTile)) + max_slots;
  return sizeof(MvState) + sizeof(int32_t) * (max_slots + 1) + sizeof(int32_t) * tiles +
         sizeof(int64_t) * (tiles + 1) + sizeof(int64_t) * max_slots + 6 * kWsAlign;
}

size_t pair_scratch_bytes(int64_t N, int32_t max_slots) {
  const size_t pairs = static_cast<size_t>(max_slots) / 2 + 1;
  const size_t tiles = static_cast<size_t>(ceil_div(N, kMvTile)) + pairs;
  return sizeof(PairState) + sizeof(PairRoute) * pairs + sizeof(int32_t) * (pairs + 1) + sizeof(int4) * tiles +
         sizeof(unsigned long long) * tiles + 6 * kWsAlign;
}

struct PairScratch {
  PairState* st;
  PairRoute* pairs;
  int32_t* tile_start;
  int4* tile_cnt;  // per tile: its runs' inclusive prefix within its pair (the look-back)
  unsigned long long* tile_status;
  int max_tiles;
};

PairScratch carve_pairs(void* scratch, int64_t N, int32_t max_slots) {
  Carve c(scratch, pair_scratch_bytes(N, max_slots));
  PairScratch p;
  const int pairs = max_slots / 2 + 1;
  p.max_tiles = ceil_div(N, kMvTile) + pairs;
  p.st = c.take<PairState>(1);
  p.pairs = c.take<PairRoute>(pairs);
  p.tile_start = c.take<int32_t>(pairs + 1);
  p.tile_cnt = c.take<int4>(p.max_tiles);
  p.tile_status = c.take<unsigned long long>(p.max_tiles);
  return p;
}
}  // namespace

RowsSetup rows_setup_slot_tiles(void* scratch, int64_t N, int32_t max_slots) {
  Carve c(scratch, two_way_scratch_bytes(N, max_slots));  // as launch_leaf_rows carves it
  RowsSetup r{};
  r.kind = kRowsSlotTiles;
  r.mv_st = c.take<MvState>(1);
  r.mv_tile_start = c.take<int32_t>(max_slots + 1);
  return r;
}

RowsSetup rows_setup_pairs(void* scratch, int64_t N, int32_t max_slots, bool move, const Route* route_prev,
                           const int32_t* pair_parent, const uint32_t* floc) {
  const PairScratch p = carve_pairs(scratch, N, max_slots);  // as launch_move_pairs / launch_leaf_pairs carve it
  RowsSetup r{};
  r.kind = kRowsPairRoutes;
  r.pairs = p.pairs;
  r.pair_tile_start = p.tile_start;
  r.pair_st = p.st;
  r.tile_status = move ? p.tile_status : nullptr;
  r.n_status = move ? p.max_tiles : 0;
  r.route_prev = route_prev;
  r.pair_parent = pair_parent;
  r.floc = floc;
  return r;
}

size_t move_scratch_bytes(int64_t N, int32_t max_slots) {
  const size_t a = two_way_scratch_bytes(N, max_slots), b = pair_scratch_bytes(N, max_slots);
  return a > b ? a : b;
}

void launch_move_rows(const uint8_t* bins_in, uint8_t* bins_out, int64_t ldb, int64_t N, int32_t F,
                      const void* g_in, void* g_out, int g_size, const uint32_t* orig_in, uint32_t* orig_out,
                      const uint8_t* go_right, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, const gbdt_split* splits, gbdt_segment* seg_out,
                      uint16_t* leaf_of_row, void* scratch, int32_t* err, cudaStream_t s) {
  Carve c(scratch, two_way_scratch_bytes(N, max_slots));
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
                                                  go_right, level, max_slots, seg, route, tile_start, st, tile_excl,
                                                  seg_left, leaf_of_row, err);
  count_launches();
}

void launch_leaf_rows(const uint8_t* bins_rb, int64_t pitch, const uint32_t* floc, int64_t N,
                      const uint32_t* orig_in, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                      const Route* route, bool frozen_only, uint16_t* leaf_of_row, void* scratch, cudaStream_t s,
                      bool setup_done) {
  Carve c(scratch, two_way_scratch_bytes(N, max_slots));
  MvState* st = c.take<MvState>(1);
  int32_t* tile_start = c.take<int32_t>(max_slots + 1);
  const int max_tiles = ceil_div(N, kMvTile) + max_slots;
  if (!setup_done) {  // else rows_setup_slot_tiles' setup was done by the kernel before
    mv_setup_kernel<<<1, 1024, 0, s>>>(level, max_slots, seg, tile_start, st);
    count_launches();
  }
  mv_leaves_kernel<<<max_tiles, kMvThreads, 0, s>>>(bins_rb, pitch, floc, orig_in, level, max_slots, seg, route,
                                                    tile_start, st, frozen_only, leaf_of_row);
  count_launches();
}

void launch_move_pairs(const CUtensorMap& map_in, const uint8_t* bins_rb_in, uint8_t* bins_rb_out, int64_t pitch,
                       const uint32_t* floc, int64_t N, int32_t S, const double* g_in, double* g_out,
                       const uint32_t* orig_in, uint32_t* orig_out, const gbdt_level* level, int32_t max_slots,
                       const gbdt_segment* seg, const Route* route_cur, const Route* route_prev,
                       const int32_t* pair_parent, const gbdt_segment* seg_next, uint16_t* leaf_of_row, void* scratch,
                       int32_t* err, cudaStream_t s, bool setup_done) {
  const PairScratch p = carve_pairs(scratch, N, max_slots);
  if (!setup_done) {  // else rows_setup_pairs' setup (move true) was done by the kernel before
    pair_routes_kernel<<<1, 1024, 0, s>>>(level, max_slots, seg, route_cur, route_prev, pair_parent, seg_next, floc,
                                          p.pairs, p.tile_start, p.st, p.tile_status, p.max_tiles);
    count_launches();
  }
  pair_move_kernel<<<p.max_tiles, kMvThreads, 0, s>>>(
      map_in, bins_rb_out, pitch, bins_rb_in, S, reinterpret_cast<const uint64_t*>(g_in),
      reinterpret_cast<uint64_t*>(g_out), orig_in, orig_out, p.pairs, p.tile_start, p.st, p.tile_status, p.tile_cnt,
      leaf_of_row, err);
  count_launches();
}

void launch_leaf_pairs(const uint8_t* bins_rb, int64_t pitch, const uint32_t* floc, int64_t N,
                       const uint32_t* orig_in, const gbdt_level* level, int32_t max_slots, const gbdt_segment* seg,
                       const Route* route_cur, const Route* route_prev, const int32_t* pair_parent,
                       const gbdt_segment* seg_next, uint16_t* leaf_of_row, void* scratch, cudaStream_t s,
                       bool setup_done) {
  const PairScratch p = carve_pairs(scratch, N, max_slots);
  if (!setup_done) {  // else rows_setup_pairs' setup (move false) was done by the kernel before
    pair_routes_kernel<<<1, 1024, 0, s>>>(level, max_slots, seg, route_cur, route_prev, pair_parent, seg_next, floc,
                                          p.pairs, p.tile_start, p.st, nullptr, 0);
    count_launches();
  }
  pair_leaves_kernel<<<p.max_tiles, kPairLeafThreads, 0, s>>>(bins_rb, pitch, orig_in, p.pairs, p.tile_start,
                                                               p.st, leaf_of_row);
  count_launches();
}

size_t row_block_bytes(int64_t N, int32_t S) { return static_cast<size_t>(rb_blocks(N)) * rb_pitch(S); }

void launch_cols_to_row_blocks(const uint8_t* cols, int64_t ldb, int64_t N, int32_t S, const uint32_t* slot_src,
                               const int32_t* n_bins, uint8_t* rb, int32_t* err, cudaStream_t s) {
  const int64_t pieces = rb_blocks(N) * S;
  const int grid = static_cast<int>(std::min<int64_t>((pieces + 255) / 256, static_cast<int64_t>(sm_count()) * 16));
  cols_to_row_blocks_kernel<<<grid, 256, 0, s>>>(cols, ldb, N, rb_blocks(N), S, slot_src, n_bins, rb, rb_pitch(S),
                                                 err);
  count_launches();
}

int plan_row_block_slots(const int32_t* n_bins, int32_t F, bool pack, uint32_t* loc, uint32_t* src) {
  int S = 0, open = -1;  // open: the slot whose low nibble holds an unpaired feature
  for (int f = 0; f < F; ++f) {
    if (pack && n_bins[f] <= kMaxPackedBins) {
      if (open >= 0) {
        loc[f] = static_cast<uint32_t>(open) | (2u << 16);
        src[open] = (src[open] & 0xffffu) | (static_cast<uint32_t>(f) << 16);
        open = -1;
        continue;
      }
      open = S;
      loc[f] = static_cast<uint32_t>(S) | (1u << 16);
    } else {
      loc[f] = static_cast<uint32_t>(S);
    }
    src[S++] = static_cast<uint32_t>(f) | 0xffff0000u;
  }
  if (open >= 0) loc[src[open] & 0xffffu] = static_cast<uint32_t>(open);  // unpaired: a whole byte
  return S;
}

int plan_row_block_slots_ex(const int32_t* n_bins, int32_t F, bool pack, bool regs, uint32_t* loc, uint32_t* src,
                            int* reg_begin, int* reg_codes) {
  *reg_codes = 0;
  if (!regs) {
    const int S = plan_row_block_slots(n_bins, F, pack, loc, src);
    *reg_begin = S;
    return S;
  }
  // ordinary slots: the features with more than kRegMaxCodes bins, as plan_row_block_slots pairs them
  int S = 0, open = -1;
  for (int f = 0; f < F; ++f) {
    if (n_bins[f] <= kRegMaxCodes) continue;
    if (pack && n_bins[f] <= kMaxPackedBins) {
      if (open >= 0) {
        loc[f] = static_cast<uint32_t>(open) | (2u << 16);
        src[open] = (src[open] & 0xffffu) | (static_cast<uint32_t>(f) << 16);
        open = -1;
        continue;
      }
      open = S;
      loc[f] = static_cast<uint32_t>(S) | (1u << 16);
    } else {
      loc[f] = static_cast<uint32_t>(S);
    }
    src[S++] = static_cast<uint32_t>(f) | 0xffff0000u;
  }
  if (open >= 0) loc[src[open] & 0xffffu] = static_cast<uint32_t>(open);
  *reg_begin = S;
  // register slots: the others in feature order, a pair when the two bin counts multiply to at most
  // kRegMaxCodes (the first in the low nibble), else one feature in a whole byte
  open = -1;
  auto close_open = [&]() {
    if (open < 0) return;
    const int fa = static_cast<int>(src[open] & 0xffffu);
    loc[fa] = static_cast<uint32_t>(open);
    *reg_codes = std::max(*reg_codes, static_cast<int>(n_bins[fa]));
    open = -1;
  };
  for (int f = 0; f < F; ++f) {
    if (n_bins[f] > kRegMaxCodes) continue;
    if (pack && open >= 0 && n_bins[src[open] & 0xffffu] * n_bins[f] <= kRegMaxCodes) {
      const int fa = static_cast<int>(src[open] & 0xffffu);
      loc[fa] = static_cast<uint32_t>(open) | (1u << 16);
      loc[f] = static_cast<uint32_t>(open) | (2u << 16);
      src[open] = (src[open] & 0xffffu) | (static_cast<uint32_t>(f) << 16);
      *reg_codes = std::max(*reg_codes, static_cast<int>(n_bins[fa] * n_bins[f]));
      open = -1;
      continue;
    }
    close_open();
    open = S;
    loc[f] = static_cast<uint32_t>(S);
    src[S++] = static_cast<uint32_t>(f) | 0xffff0000u;
  }
  close_open();
  return S;
}

// The tensor map the pair move reads a row-block buffer through: a 3-D byte tensor (32 bytes of a
// row block, S slots, the row blocks) and a box of one slot over kMvBoxBlocks row blocks.
int make_row_block_map(CUtensorMap* map, const uint8_t* rb, int64_t N, int32_t S) {
  using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeTiled encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<EncodeTiled>(fn);
  });
  if (!encode) {
    set_error("tensor-map encoding is not available from the CUDA driver");
    return GBDT_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kRowBlock), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(rb_blocks(N))};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBlock), static_cast<cuuint64_t>(rb_pitch(S))};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kRowBlock), 1u, static_cast<cuuint32_t>(kMvBoxBlocks)};
  const cuuint32_t elem[3] = {1u, 1u, 1u};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(rb), dims, strides, box, elem,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return GBDT_ERR_CUDA;
  }
  return GBDT_OK;
}

}  // namespace gbdt

using namespace gbdt;

extern "C" size_t gbdt_histograms_segmented_workspace_size(int32_t max_slots) {
  return kWsAlign + seg_hist_scratch_bytes(max_slots);  // the error word, then the level's work list
}

extern "C" int64_t gbdt_row_block_pitch(int32_t F) { return F >= 1 ? rb_pitch(F) : 0; }

extern "C" int32_t gbdt_row_block_slots(const int32_t* n_bins, int32_t F, int32_t packing, uint32_t* loc,
                                        uint32_t* src) {
  clear_error();
  GBDT_CHECK_ARG(n_bins && loc && src, "gbdt_row_block_slots: null pointer");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096, "gbdt_row_block_slots: F out of range");
  GBDT_CHECK_ARG(packing == GBDT_BIN_PACKING_4BIT || packing == GBDT_BIN_PACKING_OFF,
                 "gbdt_row_block_slots: bad packing mode");
  for (int f = 0; f < F; ++f)
    GBDT_CHECK_ARG(n_bins[f] >= 1 && n_bins[f] <= GBDT_MAX_BINS, "gbdt_row_block_slots: n_bins[%d] out of range", f);
  return plan_row_block_slots(n_bins, F, packing == GBDT_BIN_PACKING_4BIT, loc, src);
}

extern "C" int32_t gbdt_row_block_slots_ex(const int32_t* n_bins, int32_t F, int32_t packing, int32_t hist_registers,
                                           uint32_t* loc, uint32_t* src, int32_t* reg_begin) {
  clear_error();
  GBDT_CHECK_ARG(n_bins && loc && src && reg_begin, "gbdt_row_block_slots_ex: null pointer");
  GBDT_CHECK_ARG(F >= 1 && F <= 4096, "gbdt_row_block_slots_ex: F out of range");
  GBDT_CHECK_ARG(packing == GBDT_BIN_PACKING_4BIT || packing == GBDT_BIN_PACKING_OFF,
                 "gbdt_row_block_slots_ex: bad packing mode");
  GBDT_CHECK_ARG(hist_registers == GBDT_HIST_REGISTERS_OFF || hist_registers == GBDT_HIST_REGISTERS_ON,
                 "gbdt_row_block_slots_ex: bad hist_registers mode");
  for (int f = 0; f < F; ++f)
    GBDT_CHECK_ARG(n_bins[f] >= 1 && n_bins[f] <= GBDT_MAX_BINS, "gbdt_row_block_slots_ex: n_bins[%d] out of range",
                   f);
  int rb = 0, codes = 0;
  const int S = plan_row_block_slots_ex(n_bins, F, packing == GBDT_BIN_PACKING_4BIT,
                                        hist_registers == GBDT_HIST_REGISTERS_ON, loc, src, &rb, &codes);
  *reg_begin = rb;
  return S;
}

extern "C" size_t gbdt_row_block_bytes(int64_t N, int32_t F) {
  return (N >= 1 && F >= 1) ? row_block_bytes(N, F) : 0;
}

extern "C" int gbdt_bins_to_row_blocks(const uint8_t* bins, int64_t ldb, int64_t N, int32_t F, uint8_t* out,
                                       void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && out, "gbdt_bins_to_row_blocks: null pointer");
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 4096, "gbdt_bins_to_row_blocks: sizes out of range");
  GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins, 16) && aligned(out, 32),
                 "gbdt_bins_to_row_blocks: need ldb >= N, ldb %% 16 == 0, 16-byte aligned bins, 32-byte aligned out");
  launch_cols_to_row_blocks(bins, ldb, N, F, nullptr, nullptr, out, nullptr, static_cast<cudaStream_t>(stream));
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

namespace {
int build_segmented(const char* fn, const uint8_t* bins, int64_t ldb, int32_t layout, int64_t N, int32_t F,
                    const void* g, int32_t g_dtype, const int32_t* fixed_exp, const gbdt_level* level,
                    int32_t max_slots, const uint8_t* build_flag, int32_t max_build, const gbdt_segment* segments,
                    const gbdt_filter* filters, uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, bool with_h,
                    void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(bins && g && fixed_exp && level && build_flag && segments && hist_cnt && hist_q && (hist_h || !with_h),
                 "%s: null pointer", fn);
  GBDT_CHECK_ARG(N >= 1 && N < (int64_t(1) << 31) && F >= 1 && F <= 4096, "%s: sizes out of range", fn);
  GBDT_CHECK_ARG(layout == GBDT_LAYOUT_COLUMNS || layout == GBDT_LAYOUT_ROW_BLOCKS, "%s: bad layout", fn);
  if (layout == GBDT_LAYOUT_COLUMNS) {
    GBDT_CHECK_ARG(ldb >= N && ldb % 16 == 0 && aligned(bins, 16) && aligned(g, 16),
                   "%s: need ldb >= N, ldb %% 16 == 0, 16-byte aligned bins and g", fn);
  } else {
    GBDT_CHECK_ARG(ldb == rb_pitch(F) && aligned(bins, 32) && aligned(g, 16),
                   "%s: row blocks need ldb = gbdt_row_block_pitch(F), 32-byte aligned bins, 16-byte aligned g", fn);
  }
  GBDT_CHECK_ARG(g_dtype == GBDT_DTYPE_F32 || g_dtype == GBDT_DTYPE_F64, "%s: bad dtype", fn);
  GBDT_CHECK_ARG(max_slots >= 1 && max_slots <= kMaxSlots && max_build >= 1 && max_build <= max_slots,
                 "%s: slot bounds out of range", fn);
  const size_t need = gbdt_histograms_segmented_workspace_size(max_slots);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("%s: workspace needs %zu bytes", fn, need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word (gbdt_workspace_status; these kernels raise nothing, so it stays 0) and the scratch
  GBDT_CUDA(cudaMemsetAsync(ws, 0, sizeof(int32_t), s));
  void* scratch = static_cast<char*>(ws) + kWsAlign;
  const SegHistPlan plan = plan_seg_histograms(N, F, max_slots, max_build, with_h, filters != nullptr);
  int rc = launch_seg_histograms(plan, bins, ldb, N, F, g, g_dtype, fixed_exp, level, max_slots, build_flag, segments,
                                 filters, scratch, hist_cnt, hist_q, hist_h, s, layout == GBDT_LAYOUT_ROW_BLOCKS);
  if (rc != GBDT_OK) return rc;
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}
}  // namespace

extern "C" int gbdt_build_histograms_segmented(const uint8_t* bins, int64_t ldb, int32_t layout, int64_t N, int32_t F,
                                               const void* g, int32_t g_dtype, const int32_t* fixed_exp,
                                               const gbdt_level* level, int32_t max_slots, const uint8_t* build_flag,
                                               int32_t max_build, const gbdt_segment* segments,
                                               const gbdt_filter* filters, uint32_t* hist_cnt, int64_t* hist_q,
                                               void* ws, size_t ws_bytes, void* stream) {
  return build_segmented("gbdt_build_histograms_segmented", bins, ldb, layout, N, F, g, g_dtype, fixed_exp, level,
                         max_slots, build_flag, max_build, segments, filters, hist_cnt, hist_q, nullptr, false, ws,
                         ws_bytes, stream);
}

extern "C" int gbdt_build_histograms_segmented_h(const uint8_t* bins, int64_t ldb, int32_t layout, int64_t N,
                                                 int32_t F, const void* g, int32_t g_dtype, const int32_t* fixed_exp,
                                                 const gbdt_level* level, int32_t max_slots,
                                                 const uint8_t* build_flag, int32_t max_build,
                                                 const gbdt_segment* segments, const gbdt_filter* filters,
                                                 uint32_t* hist_cnt, int64_t* hist_q, int64_t* hist_h, void* ws,
                                                 size_t ws_bytes, void* stream) {
  return build_segmented("gbdt_build_histograms_segmented_h", bins, ldb, layout, N, F, g, g_dtype, fixed_exp, level,
                         max_slots, build_flag, max_build, segments, filters, hist_cnt, hist_q, hist_h, true, ws,
                         ws_bytes, stream);
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
