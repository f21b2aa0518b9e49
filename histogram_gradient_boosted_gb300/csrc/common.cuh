// Internal helpers shared by the library's translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (the tensor-map type only; encoding goes through the runtime entry point)
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>

#include "gbdt.h"

namespace gbdt {

constexpr int kBins = 256;           // histogram width: every value of a uint8 bin
constexpr int kMaxSlots = 4096;      // slots per level the kernels support
constexpr size_t kWsAlign = 256;     // alignment of every workspace carve-out

// Bits of the device error word (kernels OR them in; the host reports INTERNAL).
enum : int32_t {
  kErrHistTotals = 1,     // a feature's histogram does not add up to the node totals
  kErrSlotRange = 2,      // a row's node id is outside the level it should be in
  kErrPartitionCount = 4, // partition left count differs from the split record
  kErrLevelSize = 8,      // a level has more slots than the launch bound
  kErrWaitTimeout = 16,   // an asynchronous copy did not complete within its wait limit
  kErrBinRange = 32,      // a caller's bin is not below its feature's n_bins
};

// ---- thread-local error message -------------------------------------------------
void set_error(const char* fmt, ...);
void clear_error();
// GBDT_OK for bits == 0; otherwise sets the message (naming each bit) and returns GBDT_ERR_INTERNAL,
// or GBDT_ERR_INVALID_ARG when the only bit is kErrBinRange (a caller's input out of range).
int report_error_bits(const char* what, int32_t bits);

#define GBDT_CHECK_ARG(cond, ...)         \
  do {                                    \
    if (!(cond)) {                        \
      ::gbdt::set_error(__VA_ARGS__);     \
      return GBDT_ERR_INVALID_ARG;        \
    }                                     \
  } while (0)

#define GBDT_CUDA(call)                                                                        \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) {                                                                   \
      ::gbdt::set_error("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return GBDT_ERR_CUDA;                                                                    \
    }                                                                                          \
  } while (0)

// Error from the launches just queued (configuration errors surface here).
#define GBDT_LAUNCH_CHECK() GBDT_CUDA(cudaGetLastError())

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bump allocator over the caller's workspace.
struct Carve {
  char* base;
  size_t cap;
  size_t used = 0;
  Carve(void* b, size_t c) : base(static_cast<char*>(b)), cap(c) {}
  template <typename T>
  T* take(size_t count) {
    size_t off = (used + kWsAlign - 1) / kWsAlign * kWsAlign;
    used = off + count * sizeof(T);
    return (base && used <= cap) ? reinterpret_cast<T*>(base + off) : nullptr;
  }
  bool ok() const { return used <= cap; }
};

// Fixed-point exponent: S = 62 - ceil(log2 N) - E with maxabs < 2^E, so that
// sum |round(g * 2^S)| < 2^62 for any row set; S = 0 when all g are zero.
// Clamped to keep 2^S a normal double.
__host__ __device__ inline int fixed_exponent(double maxabs, int64_t N) {
  if (!(maxabs > 0.0)) return 0;
  int E = 0;
  frexp(maxabs, &E);  // maxabs = m * 2^E, 0.5 <= m < 1
  int L = 0;
  while ((int64_t(1) << L) < N) ++L;
  int S = 62 - L - E;
  if (S > 1000) S = 1000;
  if (S < -1000) S = -1000;
  return S;
}

// round-half-even(g * 2^S) for the scale 2^S (an exact power of two).
__device__ __forceinline__ int64_t to_fixed(double g, double scale) { return __double2ll_rn(g * scale); }

// Hessian of the logistic loss from the row's gradient g = p - y (y is 0 or 1,
// p = sigmoid(pred)): |g| is p when y = 0 and 1 - p when y = 1, so
// p (1 - p) = |g| (1 - |g|).  For y = 0 this is the product p * (1 - p) itself;
// for y = 1 it uses the rounded g.
__device__ __forceinline__ double logistic_hess(double g) {
  const double a = fabs(g);
  return __dmul_rn(a, __dsub_rn(1.0, a));
}

// sigmoid(x) = 1 / (1 + exp(-x)) in FP64, each operation rounded once.
__device__ __forceinline__ double sigmoid(double x) { return __ddiv_rn(1.0, __dadd_rn(1.0, exp(-x))); }

// Convert a fixed-point sum back to a double: q * 2^-S.
__host__ __device__ inline double from_fixed(int64_t q, int S) { return ldexp(static_cast<double>(q), -S); }

// Exclusive scan of v over the block (blockDim.x a multiple of 32, at most 1024): warp scans by
// shuffles, one warp scans the warp totals.  *total = the block's sum.  s_warp: 33 shared
// elements.  Every thread of the block must call it (it holds three barriers).
template <typename T>
__device__ __forceinline__ T block_scan_excl(T v, T* s_warp, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    const T w = lane < nw ? s_warp[lane] : T(0);
    T wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const T t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const T r = s_warp[warp] + incl - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void raise_error(int32_t* flag, int32_t bits) {
  if (flag) atomicOr(flag, bits);
}

// ---- bulk asynchronous copies (global -> shared memory) completed on an mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t arrivals) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(arrivals) : "memory");
}

// Make initialised mbarriers visible to the asynchronous (copy) proxy.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to shared memory; the copy's completion is one phase of `bar`, which this
// call arms with the expected byte count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Wait until the phase with parity `parity` of bar has completed.  Gives up
// after `limit` polls and returns false, so that no wait can hang.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Load one box of a 3-D tensor map (coordinates innermost first) into shared
// memory; completion is one phase of `bar`, armed here with the box's bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint32_t bytes,
                                            uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ---- row-block layout of binned features (training-internal) ---------------------------------
// Position p of feature f sits at byte (p / 32) * pitch + 32 * f + p % 32, pitch = 32 * F: the 32
// rows of a row block are contiguous per feature and the features of a row block contiguous, so a
// warp reading 32 rows of 32 consecutive features reads one contiguous kilobyte.
constexpr int kRowBlock = 32;
__host__ __device__ __forceinline__ int64_t rb_offset(int f, int64_t p, int64_t pitch) {
  return (p >> 5) * pitch + static_cast<int64_t>(f) * kRowBlock + (p & 31);
}
inline int64_t rb_pitch(int32_t F) { return static_cast<int64_t>(F) * kRowBlock; }
inline int64_t rb_blocks(int64_t N) { return (N + kRowBlock - 1) / kRowBlock; }

// 4-bit slots: in the training copies two features with at most 16 bins share one 32-byte slot
// of a row block, the first of the pair in the low nibble of each byte, the second in the high
// nibble ("two cells per byte"); every other feature has a slot of its own.  A feature's
// locator says where its bins sit: loc = slot | nibble << 16, nibble 0 for a whole byte, 1 for
// the low nibble, 2 for the high nibble.  The pitch is 32 bytes per slot.
constexpr int kMaxPackedBins = 16;
__host__ __device__ __forceinline__ uint32_t loc_slot(uint32_t loc) { return loc & 0xffffu; }
__host__ __device__ __forceinline__ uint32_t loc_shift(uint32_t loc) { return (loc >> 16) == 2 ? 4u : 0u; }
__host__ __device__ __forceinline__ uint32_t loc_mask(uint32_t loc) { return (loc >> 16) == 0 ? 0xffu : 0x0fu; }
// Bin of position p of the feature at loc in a row-block buffer of the given pitch.
__device__ __forceinline__ int rb_bin(const uint8_t* __restrict__ rb, uint32_t loc, int64_t p, int64_t pitch) {
  const uint32_t b = rb[rb_offset(static_cast<int>(loc_slot(loc)), p, pitch)];
  return static_cast<int>((b >> loc_shift(loc)) & loc_mask(loc));
}

inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Number of SMs of the current device (cached per process; one device per process).
int sm_count();

// Process-wide count of kernels this library has launched (reported through
// gbdt_kernel_launch_count so a caller can count launches in a timed region).
void count_launches(int n = 1);
int64_t launch_count();

}  // namespace gbdt
