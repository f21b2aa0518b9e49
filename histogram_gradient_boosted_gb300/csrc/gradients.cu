// Gradients, label mean, prediction update, fixed-point exponents.
// "Module Design: Training Core" s.2 (squared error: g = pred - label, h = 1)
// and s.6 step 7 (update training predictions after the tree); "Gradient
// boosted trees (spec model)": forward pass (init + learning_rate * tree
// output) and the binary cross-entropy of a sigmoid (logistic: g =
// sigmoid(pred) - label, h = p (1 - p)).
#include "kernels.cuh"

namespace gbdt {

namespace {

__device__ __forceinline__ unsigned long long abs_bits(double v) {
  return static_cast<unsigned long long>(__double_as_longlong(fabs(v)));
}

__device__ __forceinline__ unsigned long long warp_max(unsigned long long v) {
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Block max of non-negative doubles held as their bit patterns, one atomic per block:
// out[0] = max(out[0], v0) and, with two, out[1] = max(out[1], v1).
__device__ __forceinline__ void block_max_to(unsigned long long v0, unsigned long long v1, unsigned long long* out,
                                             bool two) {
  __shared__ unsigned long long red[2][32];
  v0 = warp_max(v0);
  v1 = warp_max(v1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[0][warp] = v0, red[1][warp] = v1;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    v0 = warp_max(lane < nw ? red[0][lane] : 0ull);
    v1 = warp_max(lane < nw ? red[1][lane] : 0ull);
    if (lane == 0 && v0) atomicMax(out, v0);
    if (lane == 0 && two && v1) atomicMax(out + 1, v1);
  }
}
__device__ __forceinline__ void block_max_to(unsigned long long v, unsigned long long* out) {
  block_max_to(v, 0ull, out, false);
}

// The gradient of a row at margin p: squared error p - y; logistic sigmoid(p) - y.
__device__ __forceinline__ double gradient_of(double p, float y, int objective) {
  return objective == GBDT_OBJECTIVE_LOGISTIC ? __dsub_rn(sigmoid(p), static_cast<double>(y))
                                              : __dsub_rn(p, static_cast<double>(y));
}

// Fixed grid; each block sums a contiguous range in a fixed order, then a fixed tree.
// nonfinite: bit 1 for a NaN/Inf label; with binary, bit 2 for a label other than 0 or 1.
__global__ void label_sum_kernel(const float* __restrict__ label, int64_t N, double* __restrict__ partials,
                                 int32_t* __restrict__ nonfinite, int binary) {
  const int64_t per = (N + gridDim.x - 1) / gridDim.x;
  const int64_t b0 = blockIdx.x * per;
  const int64_t b1 = min(N, b0 + per);
  double acc = 0.0;
  bool bad = false, nonbin = false;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
    float v = label[i];
    bad |= !isfinite(v);
    nonbin |= binary && v != 0.0f && v != 1.0f;
    acc += static_cast<double>(v);
  }
  if (bad) atomicOr(nonfinite, 1);
  if (nonbin) atomicOr(nonfinite, 2);
  __shared__ double red[kSumThreads];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[blockIdx.x] = red[0];
}

// zero: the initial margin of the logistic objective, 0.
__global__ void label_mean_kernel(const double* __restrict__ partials, int64_t N, double* __restrict__ init,
                                  int zero) {
  __shared__ double red[kSumThreads];
  double acc = 0.0;
  for (int i = threadIdx.x; i < kSumBlocks; i += blockDim.x) acc += partials[i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *init = zero ? 0.0 : __ddiv_rn(red[0], static_cast<double>(N));
}

// maxabs[0] = max |g|; logistic: maxabs[1] = max h (h = logistic_hess(g)).
__global__ void start_tree0_kernel(const double* __restrict__ init, const float* __restrict__ label, int64_t N,
                                   int objective, double* __restrict__ pred, double* __restrict__ g,
                                   uint16_t* __restrict__ node, unsigned long long* maxabs) {
  const double p0 = *init;
  const bool logistic = objective == GBDT_OBJECTIVE_LOGISTIC;
  unsigned long long m = 0, mh = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    pred[i] = p0;
    const double gi = gradient_of(p0, label[i], objective);
    g[i] = gi;
    node[i] = 0;
    const unsigned long long a = abs_bits(gi);
    m = a > m ? a : m;
    if (logistic) {
      const unsigned long long b = abs_bits(logistic_hess(gi));
      mh = b > mh ? b : mh;
    }
  }
  block_max_to(m, mh, maxabs, logistic);
}

__global__ void finish_tree_kernel(const gbdt_node* __restrict__ trees, const int32_t* __restrict__ n_nodes,
                                   const int32_t* __restrict__ tree_index, int32_t max_nodes, double lr,
                                   const float* __restrict__ label, int64_t N, int objective,
                                   double* __restrict__ pred, double* __restrict__ g, uint16_t* __restrict__ node,
                                   unsigned long long* maxabs, int next) {
  extern __shared__ double s_step[];  // lr * leaf_value per node of the tree
  const int t = *tree_index;
  const gbdt_node* __restrict__ tree = trees + static_cast<int64_t>(t) * max_nodes;
  const int nn = min(n_nodes[t], max_nodes);
  const bool logistic = objective == GBDT_OBJECTIVE_LOGISTIC;
  for (int i = threadIdx.x; i < nn; i += blockDim.x) s_step[i] = __dmul_rn(lr, tree[i].leaf_value);
  __syncthreads();
  unsigned long long m = 0, mh = 0;
  // two rows per thread and step (stride apart), their loads issued before either is used, so that each
  // SM has twice the bytes in flight of one row per step
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += 2 * stride) {
    const int64_t j = i + stride;
    const bool two = j < N;
    const int v0 = node[i], v1 = two ? node[j] : 0;
    const double q0 = pred[i], q1 = two ? pred[j] : 0.0;
    float y0 = 0.f, y1 = 0.f;
    if (next) {
      y0 = label[i];
      y1 = two ? label[j] : 0.f;
    }
    const double p0 = (v0 < nn) ? __dadd_rn(q0, s_step[v0]) : q0;
    const double p1 = (v1 < nn) ? __dadd_rn(q1, s_step[v1]) : q1;
    pred[i] = p0;
    if (two) pred[j] = p1;
    if (next) {
      const double g0 = gradient_of(p0, y0, objective), g1 = gradient_of(p1, y1, objective);
      g[i] = g0;
      node[i] = 0;
      unsigned long long a = abs_bits(g0);
      m = a > m ? a : m;
      if (logistic) {
        const unsigned long long b = abs_bits(logistic_hess(g0));
        mh = b > mh ? b : mh;
      }
      if (two) {
        g[j] = g1;
        node[j] = 0;
        a = abs_bits(g1);
        m = a > m ? a : m;
        if (logistic) {
          const unsigned long long b = abs_bits(logistic_hess(g1));
          mh = b > mh ? b : mh;
        }
      }
    }
  }
  if (next) block_max_to(m, mh, maxabs, logistic);
}

__global__ void gradients_kernel(const double* __restrict__ pred, const float* __restrict__ label, int64_t N,
                                 int objective, double* __restrict__ g, unsigned long long* maxabs) {
  const bool logistic = objective == GBDT_OBJECTIVE_LOGISTIC;
  unsigned long long m = 0, mh = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    const double gi = gradient_of(pred[i], label[i], objective);
    g[i] = gi;
    const unsigned long long a = abs_bits(gi);
    m = a > m ? a : m;
    if (logistic) {
      const unsigned long long b = abs_bits(logistic_hess(gi));
      mh = b > mh ? b : mh;
    }
  }
  block_max_to(m, mh, maxabs, logistic);
}

template <typename T>
__global__ void maxabs_kernel(const T* __restrict__ g, int64_t N, unsigned long long* maxabs) {
  unsigned long long m = 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    const unsigned long long a = abs_bits(static_cast<double>(g[i]));
    m = a > m ? a : m;
  }
  block_max_to(m, maxabs);
}

// fixed_exp[0] from maxabs[0]; with_h: fixed_exp[1] (S_h of the hessians) from maxabs[1].  clear: the
// maxima are then reset to 0 for the next tree's gradients to raise (training reads them only here).
__global__ void fixed_exp_kernel(unsigned long long* maxabs, int64_t N, int32_t* fixed_exp, int with_h, int clear) {
  const unsigned long long m = maxabs[0], mh = with_h ? maxabs[1] : 0ull;
  fixed_exp[0] = fixed_exponent(__longlong_as_double(static_cast<long long>(m)), N);
  if (with_h) fixed_exp[1] = fixed_exponent(__longlong_as_double(static_cast<long long>(mh)), N);
  if (clear) {
    maxabs[0] = 0;
    maxabs[1] = 0;
  }
}

__global__ void update_predictions_kernel(double* __restrict__ pred, const uint16_t* __restrict__ leaf_of_row,
                                          const double* __restrict__ leaf_value, int32_t n_values, int64_t N,
                                          double lr) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    const int v = leaf_of_row[i];
    if (v < n_values) pred[i] = __dadd_rn(pred[i], __dmul_rn(lr, leaf_value[v]));
  }
}

int elementwise_grid(int64_t N) {
  const int64_t want = (N + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

void launch_label_sum(const float* label, int64_t N, double* partials, int32_t* nonfinite, bool binary,
                      cudaStream_t s) {
  label_sum_kernel<<<kSumBlocks, kSumThreads, 0, s>>>(label, N, partials, nonfinite, binary ? 1 : 0);
  count_launches();
}
void launch_label_mean(const double* partials, int64_t N, double* init, bool zero, cudaStream_t s) {
  label_mean_kernel<<<1, kSumThreads, 0, s>>>(partials, N, init, zero ? 1 : 0);
  count_launches();
}
void launch_start_tree0(const double* init, const float* label, int64_t N, int32_t objective, double* pred,
                        double* g, uint16_t* node, unsigned long long* maxabs, cudaStream_t s) {
  start_tree0_kernel<<<elementwise_grid(N), 256, 0, s>>>(init, label, N, objective, pred, g, node, maxabs);
  count_launches();
}
void launch_finish_tree(const gbdt_node* trees, const int32_t* n_nodes, const int32_t* tree_index,
                        int32_t max_nodes, double lr, const float* label, int64_t N, int32_t objective, double* pred,
                        double* g, uint16_t* node, unsigned long long* maxabs, bool next, cudaStream_t s) {
  static bool once = (cudaFuncSetAttribute(finish_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sizeof(double) * ((1 << (GBDT_MAX_DEPTH + 1)) - 1))),
                      true);
  (void)once;
  finish_tree_kernel<<<elementwise_grid(N), 256, sizeof(double) * max_nodes, s>>>(
      trees, n_nodes, tree_index, max_nodes, lr, label, N, objective, pred, g, node, maxabs, next ? 1 : 0);
  count_launches();
}
void launch_gradients(const double* pred, const float* label, int64_t N, int32_t objective, double* g,
                      unsigned long long* maxabs, cudaStream_t s) {
  gradients_kernel<<<elementwise_grid(N), 256, 0, s>>>(pred, label, N, objective, g, maxabs);
  count_launches();
}
void launch_maxabs(const void* g, int32_t dtype, int64_t N, unsigned long long* maxabs, cudaStream_t s) {
  if (dtype == GBDT_DTYPE_F32)
    maxabs_kernel<float><<<elementwise_grid(N), 256, 0, s>>>(static_cast<const float*>(g), N, maxabs);
  else
    maxabs_kernel<double><<<elementwise_grid(N), 256, 0, s>>>(static_cast<const double*>(g), N, maxabs);
  count_launches();
}
void launch_fixed_exp(unsigned long long* maxabs, int64_t N, int32_t* fixed_exp, bool with_h, cudaStream_t s,
                      bool clear) {
  fixed_exp_kernel<<<1, 1, 0, s>>>(maxabs, N, fixed_exp, with_h ? 1 : 0, clear ? 1 : 0);
  count_launches();
}

}  // namespace gbdt

using namespace gbdt;

extern "C" size_t gbdt_gradients_workspace_size(int64_t N) {
  (void)N;
  return 2 * kWsAlign;  // the error word (no check here: it stays 0), then two 8-byte max accumulators
}

extern "C" int gbdt_compute_gradients_objective(const double* pred, const float* label, int64_t N,
                                                int32_t objective, double* g, int32_t* fixed_exp, void* ws,
                                                size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(pred && label && g && fixed_exp, "gbdt_compute_gradients: null pointer");
  GBDT_CHECK_ARG(N >= 1, "gbdt_compute_gradients: N must be >= 1 (got %lld)", (long long)N);
  GBDT_CHECK_ARG(objective == GBDT_OBJECTIVE_SQUARED_ERROR || objective == GBDT_OBJECTIVE_LOGISTIC,
                 "gbdt_compute_gradients: unknown objective %d", objective);
  if (!ws || ws_bytes < gbdt_gradients_workspace_size(N) || !aligned(ws, kWsAlign)) {
    set_error("gbdt_compute_gradients: workspace too small or misaligned");
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GBDT_CUDA(cudaMemsetAsync(ws, 0, sizeof(int32_t), s));
  auto* maxabs = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + kWsAlign);
  GBDT_CUDA(cudaMemsetAsync(maxabs, 0, 2 * sizeof(*maxabs), s));
  launch_gradients(pred, label, N, objective, g, maxabs, s);
  launch_fixed_exp(maxabs, N, fixed_exp, objective == GBDT_OBJECTIVE_LOGISTIC, s);
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" int gbdt_compute_gradients(const double* pred, const float* label, int64_t N, double* g,
                                      int32_t* fixed_exp, void* ws, size_t ws_bytes, void* stream) {
  return gbdt_compute_gradients_objective(pred, label, N, GBDT_OBJECTIVE_SQUARED_ERROR, g, fixed_exp, ws, ws_bytes,
                                          stream);
}

extern "C" int gbdt_gradient_scale(const void* g, int32_t g_dtype, int64_t N, int32_t* fixed_exp, void* ws,
                                   size_t ws_bytes, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(g && fixed_exp, "gbdt_gradient_scale: null pointer");
  GBDT_CHECK_ARG(N >= 1, "gbdt_gradient_scale: N must be >= 1");
  GBDT_CHECK_ARG(g_dtype == GBDT_DTYPE_F32 || g_dtype == GBDT_DTYPE_F64, "gbdt_gradient_scale: bad dtype %d",
                 g_dtype);
  if (!ws || ws_bytes < gbdt_gradients_workspace_size(N) || !aligned(ws, kWsAlign)) {
    set_error("gbdt_gradient_scale: workspace too small or misaligned");
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GBDT_CUDA(cudaMemsetAsync(ws, 0, sizeof(int32_t), s));
  auto* maxabs = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + kWsAlign);
  GBDT_CUDA(cudaMemsetAsync(maxabs, 0, sizeof(*maxabs), s));
  launch_maxabs(g, g_dtype, N, maxabs, s);
  launch_fixed_exp(maxabs, N, fixed_exp, false, s);
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}

extern "C" int gbdt_update_predictions(double* pred, const uint16_t* leaf_of_row, const double* leaf_value,
                                       int32_t n_leaf_values, int64_t N, double lr, void* stream) {
  clear_error();
  GBDT_CHECK_ARG(pred && leaf_of_row && leaf_value, "gbdt_update_predictions: null pointer");
  GBDT_CHECK_ARG(N >= 1 && n_leaf_values >= 1, "gbdt_update_predictions: bad sizes");
  GBDT_CHECK_ARG(isfinite(lr), "gbdt_update_predictions: learning rate must be finite");
  update_predictions_kernel<<<elementwise_grid(N), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      pred, leaf_of_row, leaf_value, n_leaf_values, N, lr);
  count_launches();
  GBDT_LAUNCH_CHECK();
  return GBDT_OK;
}
