// Batched prediction on raw fp32 features.
//
// "Gradient boosted trees (spec model)", Forward pass: a row's prediction is
// init + learning_rate * (sum of its tree outputs); Tree representation: a
// split sends x right when x > threshold.  On raw values the threshold of a
// split (feature j, bin b) is the quantize edge edges[j][b] (bin(x) = number of
// edges below x, so x > edges[b] exactly when bin(x) > b: the training routing).
// The sum is taken tree by tree as in training, pred + (lr * leaf value), so
// the predictions of the training rows are the training predictions bit for
// bit.  A NaN compares false and goes left.
//
// A preparation pass turns each tree's gbdt_node records into 16-byte nodes
// holding the threshold value itself (and checks them); the prediction kernel
// runs one thread per row and, for up to kStagedF features, first stages its
// CTA's rows x features in shared memory (feature-major, so lanes reading
// different features of their own rows never share a bank).
#include <algorithm>
#include <cmath>

#include "kernels.cuh"

namespace gbdt {

namespace {

constexpr int kPredRows = 128;    // rows (threads) per CTA
constexpr int kStagedF = 320;     // up to this many features the rows are staged (160 KB)

struct PNode {
  float thr;        // threshold value (internal nodes)
  int32_t feature;  // -1: leaf
  int32_t left;     // left child (right = left + 1)
  int32_t pad;
};

// One thread per node: threshold values, and a check of every internal node
// (feature and bin in range, children a pair after the node and inside the
// tree).  A bad node becomes a leaf and raises the error flag, so the
// traversal can never leave the tree.
__global__ void predict_prep_kernel(const gbdt_node* __restrict__ nodes, const int32_t* __restrict__ nodes_per_tree,
                                    int64_t total, int32_t max_nodes, int32_t F, const float* __restrict__ edges,
                                    int32_t max_bins, PNode* __restrict__ pn, double* __restrict__ leaf,
                                    int32_t* __restrict__ err) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(i % max_nodes);
    const int t = static_cast<int>(i / max_nodes);
    int n_t = nodes_per_tree ? nodes_per_tree[t] : max_nodes;
    if (n_t < 1 || n_t > max_nodes) {
      if (err && v == 0) atomicOr(err, 1);
      n_t = 1;
    }
    PNode p{0.0f, -1, -1, 0};
    if (v >= n_t) {  // a slot the tree does not use: never reached from a valid root
      pn[i] = p;
      leaf[i] = 0.0;
      continue;
    }
    const gbdt_node nd = nodes[i];
    if (!nd.is_leaf) {
      const bool ok = nd.feature >= 0 && nd.feature < F && nd.threshold_bin >= 0 &&
                      nd.threshold_bin < max_bins - 1 && nd.left > v && nd.right == nd.left + 1 && nd.right < n_t;
      if (ok) {
        p.thr = edges[static_cast<int64_t>(nd.feature) * (max_bins - 1) + nd.threshold_bin];
        p.feature = nd.feature;
        p.left = nd.left;
      } else if (err) {
        atomicOr(err, 1);
      }
    }
    pn[i] = p;
    leaf[i] = nd.leaf_value;
  }
}

template <bool kStaged>
__global__ void __launch_bounds__(kPredRows)
    predict_kernel(const float* __restrict__ X, int64_t ldx, int64_t N, int32_t F, const PNode* __restrict__ pn,
                   const double* __restrict__ leaf, int32_t n_trees, int32_t max_nodes, double init, double lr,
                   double* __restrict__ out) {
  extern __shared__ float xs[];  // [F][kPredRows] when staged
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPredRows;
  const int r = threadIdx.x;
  const int64_t row = row0 + r;
  const bool in = row < N;
  if (kStaged) {
    for (int f = 0; f < F; ++f) xs[f * kPredRows + r] = in ? X[static_cast<int64_t>(f) * ldx + row] : 0.0f;
    __syncthreads();
  }
  if (!in) return;
  double acc = init;
  for (int t = 0; t < n_trees; ++t) {
    const PNode* tn = pn + static_cast<int64_t>(t) * max_nodes;
    int v = 0;
    for (int step = 0; step < max_nodes; ++step) {  // children come after their node: a path ends in time
      const PNode nd = tn[v];
      if (nd.feature < 0) break;
      const float x = kStaged ? xs[nd.feature * kPredRows + r] : X[static_cast<int64_t>(nd.feature) * ldx + row];
      v = x > nd.thr ? nd.left + 1 : nd.left;
    }
    acc = __dadd_rn(acc, __dmul_rn(lr, leaf[static_cast<int64_t>(t) * max_nodes + v]));
  }
  out[row] = acc;
}

size_t predict_bytes(int32_t n_trees, int32_t max_nodes) {
  const size_t total = static_cast<size_t>(n_trees > 0 ? n_trees : 0) * static_cast<size_t>(max_nodes);
  return sizeof(PNode) * total + sizeof(double) * total + sizeof(int32_t) + 3 * kWsAlign;
}

}  // namespace

}  // namespace gbdt

using namespace gbdt;

extern "C" size_t gbdt_predict_workspace_size(int32_t n_trees, int32_t max_nodes) {
  return predict_bytes(n_trees, max_nodes < 1 ? 1 : max_nodes);
}

extern "C" int gbdt_predict(const float* X, int64_t ldx, int64_t N, int32_t F, const float* edges, int32_t max_bins,
                            const gbdt_node* nodes, const int32_t* nodes_per_tree, int32_t n_trees, int32_t max_nodes,
                            double init_pred, double learning_rate, double* out, void* ws, size_t ws_bytes,
                            void* stream) {
  clear_error();
  GBDT_CHECK_ARG(X && edges && out && (nodes || n_trees == 0), "gbdt_predict: null pointer");
  GBDT_CHECK_ARG(N >= 0 && N < (int64_t(1) << 40) && F >= 1 && F <= 65535 && ldx >= N,
                 "gbdt_predict: need N >= 0, 1 <= F <= 65535, ldx >= N");
  GBDT_CHECK_ARG(max_bins >= 2 && max_bins <= GBDT_MAX_BINS, "gbdt_predict: max_bins must be in 2..256");
  GBDT_CHECK_ARG(n_trees >= 0 && max_nodes >= 1 && max_nodes <= (1 << 16), "gbdt_predict: bad tree sizes");
  GBDT_CHECK_ARG(std::isfinite(init_pred) && std::isfinite(learning_rate), "gbdt_predict: non-finite init or rate");
  const size_t need = predict_bytes(n_trees, max_nodes);
  if (!ws || ws_bytes < need || !aligned(ws, kWsAlign)) {
    set_error("gbdt_predict: workspace needs %zu bytes", need);
    return ws ? GBDT_ERR_WORKSPACE : GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t total = static_cast<int64_t>(n_trees) * max_nodes;
  Carve c(ws, ws_bytes);
  PNode* pn = c.take<PNode>(total > 0 ? total : 1);
  double* leaf = c.take<double>(total > 0 ? total : 1);
  int32_t* err = c.take<int32_t>(1);
  GBDT_CUDA(cudaMemsetAsync(err, 0, sizeof(int32_t), s));
  if (total > 0) {
    const int grid = static_cast<int>(std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(sm_count()) * 8));
    predict_prep_kernel<<<grid, 256, 0, s>>>(nodes, nodes_per_tree, total, max_nodes, F, edges, max_bins, pn, leaf,
                                             err);
    count_launches();
  }
  if (N > 0) {
    const int64_t blocks = (N + kPredRows - 1) / kPredRows;
    GBDT_CHECK_ARG(blocks < (int64_t(1) << 31), "gbdt_predict: too many rows for one call");
    if (F <= kStagedF) {
      const size_t smem = static_cast<size_t>(F) * kPredRows * sizeof(float);
      GBDT_CUDA(cudaFuncSetAttribute(predict_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)));
      predict_kernel<true><<<static_cast<unsigned>(blocks), kPredRows, smem, s>>>(
          X, ldx, N, F, pn, leaf, n_trees, max_nodes, init_pred, learning_rate, out);
    } else {
      predict_kernel<false><<<static_cast<unsigned>(blocks), kPredRows, 0, s>>>(
          X, ldx, N, F, pn, leaf, n_trees, max_nodes, init_pred, learning_rate, out);
    }
    count_launches();
  }
  GBDT_LAUNCH_CHECK();
  int32_t h_err = 0;
  GBDT_CUDA(cudaMemcpyAsync(&h_err, err, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (h_err) {
    set_error("gbdt_predict: the model has an invalid node count, or an internal node with an invalid feature, "
              "bin or child index");
    return GBDT_ERR_INVALID_ARG;
  }
  return GBDT_OK;
}
