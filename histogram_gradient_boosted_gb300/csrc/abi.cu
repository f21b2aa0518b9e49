// Error reporting, version, parameter rules and device queries of the C ABI.
#include <atomic>
#include <cmath>
#include <cstring>

#include "common.cuh"

namespace gbdt {

namespace {
thread_local char t_msg[512] = "";
}

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
}

void clear_error() { t_msg[0] = '\0'; }

int report_error_bits(const char* what, int32_t bits) {
  if (bits == 0) return GBDT_OK;
  char names[256] = "";
  const struct {
    int32_t bit;
    const char* name;
  } known[] = {{kErrHistTotals, "histogram totals"},
               {kErrSlotRange, "node id outside the level"},
               {kErrPartitionCount, "partition count differs from the split record"},
               {kErrLevelSize, "level larger than max_slots"},
               {kErrWaitTimeout, "asynchronous copy wait limit"},
               {kErrBinRange, "bin not below n_bins"}};
  for (const auto& k : known) {
    if (!(bits & k.bit)) continue;
    const size_t used = strlen(names);
    snprintf(names + used, sizeof(names) - used, "%s%s", used ? "; " : "", k.name);
  }
  set_error("%s: device consistency check failed (error bits 0x%x: %s)", what, bits, names);
  return (bits & ~kErrBinRange) ? GBDT_ERR_INTERNAL : GBDT_ERR_INVALID_ARG;
}

namespace {
std::atomic<int64_t> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
int64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

int sm_count() {
  static int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 152;
    return v;
  }();
  return n;
}

}  // namespace gbdt

// "Module Design: Training Core" s.3: min_samples_leaf >= 1, min_child_weight >= 0,
// reg_lambda >= 0, gamma >= 0, every floating parameter finite.
int validate_params(const gbdt_params* p) {
  using gbdt::set_error;
  if (!p) {
    set_error("parameters: null pointer");
    return GBDT_ERR_INVALID_ARG;
  }
  if (!std::isfinite(p->learning_rate) || !std::isfinite(p->reg_lambda) || !std::isfinite(p->gamma) ||
      !std::isfinite(p->min_child_weight)) {
    set_error("parameters: every floating parameter must be finite");
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->min_samples_leaf < 1 || p->min_child_weight < 0.0 || p->reg_lambda < 0.0 || p->gamma < 0.0) {
    set_error("parameters: need min_samples_leaf >= 1, min_child_weight >= 0, reg_lambda >= 0, gamma >= 0");
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->n_trees < 0 || p->max_depth < 0 || p->max_depth > GBDT_MAX_DEPTH) {
    set_error("parameters: need n_trees >= 0 and 0 <= max_depth <= %d", GBDT_MAX_DEPTH);
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->num_leaves < 0 || p->num_leaves == 1) {
    set_error("parameters: num_leaves must be 0 (no budget) or at least 2");
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->bin_packing != GBDT_BIN_PACKING_4BIT && p->bin_packing != GBDT_BIN_PACKING_OFF) {
    set_error("parameters: bin_packing must be %d (4-bit) or %d (off)", GBDT_BIN_PACKING_4BIT, GBDT_BIN_PACKING_OFF);
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->hist_registers != GBDT_HIST_REGISTERS_OFF && p->hist_registers != GBDT_HIST_REGISTERS_ON) {
    set_error("parameters: hist_registers must be %d (off) or %d (on)", GBDT_HIST_REGISTERS_OFF,
              GBDT_HIST_REGISTERS_ON);
    return GBDT_ERR_INVALID_ARG;
  }
  if (p->objective != GBDT_OBJECTIVE_SQUARED_ERROR && p->objective != GBDT_OBJECTIVE_LOGISTIC) {
    set_error("parameters: objective must be %d (squared error) or %d (logistic)", GBDT_OBJECTIVE_SQUARED_ERROR,
              GBDT_OBJECTIVE_LOGISTIC);
    return GBDT_ERR_INVALID_ARG;
  }
  return GBDT_OK;
}

extern "C" const char* gbdt_last_error(void) { return gbdt::t_msg; }

extern "C" const char* gbdt_version(void) { return "gbdt-gb300 0.1 (sm_103a)"; }

extern "C" int gbdt_validate_params(const gbdt_params* p) {
  gbdt::clear_error();
  return validate_params(p);
}

extern "C" int64_t gbdt_kernel_launch_count(void) { return gbdt::launch_count(); }

extern "C" int gbdt_workspace_status(const void* ws, int32_t* bits, void* stream) {
  gbdt::clear_error();
  if (bits) *bits = 0;
  if (!ws || !gbdt::aligned(ws, gbdt::kWsAlign)) {
    gbdt::set_error("gbdt_workspace_status: ws must be a 256-byte aligned workspace");
    return GBDT_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  GBDT_CUDA(cudaMemcpyAsync(&h, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  GBDT_CUDA(cudaStreamSynchronize(s));
  if (bits) *bits = h;
  return gbdt::report_error_bits("gbdt_workspace_status", h);
}
