// Per-kernel CUDA-event timing of the library's launches (see attn_profile.h
// and attn_profile_start / attn_profile_stop in include/attn_gb300.h).
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/attn_gb300.h"
#include "attn_profile.h"

namespace attn {
namespace {

struct Record {
  int id;
  cudaEvent_t start, stop;
};

std::atomic<bool> g_enabled{false};
std::mutex g_mu;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;
cudaEvent_t g_open[kKernelCount] = {};

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

const char* kNames[kKernelCount] = {
    "fwd_tc05", "bwd_dkdv_tc05", "bwd_dq_tc05", "bwd_row_dot",
    "rope_qk", "fwd_simt", "bwd_dkdv_simt", "bwd_dq_simt", "bwd_prologue", "decode", "qkv_proj",
    "fp8_prep", "fwd_fp8", "split_prep", "fwd_split", "bwd_dkdv_split", "bwd_dq_split",
};

}  // namespace

void prof_begin(int id, cudaStream_t stream) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_mu);
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, stream) == cudaSuccess) g_open[id] = e;
}

void prof_end(int id, cudaStream_t stream) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_mu);
  cudaEvent_t s = g_open[id];
  g_open[id] = nullptr;
  if (!s) return;
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, stream) == cudaSuccess) g_records.push_back({id, s, e});
}

}  // namespace attn

using namespace attn;

extern "C" int attn_profile_start(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& r : g_records) {
    g_pool.push_back(r.start);
    g_pool.push_back(r.stop);
  }
  g_records.clear();
  g_enabled.store(true);
  return ATTN_OK;
}

extern "C" int attn_profile_stop(double* total_ms, int* launches, int n) {
  g_enabled.store(false);
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < n; ++i) {
    if (total_ms) total_ms[i] = 0.0;
    if (launches) launches[i] = 0;
  }
  int status = ATTN_OK;
  for (auto& r : g_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      status = ATTN_ERR_CUDA;
      continue;
    }
    if (r.id < n) {
      if (total_ms) total_ms[r.id] += ms;
      if (launches) launches[r.id] += 1;
    }
  }
  return status;
}

extern "C" const char* attn_kernel_name(int id) {
  return (id >= 0 && id < kKernelCount) ? kNames[id] : "unknown";
}
