// Optional per-kernel device timing (nvq_timing_enable / nvq_timing_read).
//
// While enabled, every kernel launch made through the C ABI is bracketed by two
// CUDA events recorded on the stream it is launched on, filed under the
// launch's kernel kind.  Reading synchronizes the stop events of that kind and
// sums the elapsed times.  This measures one kernel of a multi-kernel call (for
// instance the dK/dV kernel inside attn_qat_bwd) live, inside a longer timed
// region, on the launching stream.
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "nvfp4attn.h"
#include "nvq_internal.h"

namespace nvq {

namespace {

struct Interval {
  cudaEvent_t start, stop;
};

std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<Interval> g_records[NVQ_KERNEL_KINDS];

void discard_all_locked() {
  for (auto& v : g_records) {
    for (const Interval& r : v) {
      cudaEventDestroy(r.start);
      cudaEventDestroy(r.stop);
    }
    v.clear();
  }
}

}  // namespace

TimedLaunch::TimedLaunch(int kind, cudaStream_t stream) : kind_(kind), stream_(stream) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (!g_timing_on || kind < 0 || kind >= NVQ_KERNEL_KINDS) return;
  if (cudaEventCreate(&start_) != cudaSuccess) return;
  if (cudaEventCreate(&stop_) != cudaSuccess) {
    cudaEventDestroy(start_);
    start_ = nullptr;
    return;
  }
  if (cudaEventRecord(start_, stream_) != cudaSuccess) {
    cudaEventDestroy(start_);
    cudaEventDestroy(stop_);
    start_ = stop_ = nullptr;
  }
}

TimedLaunch::~TimedLaunch() {
  if (start_ == nullptr) return;
  const bool recorded = cudaEventRecord(stop_, stream_) == cudaSuccess;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (recorded && g_timing_on) {
    g_records[kind_].push_back({start_, stop_});
  } else {
    cudaEventDestroy(start_);
    cudaEventDestroy(stop_);
  }
}

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status nvq_timing_enable(int on) {
  if (on != 0 && on != 1) return NVQ_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  discard_all_locked();
  g_timing_on = on != 0;
  return NVQ_OK;
}

extern "C" nvq_status nvq_timing_read(int kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= NVQ_KERNEL_KINDS || launches == nullptr || total_ms == nullptr)
    return NVQ_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  double sum = 0.0;
  for (const Interval& r : g_records[kind]) {
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e != cudaSuccess) return fail_cuda("cudaEventSynchronize (timing)", e);
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) return fail_cuda("cudaEventElapsedTime (timing)", e);
    sum += ms;
  }
  *launches = static_cast<int64_t>(g_records[kind].size());
  *total_ms = sum;
  return NVQ_OK;
}
