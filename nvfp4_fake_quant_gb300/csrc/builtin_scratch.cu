// attn_qat_bwd_builtin_scratch: the straight-through backward with its scratch
// memory taken from a fixed array that lives inside this library, for callers
// that cannot allocate device memory themselves.  Typical such callers run
// inside a host framework that owns every byte of device memory through its
// own pool and gives plug-in code no allocator, or sit on a latency-critical
// path where cudaMalloc/cudaFree would synchronize the whole device.
//
// The array (kBuiltinScratchBytes) is part of this library's device image:
// every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress, with that device current, on the first
// call made on that device (and again if the thread's current context for the
// device has changed since, e.g. after a device reset reloaded the module).
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "nvfp4attn.h"
#include "nvq_internal.h"

namespace {

constexpr size_t kBuiltinScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kBuiltinScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device and context (the
// first call per device, or per new context, performs the lookup).
nvq_status scratch_address(void** out) {
  int dev = 0;
  CUcontext ctx = nullptr;
  cudaError_t e = nvq::current_device_context(&dev, &ctx);
  if (e != cudaSuccess) return nvq::fail_cuda("bind the device's context to this thread", e);
  if (dev < 0 || dev >= kMaxDevices)
    return nvq::fail_cuda("device ordinal out of range", cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return nvq::fail_cuda("cudaGetSymbolAddress(scratch)", e);
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return NVQ_OK;
}

}  // namespace

extern "C" nvq_status attn_qat_bwd_builtin_scratch(const void* q, const void* k, const void* v,
                                                   const void* o, const float* stats,
                                                   const void* dout, void* dq, void* dk, void* dv,
                                                   int B, int Nq, int Nkv, int H, int D,
                                                   float scale, int causal, nvq_stream_t stream) {
  // The same argument checks as attn_qat_bwd, so a call gets the status that
  // call would give; only then the limit of the built-in array.
  const nvq_status chk = nvq::check_bwd_args(q, k, v, o, stats, dout, dq, dk, dv, B, Nq, Nkv, H,
                                             D, scale, causal);
  if (chk != NVQ_OK) return chk;
  const size_t need = attn_qat_bwd_workspace(B, Nq, Nkv, H, D);
  if (need == 0) return NVQ_ERR_INVALID;
  if (need > kBuiltinScratchBytes) return NVQ_ERR_WORKSPACE;  // problem too large for the array
  void* ws = nullptr;
  const nvq_status st = scratch_address(&ws);
  if (st != NVQ_OK) return st;
  // The scratch needs no clearing: the backward writes the quantized copies and
  // delta before reading them.
  return attn_qat_bwd(q, k, v, o, stats, dout, dq, dk, dv, B, Nq, Nkv, H, D, scale, causal, ws,
                      kBuiltinScratchBytes, stream);
}
