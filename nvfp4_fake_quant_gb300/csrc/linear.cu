// The NVFP4 linear of the quantization-aware recipe ("nvfp4_qad.py": nvfp4_gemm,
// _NVFP4STE): forward = both operands quantized to packed E2M1 codes with E4M3
// scales per 16 elements (128x4 tiled scale layout) under a per-tensor global
// scale, an FP4 block-scaled GEMM with alpha = 1 / (gsf_w * gsf_x), plus bias;
// backward = the full-precision linear gradients (straight-through).
//
// Every step runs in this library's kernels: the global scales, the tiled
// quantizer, the FP4 block-scaled GEMM with the alpha and bias epilogue, the two
// BF16 gradient GEMMs (one launch; gemm.cu) and the bias gradient.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"

namespace nvq {

namespace {

size_t rup(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Forward workspace, each region 256-byte aligned: packed codes and tiled scales
// of x and w, the two global scales, alpha.
struct LinWs {
  size_t cx, sx, cw, sw, gx, gw, ab, total;
};

LinWs lin_ws(int64_t M, int64_t N, int64_t K) {
  LinWs w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = rup(off + bytes, 256);
    return at;
  };
  w.cx = take(static_cast<size_t>(M) * static_cast<size_t>(K / 2));
  w.sx = take(tiled_scale_bytes(M, K));
  w.cw = take(static_cast<size_t>(N) * static_cast<size_t>(K / 2));
  w.sw = take(tiled_scale_bytes(N, K));
  w.gx = take(4);
  w.gw = take(4);
  w.ab = take(8);
  w.total = off;
  return w;
}

// alpha = 1 / (gsf_w * gsf_x) (a NULL scale counts as 1).
__global__ void alpha_kernel(const float* gx, const float* gw, float* ab) {
  const float a = (gx != nullptr ? *gx : 1.0f) * (gw != nullptr ? *gw : 1.0f);
  ab[0] = 1.0f / a;
}

// grad_b[n] = sum over m of grad[m, n] (bf16 in, fp32 sums, bf16 out).  A
// thread owns 8 consecutive columns (one 16-byte load per row) of a chunk of
// rows (blockIdx.y) and keeps four rows' loads in flight; a block's threads
// take consecutive column groups, so every row's loads are coalesced.  The
// chunks' partial sums meet in fp32 scratch by atomics, and the last chunk to
// finish a column group writes the bf16 result.  N % 8 == 0.
__global__ void __launch_bounds__(256) bias_grad_kernel(const __nv_bfloat16* __restrict__ g,
                                                        int64_t M, int64_t N,
                                                        float* __restrict__ acc,
                                                        unsigned int* __restrict__ done,
                                                        __nv_bfloat16* __restrict__ gb) {
  const int64_t c8 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  const int64_t chunk = (M + gridDim.y - 1) / gridDim.y;
  const int64_t m0 = blockIdx.y * chunk, m1 = m0 + chunk < M ? m0 + chunk : M;
  if (c8 < N) {
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16* col = g + c8;
    int64_t m = m0;
    for (; m + 4 <= m1; m += 4) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldg(reinterpret_cast<const uint4*>(col + (m + u) * N));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s[2 * k] += __uint_as_float(w[k] << 16);
          s[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
        }
      }
    }
    for (; m < m1; ++m) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(col + m * N));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s[2 * k] += __uint_as_float(w[k] << 16);
        s[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) atomicAdd(&acc[c8 + k], s[k]);
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned int last;
  if (threadIdx.x == 0) last = (atomicAdd(&done[blockIdx.x], 1u) == gridDim.y - 1) ? 1u : 0u;
  __syncthreads();
  if (last && c8 < N) {
    __threadfence();
#pragma unroll
    for (int k = 0; k < 8; ++k) gb[c8 + k] = __float2bfloat16_rn(atomicAdd(&acc[c8 + k], 0.0f));
  }
}

}  // namespace

}  // namespace nvq

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

nvq_status check_lin(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 1) return NVQ_ERR_INVALID;
  if (K % 64 != 0 || N % 16 != 0) return NVQ_ERR_UNSUPPORTED;
  return NVQ_OK;
}

nvq_status cuda_st(const char* where, cudaError_t e) {
  return e == cudaSuccess ? NVQ_OK : nvq::fail_cuda(where, e);
}

// bias gradient scratch: fp32 sums [N] and one counter per block of 2048 columns
size_t bwd_scratch(int64_t N) {
  return nvq::rup(static_cast<size_t>(N) * 4, 256) +
         nvq::rup(static_cast<size_t>((N + 2047) / 2048) * 4, 256);
}

}  // namespace

extern "C" {

size_t nvfp4_tiled_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 16 || cols % 16 != 0) return 0;
  return nvq::tiled_scale_bytes(rows, cols);
}

nvq_status nvfp4_quantize_tiled(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                const float* global_sf, uint8_t* codes, uint8_t* scales,
                                nvq_stream_t stream) {
  if (x == nullptr || !al16(x) || codes == nullptr || !al16(codes) || scales == nullptr ||
      !al16(scales))
    return NVQ_ERR_INVALID;
  if (rows < 1 || cols < 16 || cols % 16 != 0 || ld_x < cols || ld_x % 8 != 0) return NVQ_ERR_INVALID;
  if (global_sf != nullptr && (reinterpret_cast<uintptr_t>(global_sf) & 3u) != 0) return NVQ_ERR_INVALID;
  return cuda_st("quantize (tiled scales)", nvq::timed(NVQ_KERNEL_QUANTIZE, stream, [&] {
                   return nvq::launch_quant_tiled(x, rows, cols, ld_x, global_sf, codes, scales, stream);
                 }));
}

size_t nvfp4_linear_workspace(int64_t M, int64_t N, int64_t K) {
  if (check_lin(M, N, K) != NVQ_OK) return 0;
  return nvq::lin_ws(M, N, K).total;
}

nvq_status nvfp4_linear_fwd(const void* x, const void* w, const void* bias, int64_t M, int64_t N,
                            int64_t K, const float* x_global_sf, const float* w_global_sf,
                            void* out, void* ws, size_t ws_bytes, nvq_stream_t stream) {
  nvq_status st = check_lin(M, N, K);
  if (st != NVQ_OK) return st;
  if (x == nullptr || w == nullptr || out == nullptr || !al16(x) || !al16(w) || !al16(out) ||
      (bias != nullptr && !al16(bias)))
    return NVQ_ERR_INVALID;
  const float* gsfs[] = {x_global_sf, w_global_sf};
  for (const float* g : gsfs)
    if (g != nullptr && (reinterpret_cast<uintptr_t>(g) & 3u) != 0) return NVQ_ERR_INVALID;
  const nvq::LinWs L = nvq::lin_ws(M, N, K);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  uint8_t* wb = static_cast<uint8_t*>(ws);
  float* gx = reinterpret_cast<float*>(wb + L.gx);
  float* gw = reinterpret_cast<float*>(wb + L.gw);
  float* ab = reinterpret_cast<float*>(wb + L.ab);
  cudaError_t e = cudaSuccess;
  // global scales: the caller's, else 448*6/amax of the operand itself
  if (x_global_sf == nullptr)
    e = nvq::timed(NVQ_KERNEL_GLOBAL_SF, stream, [&] { return nvq::launch_global_sf(x, M, K, K, gx, stream); });
  if (e == cudaSuccess && w_global_sf == nullptr)
    e = nvq::timed(NVQ_KERNEL_GLOBAL_SF, stream, [&] { return nvq::launch_global_sf(w, N, K, K, gw, stream); });
  if (e != cudaSuccess) return nvq::fail_cuda("global scale", e);
  const float* use_gx = x_global_sf != nullptr ? x_global_sf : gx;
  const float* use_gw = w_global_sf != nullptr ? w_global_sf : gw;
  e = nvq::timed(NVQ_KERNEL_QUANTIZE, stream, [&] {
    cudaError_t r = nvq::launch_quant_tiled(x, M, K, K, use_gx, wb + L.cx, wb + L.sx, stream);
    if (r == cudaSuccess) r = nvq::launch_quant_tiled(w, N, K, K, use_gw, wb + L.cw, wb + L.sw, stream);
    return r;
  });
  if (e != cudaSuccess) return nvq::fail_cuda("quantize x, w", e);
  nvq::alpha_kernel<<<1, 1, 0, stream>>>(use_gx, use_gw, ab);
  if ((e = cudaGetLastError()) != cudaSuccess) return nvq::fail_cuda("alpha", e);
  int* err = nvq::device_error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  CUtensorMap tx, tw;
  int r;
  if ((r = nvq::make_codes_map(&tx, wb + L.cx, M, K / 2)) != 0)
    return nvq::fail_driver("cuTensorMapEncodeTiled", r);
  if (K <= nvq::kGemmFp4XresMaxK) {
    // x resident per CTA, W shared across a cluster by multicast, TMA stores
    CUtensorMap tout;
    if ((r = nvq::make_codes_map(&tw, wb + L.cw, N, K / 2, 32)) != 0 ||
        (r = nvq::make_2d_map(&tout, out, M, N, 32)) != 0)
      return nvq::fail_driver("cuTensorMapEncodeTiled", r);
    return cuda_st("fp4 gemm", nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
                     return nvq::launch_gemm_fp4_xres(tx, tw, tout, wb + L.sx, wb + L.sw, ab, bias,
                                                      M, N, K, out, err, stream);
                   }));
  }
  if ((r = nvq::make_codes_map(&tw, wb + L.cw, N, K / 2)) != 0)
    return nvq::fail_driver("cuTensorMapEncodeTiled", r);
  return cuda_st("fp4 gemm", nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
                   return nvq::launch_gemm_fp4(tx, tw, wb + L.sx, wb + L.sw, ab, bias, M, N, K, out,
                                               err, stream);
                 }));
}

size_t nvfp4_linear_bwd_workspace(int64_t M, int64_t N, int64_t K) {
  if (check_lin(M, N, K) != NVQ_OK) return 0;
  return bwd_scratch(N);
}

nvq_status nvfp4_linear_bwd(const void* grad_out, const void* x, const void* w, int64_t M,
                            int64_t N, int64_t K, void* grad_x, void* grad_w, void* grad_b,
                            void* ws, size_t ws_bytes, nvq_stream_t stream) {
  nvq_status st = check_lin(M, N, K);
  if (st != NVQ_OK) return st;
  const void* ins[] = {grad_out, x, w};
  for (const void* p : ins)
    if (p == nullptr || !al16(p)) return NVQ_ERR_INVALID;
  if ((grad_x != nullptr && !al16(grad_x)) || (grad_w != nullptr && !al16(grad_w)) ||
      (grad_b != nullptr && !al16(grad_b)))
    return NVQ_ERR_INVALID;
  const size_t need = nvfp4_linear_bwd_workspace(M, N, K);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  uint8_t* wb = static_cast<uint8_t*>(ws);
  const int col_blocks = static_cast<int>((N + 2047) / 2048);  // 256 threads x 8 columns
  float* acc = reinterpret_cast<float*>(wb);
  unsigned int* done = reinterpret_cast<unsigned int*>(wb + nvq::rup(static_cast<size_t>(N) * 4, 256));
  cudaError_t e = cudaSuccess;
  if (grad_x != nullptr || grad_w != nullptr) {
    int* err = nvq::device_error_word();
    if (err == nullptr) return NVQ_ERR_CUDA;
    // grad_w [N, K] = grad^T x: D[n, k] = sum_m grad[m, n] x[m, k], both operands
    // stored with the contraction (m) as rows (MN-major).  grad_x [M, K] = grad w:
    // D[m, k] = sum_n grad[m, n] w[n, k], grad K-major, w MN-major.  grad_w's
    // tiles (contraction M) are the long ones: they come first in the launch.
    CUtensorMap g_mn, x_mn, g_k, w_mn;
    int r;
    if ((r = nvq::make_2d_map(&g_mn, grad_out, M, N, 64)) != 0 ||
        (r = nvq::make_2d_map(&x_mn, x, M, K, 64)) != 0 ||
        (r = nvq::make_2d_map(&g_k, grad_out, M, N, 128)) != 0 ||
        (r = nvq::make_2d_map(&w_mn, w, N, K, 64)) != 0)
      return nvq::fail_driver("cuTensorMapEncodeTiled", r);
    e = nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
      return nvq::launch_gemm_bf16_pair(g_mn, x_mn, 1, 1, N, K, M, grad_w, g_k, w_mn, 0, 1, M, K,
                                        N, grad_x, err, stream);
    });
    if (e != cudaSuccess) return nvq::fail_cuda("bf16 gemms", e);
  }
  if (grad_b != nullptr) {
    e = cudaMemsetAsync(wb, 0, bwd_scratch(N), stream);
    if (e != cudaSuccess) return nvq::fail_cuda("bias gradient scratch", e);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // enough row chunks for about four blocks per SM, at least 32 rows each
    const int64_t chunks = std::max<int64_t>(
        1, std::min<int64_t>((M + 31) / 32, (4 * static_cast<int64_t>(sms) + col_blocks - 1) / col_blocks));
    e = nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
      nvq::bias_grad_kernel<<<dim3(col_blocks, static_cast<unsigned>(std::min<int64_t>(chunks, 65535))),
                              256, 0, stream>>>(static_cast<const __nv_bfloat16*>(grad_out), M, N,
                                                acc, done, static_cast<__nv_bfloat16*>(grad_b));
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return nvq::fail_cuda("bias gradient", e);
  }
  return NVQ_OK;
}

}  // extern "C"
