// The NVFP4 linear of the quantization-aware recipe ("nvfp4_qad.py": nvfp4_gemm,
// _NVFP4STE): forward = both operands quantized to packed E2M1 codes with E4M3
// scales per 16 elements (128x4 tiled scale layout) under a per-tensor global
// scale, an FP4 block-scaled GEMM with alpha = 1 / (gsf_w * gsf_x), plus bias;
// backward = the full-precision linear gradients (straight-through).
//
// The quantizers, the global scales and the bias gradient are this library's
// kernels; the GEMMs are cuBLASLt's (FP4 block-scaled forward, BF16 backward):
// plain library GEMMs with nothing fused into them but the bias epilogue.
#include <algorithm>
#include <map>
#include <mutex>

#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"

namespace nvq {

namespace {

constexpr int kMaxDev = 64;
constexpr size_t kGemmWs = 32u << 20;  // cuBLASLt workspace inside the caller's buffer

size_t rup(size_t v, size_t a) { return (v + a - 1) / a * a; }

// One cuBLASLt handle per device, created on first use.
cublasLtHandle_t lt_handle(int dev) {
  static std::mutex mu;
  static cublasLtHandle_t h[kMaxDev] = {};
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (h[dev] == nullptr && cublasLtCreate(&h[dev]) != CUBLAS_STATUS_SUCCESS) h[dev] = nullptr;
  return h[dev];
}

// Forward workspace, each region 256-byte aligned: packed codes and tiled scales
// of x and w, the two global scales, alpha and beta, the GEMM workspace.
struct LinWs {
  size_t cx, sx, cw, sw, gx, gw, ab, gemm, total;
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
  w.gemm = take(kGemmWs);
  w.total = off;
  return w;
}

// alpha = 1 / (gsf_w * gsf_x) (a NULL scale counts as 1), beta = 0.
__global__ void alpha_kernel(const float* gx, const float* gw, float* ab) {
  const float a = (gx != nullptr ? *gx : 1.0f) * (gw != nullptr ? *gw : 1.0f);
  ab[0] = 1.0f / a;
  ab[1] = 0.0f;
}

// grad_b[n] = sum over m of grad[m, n] (bf16 in, fp32 sums, bf16 out).  Threads
// of a block take consecutive columns (coalesced rows); blockIdx.y splits the
// rows into chunks whose partial sums meet in fp32 scratch; the last chunk to
// finish a column group writes the bf16 result.
__global__ void __launch_bounds__(256) bias_grad_kernel(const __nv_bfloat16* __restrict__ g,
                                                        int64_t M, int64_t N,
                                                        float* __restrict__ acc,
                                                        unsigned int* __restrict__ done,
                                                        __nv_bfloat16* __restrict__ gb) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t chunk = (M + gridDim.y - 1) / gridDim.y;
  const int64_t m0 = blockIdx.y * chunk, m1 = m0 + chunk < M ? m0 + chunk : M;
  if (n < N) {
    float s = 0.f;
    for (int64_t m = m0; m < m1; ++m) s += __bfloat162float(g[m * N + n]);
    atomicAdd(&acc[n], s);
  }
  __threadfence();
  __syncthreads();
  __shared__ unsigned int last;
  if (threadIdx.x == 0) last = (atomicAdd(&done[blockIdx.x], 1u) == gridDim.y - 1) ? 1u : 0u;
  __syncthreads();
  if (last && n < N) {
    __threadfence();
    gb[n] = __float2bfloat16_rn(atomicAdd(&acc[n], 0.0f));
  }
}

// One cuBLASLt GEMM D = alpha op(A) op(B) (+ bias per row of D), column-major
// as cuBLASLt sees it: D is m x n with leading dimension ldd; A is stored m x k
// (op N) or k x m (op T), B k x n (op N) or n x k (op T).  alpha and beta are
// device pointers (ab[0], ab[1]).  block_scaled: A and B are packed E2M1 with
// E4M3 scales per 16 elements in the 128x4 tiled layout.
struct Gemm {
  cublasOperation_t ta, tb;
  cudaDataType_t ab_type;
  int64_t m, n, k, lda, ldb, ldd;
  bool block_scaled;
};

struct AlgoKey {
  int ta, tb, type, bias;
  int64_t m, n, k, lda, ldb, ldd;
  bool operator<(const AlgoKey& o) const {
    const int64_t a[] = {ta, tb, type, bias, m, n, k, lda, ldb, ldd};
    const int64_t b[] = {o.ta, o.tb, o.type, o.bias, o.m, o.n, o.k, o.lda, o.ldb, o.ldd};
    return std::lexicographical_compare(a, a + 10, b, b + 10);
  }
};

// NVQ_OK, NVQ_ERR_UNSUPPORTED (no cuBLASLt algorithm for the problem) or
// NVQ_ERR_CUDA with the failing step recorded.
nvq_status run_gemm(const Gemm& g, const void* A, const void* B, void* D, const void* a_scale,
                    const void* b_scale, const float* ab, const void* bias, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail_cuda("cudaGetDevice", cudaErrorInvalidDevice);
  cublasLtHandle_t h = lt_handle(dev);
  if (h == nullptr) return fail_cuda("cublasLtCreate", cudaErrorInitializationError);
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  nvq_status st = NVQ_OK;
  const char* where = nullptr;
  auto chk = [&](cublasStatus_t r, const char* w) {
    if (r != CUBLAS_STATUS_SUCCESS && where == nullptr) where = w;
    return r == CUBLAS_STATUS_SUCCESS;
  };
  const cublasLtPointerMode_t pm = CUBLASLT_POINTER_MODE_DEVICE;
  const cublasLtMatmulMatrixScale_t sm = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
  const cublasLtEpilogue_t epi = CUBLASLT_EPILOGUE_BIAS;
  const cudaDataType_t bias_t = CUDA_R_16BF;
  const uint64_t wsb = ws_bytes;
  bool ok = chk(cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F), "matmul desc") &&
            chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &g.ta, sizeof(g.ta)), "transa") &&
            chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &g.tb, sizeof(g.tb)), "transb") &&
            chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_POINTER_MODE, &pm, sizeof(pm)), "pointer mode");
  if (ok && g.block_scaled)
    ok = chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &sm, sizeof(sm)), "a scale mode") &&
         chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &sm, sizeof(sm)), "b scale mode") &&
         chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &a_scale, sizeof(a_scale)), "a scales") &&
         chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &b_scale, sizeof(b_scale)), "b scales");
  if (ok && bias != nullptr)
    ok = chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_EPILOGUE, &epi, sizeof(epi)), "epilogue") &&
         chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)), "bias") &&
         chk(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_DATA_TYPE, &bias_t, sizeof(bias_t)), "bias type");
  const bool at = g.ta == CUBLAS_OP_T, bt = g.tb == CUBLAS_OP_T;
  if (ok)
    ok = chk(cublasLtMatrixLayoutCreate(&la, g.ab_type, at ? g.k : g.m, at ? g.m : g.k, g.lda), "layout a") &&
         chk(cublasLtMatrixLayoutCreate(&lb, g.ab_type, bt ? g.n : g.k, bt ? g.k : g.n, g.ldb), "layout b") &&
         chk(cublasLtMatrixLayoutCreate(&ld, CUDA_R_16BF, g.m, g.n, g.ldd), "layout d") &&
         chk(cublasLtMatmulPreferenceCreate(&pref), "preference") &&
         chk(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)), "workspace pref");
  if (ok) {
    static std::mutex mu;
    static std::map<AlgoKey, cublasLtMatmulAlgo_t> cache;
    const AlgoKey key{static_cast<int>(g.ta), static_cast<int>(g.tb), static_cast<int>(g.ab_type),
                      bias != nullptr ? 1 : 0, g.m, g.n, g.k, g.lda, g.ldb, g.ldd};
    cublasLtMatmulAlgo_t algo;
    bool have = false;
    {
      std::lock_guard<std::mutex> lock(mu);
      auto it = cache.find(key);
      if (it != cache.end()) {
        algo = it->second;
        have = true;
      }
    }
    if (!have) {
      cublasLtMatmulHeuristicResult_t res{};
      int count = 0;
      if (cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, ld, ld, pref, 1, &res, &count) !=
              CUBLAS_STATUS_SUCCESS ||
          count < 1) {
        st = NVQ_ERR_UNSUPPORTED;
        ok = false;
      } else {
        algo = res.algo;
        std::lock_guard<std::mutex> lock(mu);
        cache[key] = algo;
      }
    }
    if (ok)
      ok = chk(cublasLtMatmul(h, op, ab, A, la, B, lb, ab + 1, D, ld, D, ld, &algo, ws, ws_bytes, stream),
               "cublasLtMatmul");
  }
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (ld) cublasLtMatrixLayoutDestroy(ld);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  if (st != NVQ_OK) return st;
  if (!ok) return fail_cuda(where != nullptr ? where : "cuBLASLt", cudaErrorUnknown);
  return NVQ_OK;
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

size_t bwd_scratch(int64_t N) { return nvq::rup(static_cast<size_t>(N) * 4, 256) + nvq::rup(static_cast<size_t>((N + 255) / 256) * 4, 256); }

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
  // out [M, N] row-major = column-major N x M: D = W (op T of the stored K x N)
  // times X (op N of the stored K x M)
  const nvq::Gemm g{CUBLAS_OP_T, CUBLAS_OP_N, CUDA_R_4F_E2M1, N, M, K, K, K, N, true};
  nvq_status gs = NVQ_OK;
  nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
    gs = nvq::run_gemm(g, wb + L.cw, wb + L.cx, out, wb + L.sw, wb + L.sx, ab, bias, wb + L.gemm,
                       nvq::kGemmWs, stream);
    return gs == NVQ_OK ? cudaSuccess : cudaErrorUnknown;
  });
  return gs;
}

size_t nvfp4_linear_bwd_workspace(int64_t M, int64_t N, int64_t K) {
  if (check_lin(M, N, K) != NVQ_OK) return 0;
  return bwd_scratch(N) + 256 + nvq::kGemmWs;
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
  const int col_blocks = static_cast<int>((N + 255) / 256);
  float* acc = reinterpret_cast<float*>(wb);
  unsigned int* done = reinterpret_cast<unsigned int*>(wb + nvq::rup(static_cast<size_t>(N) * 4, 256));
  float* ab = reinterpret_cast<float*>(wb + bwd_scratch(N));
  void* gemm_ws = wb + bwd_scratch(N) + 256;
  nvq::alpha_kernel<<<1, 1, 0, stream>>>(nullptr, nullptr, ab);  // alpha 1, beta 0
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return nvq::fail_cuda("alpha", e);
  nvq_status gs = NVQ_OK;
  e = nvq::timed(NVQ_KERNEL_LINEAR, stream, [&] {
    // grad_x [M, K] = grad [M, N] W [N, K]: column-major K x M = W^T (stored K x N)
    // times grad^T (stored N x M)
    if (grad_x != nullptr) {
      const nvq::Gemm g{CUBLAS_OP_N, CUBLAS_OP_N, CUDA_R_16BF, K, M, N, K, N, K, false};
      gs = nvq::run_gemm(g, w, grad_out, grad_x, nullptr, nullptr, ab, nullptr, gemm_ws,
                         nvq::kGemmWs, stream);
    }
    // grad_w [N, K] = grad^T X: column-major K x N = X^T (stored K x M) times
    // (grad^T stored N x M, transposed)
    if (gs == NVQ_OK && grad_w != nullptr) {
      const nvq::Gemm g{CUBLAS_OP_N, CUBLAS_OP_T, CUDA_R_16BF, K, N, M, K, N, K, false};
      gs = nvq::run_gemm(g, x, grad_out, grad_w, nullptr, nullptr, ab, nullptr, gemm_ws,
                         nvq::kGemmWs, stream);
    }
    return gs == NVQ_OK ? cudaSuccess : cudaErrorUnknown;
  });
  if (gs != NVQ_OK) return gs;
  if (grad_b != nullptr) {
    e = cudaMemsetAsync(wb, 0, bwd_scratch(N), stream);
    if (e != cudaSuccess) return nvq::fail_cuda("bias gradient scratch", e);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t chunks = std::max<int64_t>(
        1, std::min<int64_t>((M + 63) / 64, (4 * static_cast<int64_t>(sms) + col_blocks - 1) / col_blocks));
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
