// C ABI of the library (declared in include/nvfp4attn.h): argument validation,
// workspace carving, TMA descriptor creation and kernel launches.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "nvfp4attn.h"
#include "nvq_internal.h"

namespace nvq {

// Device error word (see nvq_device_status).  One copy per device that loads
// the library; kernels receive its address as an argument.
static __device__ int g_error_word = 0;

namespace {

// Description of the last NVQ_ERR_CUDA returned on this host thread.
thread_local char t_error_detail[256] = "";

}  // namespace

nvq_status fail_cuda(const char* where, cudaError_t e) {
  std::snprintf(t_error_detail, sizeof(t_error_detail), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return NVQ_ERR_CUDA;
}

nvq_status fail_driver(const char* where, int cu_result) {
  std::snprintf(t_error_detail, sizeof(t_error_detail), "%s: CUresult %d", where, cu_result);
  return NVQ_ERR_CUDA;
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
CUcontext g_err_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Makes sure a CUDA context is current on the calling host thread.  A thread
// that has not yet made a CUDA call needing a context (for instance a worker
// thread of a framework that only ever touched the device through its own
// CUDA runtime) has none, and driver calls such as cuTensorMapEncodeTiled then
// fail with CUDA_ERROR_INVALID_CONTEXT.  In that case the primary context of
// the runtime's current device is made current; a context the caller made
// current is left alone.
cudaError_t bind_context(int dev) {
  CtxGetCurrentFn get = ctx_get_current_fn();
  if (get == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
  return ctx != nullptr ? cudaSuccess : cudaSetDevice(dev);
}

}  // namespace

cudaError_t current_device_context(int* dev, CUcontext* ctx) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  e = bind_context(*dev);
  if (e != cudaSuccess) return e;
  *ctx = nullptr;
  return ctx_get_current_fn()(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorInitializationError;
}

namespace {

// Address of this device's error word, after making sure a context is current
// on this thread.  Looked up with cudaGetSymbolAddress once per device and
// context (a module reloaded into a new context after a device reset lives at
// a new address).  On failure records the reason and returns nullptr.
int* error_word() {
  int dev = 0;
  CUcontext ctx = nullptr;
  cudaError_t e = current_device_context(&dev, &ctx);
  if (e != cudaSuccess) {
    fail_cuda("bind the device's context to this thread", e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    fail_cuda("device ordinal out of range", cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_ptr[dev] == nullptr || g_err_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) {
      fail_cuda("cudaGetSymbolAddress(error word)", e);
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<int*>(p);
    g_err_ctx[dev] = ctx;
  }
  return g_err_ptr[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

nvq_status from_cuda(const char* where, cudaError_t e) {
  return e == cudaSuccess ? NVQ_OK : fail_cuda(where, e);
}

}  // namespace

int make_bnhd_map(CUtensorMap* map, const void* base, int B, int N, int H, int D, bool f16,
                  int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(N) * H * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r =
      fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

int make_bnhd_u8_map(CUtensorMap* map, const void* base, int B, int N, int H, int D) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t rb = static_cast<cuuint64_t>(D) / 2;
  const cuuint64_t dims[4] = {rb, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(H) * rb, rb,
                                 static_cast<cuuint64_t>(N) * H * rb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(rb), static_cast<cuuint32_t>(kTile), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

int* device_error_word() { return error_word(); }

int make_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                   int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows),
                              1, 1};
  const cuuint64_t rs = static_cast<cuuint64_t>(row_bytes);
  const cuuint64_t strides[3] = {rs, rs * rows, rs * rows};
  const cuuint32_t box[4] = {128, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

int make_2d_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1, 1};
  const cuuint64_t rs = static_cast<cuuint64_t>(cols) * 2;
  const cuuint64_t strides[3] = {rs, rs * rows, rs * rows};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

int make_u8_map(CUtensorMap* map, const void* base, int64_t rows, int row_bytes, int64_t ld,
                int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  if (row_bytes != 32 && row_bytes != 64 && row_bytes != 128) return CUDA_ERROR_INVALID_VALUE;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows),
                              1, 1};
  const cuuint64_t rs = static_cast<cuuint64_t>(ld);
  const cuuint64_t strides[3] = {rs, rs * rows, rs * rows};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(box_rows),
                             1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                        : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

namespace {

nvq_status check_attn(int B, int Nq, int Nkv, int H, int D, float scale, int causal) {
  if (B < 1 || Nq < 1 || Nkv < 1 || H < 1) return NVQ_ERR_INVALID;
  if (!(std::isfinite(scale) && scale > 0.f)) return NVQ_ERR_INVALID;
  if (causal != 0 && causal != 1) return NVQ_ERR_INVALID;
  if (D != 64 && D != 128) return NVQ_ERR_UNSUPPORTED;
  if (causal && Nq != Nkv) return NVQ_ERR_UNSUPPORTED;
  // grid dimensions y and z are limited to 65535
  if (B > 65535 || H > 65535) return NVQ_ERR_UNSUPPORTED;
  return NVQ_OK;
}

size_t bytes_bnhd(int B, int N, int H, int D, size_t elem) {
  return static_cast<size_t>(B) * N * H * D * elem;
}

// Forward workspace: every region at its own offset (nvq_attn_layout).  Every
// form writes the quantized operands once: the packed codes of Q~ and K~ (qc,
// kc) with their scale blocks (qs, ks), V~ as f16 (v16), and Q~, K~, V~ as bf16
// (qb, kb, vb).  The forward (dense, auxiliary-output or block-sparse) reads the
// codes, their scale blocks and v16; attn_qat_bwd_saved and its block-sparse form
// read the codes and the bf16 copies.
struct FwdWs {
  size_t qc, kc, qs, ks, v16, qb, kb, vb, total;
};
FwdWs fwd_ws(int B, int Nq, int Nkv, int H, int D) {
  FwdWs w;
  w.qc = 0;
  w.kc = round_up(w.qc + bytes_bnhd(B, Nq, H, D, 1) / 2, 256);
  w.qs = round_up(w.kc + bytes_bnhd(B, Nkv, H, D, 1) / 2, 256);
  w.ks = round_up(w.qs + attn_fp4_scale_bytes(B, Nq, H, D), 256);
  w.v16 = round_up(w.ks + attn_fp4_scale_bytes(B, Nkv, H, D), 256);
  w.qb = round_up(w.v16 + bytes_bnhd(B, Nkv, H, D, 2), 256);
  w.kb = round_up(w.qb + bytes_bnhd(B, Nq, H, D, 2), 256);
  w.vb = round_up(w.kb + bytes_bnhd(B, Nkv, H, D, 2), 256);
  w.total = round_up(w.vb + bytes_bnhd(B, Nkv, H, D, 2), 256);
  return w;
}

// Backward workspace: Q~, K~, V~ (bf16), delta, the packed codes and scale
// blocks of Q~ and K~ for the FP4 S of the dQ kernel; block-sparse (topk > 0):
// also the transposed tile lists.
struct BwdWs {
  size_t q, k, v, delta, q_off, q_list, qc, kc, qs, ks, total;
};
BwdWs bwd_ws(int B, int Nq, int Nkv, int H, int D, int topk = 0) {
  BwdWs w;
  w.q = 0;
  w.k = round_up(w.q + bytes_bnhd(B, Nq, H, D, 2), 256);
  w.v = round_up(w.k + bytes_bnhd(B, Nkv, H, D, 2), 256);
  w.delta = round_up(w.v + bytes_bnhd(B, Nkv, H, D, 2), 256);
  w.qc = round_up(w.delta + static_cast<size_t>(B) * H * Nq * 4, 256);
  w.kc = round_up(w.qc + bytes_bnhd(B, Nq, H, D, 1) / 2, 256);
  w.qs = round_up(w.kc + bytes_bnhd(B, Nkv, H, D, 1) / 2, 256);
  w.ks = round_up(w.qs + attn_fp4_scale_bytes(B, Nq, H, D), 256);
  w.total = round_up(w.ks + attn_fp4_scale_bytes(B, Nkv, H, D), 256);
  w.q_off = w.q_list = w.total;
  if (topk > 0) {
    const size_t n_qt = (Nq + kTile - 1) / kTile, n_kt = (Nkv + kTile - 1) / kTile;
    w.q_off = w.total;
    w.q_list = round_up(w.q_off + static_cast<size_t>(B) * H * (n_kt + 1) * 4, 256);
    w.total = round_up(w.q_list + static_cast<size_t>(B) * H * n_qt * topk * 4, 256);
  }
  return w;
}

// Workspace of attn_qat_bwd_saved: delta only.
size_t saved_bwd_ws_bytes(int B, int Nq, int H) {
  return round_up(static_cast<size_t>(B) * H * Nq * 4, 256);
}

nvq_status check_quant(const void* x, int64_t rows, int64_t cols, int64_t ld_x) {
  if (x == nullptr || !aligned16(x)) return NVQ_ERR_INVALID;
  if (rows < 1 || cols < 16 || cols % 16 != 0) return NVQ_ERR_INVALID;
  if (ld_x < cols || ld_x % 8 != 0) return NVQ_ERR_INVALID;
  return NVQ_OK;
}

}  // namespace
// Forward; kv_list: NULL (dense) or the block-sparse key-tile lists (validated
// by the caller); o_hp: NULL or the auxiliary high-precision output (not with
// kv_list).
nvq_status fwd_impl(const void* q, const void* k, const void* v, int B, int Nq, int Nkv, int H,
                    int D, float scale, int causal, const int* kv_list, int topk, void* o,
                    void* o_hp, float* stats, void* ws, size_t ws_bytes, cudaStream_t stream) {
  nvq_status st = check_attn(B, Nq, Nkv, H, D, scale, causal);
  if (st != NVQ_OK) return st;
  if (!q || !k || !v || !o || !stats || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(o) || !aligned16(stats) || (o_hp != nullptr && !aligned16(o_hp)))
    return NVQ_ERR_INVALID;
  const FwdWs w = fwd_ws(B, Nq, Nkv, H, D);
  if (ws == nullptr || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  uint8_t* wb = static_cast<uint8_t*>(ws);
  const AttnShape s{B, Nq, Nkv, H, D, scale, causal};
  CUtensorMap mq, mk, mv;
  int r;
  cudaError_t e;
  uint8_t* qc = wb + w.qc;
  uint8_t* kc = wb + w.kc;
  uint8_t* qs = wb + w.qs;
  uint8_t* ks = wb + w.ks;
  void* v16 = wb + w.v16;
  void* qb = wb + w.qb;
  void* kb = wb + w.kb;
  void* vb = wb + w.vb;
  // Q~, K~, V~ in every form the forward and a later backward from the saved
  // operands read
  const AttnOpSpec ops[3] = {{q, Nq, qc, qs, qb, nullptr},
                             {k, Nkv, kc, ks, kb, nullptr},
                             {v, Nkv, nullptr, nullptr, vb, v16}};
  if ((e = timed(NVQ_KERNEL_QUANTIZE, stream,
                 [&] { return launch_quant_attn_ops(ops, 3, B, H, D, stream); })) != cudaSuccess)
    return fail_cuda("quantize q, k, v", e);
  // S on FP4 UMMAs: Q~ and K~ as codes + scale blocks (dense, auxiliary output
  // or block-sparse)
  if ((r = make_bnhd_u8_map(&mq, qc, B, Nq, H, D)) != 0 ||
      (r = make_bnhd_u8_map(&mk, kc, B, Nkv, H, D)) != 0 ||
      (r = make_bnhd_map(&mv, v16, B, Nkv, H, D, true)) != 0)
    return fail_driver("cuTensorMapEncodeTiled", r);
  return from_cuda("attn_fwd", timed(NVQ_KERNEL_ATTN_FWD, stream, [&] {
                     return launch_attn_fwd_fp4(s, mq, mk, mv, qs, ks, o, o_hp, stats, kv_list,
                                                topk, err, stream);
                   }));
}

// The backward's kernels on quantized operands already in device memory: qb,
// kb, vb (bf16 Q~, K~, V~) and the codes and scale blocks of Q~ and K~ (qc, kc,
// qs, ks); kv_list, q_off, q_list for the block-sparse form; delta: f32
// [B, H, Nq] scratch.
nvq_status bwd_kernels(const AttnShape& s, const void* qb, const void* kb, const void* vb,
                       const uint8_t* qc, const uint8_t* kc, const uint8_t* qs, const uint8_t* ks,
                       const void* o, const float* stats, const void* dout, const int* kv_list,
                       int topk, int* q_off, int* q_list, float* delta, void* dq, void* dk,
                       void* dv, int* err, cudaStream_t stream) {
  const int B = s.B, Nq = s.Nq, Nkv = s.Nkv, H = s.H, D = s.D;
  const int n_qt = (Nq + kTile - 1) / kTile, n_kt = (Nkv + kTile - 1) / kTile;
  CUtensorMap mq, mk, mv, mdo;
  int r;
  if ((r = make_bnhd_map(&mq, qb, B, Nq, H, D, false)) != 0 ||
      (r = make_bnhd_map(&mk, kb, B, Nkv, H, D, false)) != 0 ||
      (r = make_bnhd_map(&mv, vb, B, Nkv, H, D, false)) != 0 ||
      (r = make_bnhd_map(&mdo, dout, B, Nq, H, D, false)) != 0)
    return fail_driver("cuTensorMapEncodeTiled", r);
  cudaError_t e;
  if ((e = timed(NVQ_KERNEL_BWD_DELTA, stream,
                 [&] { return launch_bwd_prep(s, o, dout, delta, stream); })) != cudaSuccess)
    return fail_cuda("bwd_prep", e);
  if (kv_list != nullptr &&
      (e = timed(NVQ_KERNEL_VSA, stream, [&] {
         return launch_tile_transpose(kv_list, B, H, n_qt, n_kt, topk, q_off, q_list, stream);
       })) != cudaSuccess)
    return fail_cuda("tile_transpose", e);
  // both kernels form S on FP4 UMMAs from the codes and scale blocks of Q~, K~
  CUtensorMap mq4, mk4;
  if ((r = make_bnhd_u8_map(&mq4, qc, B, Nq, H, D)) != 0 ||
      (r = make_bnhd_u8_map(&mk4, kc, B, Nkv, H, D)) != 0)
    return fail_driver("cuTensorMapEncodeTiled", r);
  if ((e = timed(NVQ_KERNEL_BWD_DKDV, stream, [&] {
         return launch_attn_bwd(s, mq4, mk4, mq, mv, mdo, qs, ks, stats, delta, dk, dv, q_off,
                                q_list, n_qt * topk, err, stream);
       })) != cudaSuccess)
    return fail_cuda("attn_bwd (dK, dV)", e);
  // dQ (every key tile, or the listed ones)
  return from_cuda("attn_bwd_dq", timed(NVQ_KERNEL_BWD_DQ, stream, [&] {
                     return launch_attn_bwd_dq_fp4(s, mq4, mdo, mk4, mk, mv, qs, ks, stats, delta,
                                                   dq, kv_list, topk, err, stream);
                   }));
}

nvq_status check_bwd_args(const void* q, const void* k, const void* v, const void* o,
                          const float* stats, const void* dout, const void* dq, const void* dk,
                          const void* dv, int B, int Nq, int Nkv, int H, int D, float scale,
                          int causal) {
  nvq_status st = check_attn(B, Nq, Nkv, H, D, scale, causal);
  if (st != NVQ_OK) return st;
  const void* ptrs[] = {q, k, v, o, stats, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVQ_ERR_INVALID;
  return NVQ_OK;
}

// Straight-through backward from q, k, v: quantizes them (one launch) into the
// workspace, then runs the backward's kernels; kv_list as in fwd_impl.
nvq_status bwd_impl(const void* q, const void* k, const void* v, const void* o,
                    const float* stats, const void* dout, const int* kv_list, int topk, void* dq,
                    void* dk, void* dv, int B, int Nq, int Nkv, int H, int D, float scale,
                    int causal, void* ws, size_t ws_bytes, cudaStream_t stream) {
  nvq_status st = check_bwd_args(q, k, v, o, stats, dout, dq, dk, dv, B, Nq, Nkv, H, D, scale,
                                 causal);
  if (st != NVQ_OK) return st;
  const BwdWs w = bwd_ws(B, Nq, Nkv, H, D, kv_list != nullptr ? topk : 0);
  if (ws == nullptr || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  uint8_t* wb = static_cast<uint8_t*>(ws);
  const bool sparse = kv_list != nullptr;
  uint8_t* qc = wb + w.qc;
  uint8_t* kc = wb + w.kc;
  uint8_t* qs = wb + w.qs;
  uint8_t* ks = wb + w.ks;
  const AttnOpSpec ops[3] = {{q, Nq, qc, qs, wb + w.q, nullptr},
                             {k, Nkv, kc, ks, wb + w.k, nullptr},
                             {v, Nkv, nullptr, nullptr, wb + w.v, nullptr}};
  cudaError_t e;
  if ((e = timed(NVQ_KERNEL_QUANTIZE, stream,
                 [&] { return launch_quant_attn_ops(ops, 3, B, H, D, stream); })) != cudaSuccess)
    return fail_cuda("quantize q, k, v", e);
  const AttnShape s{B, Nq, Nkv, H, D, scale, causal};
  return bwd_kernels(s, wb + w.q, wb + w.k, wb + w.v, qc, kc, qs, ks, o, stats, dout, kv_list,
                     topk, sparse ? reinterpret_cast<int*>(wb + w.q_off) : nullptr,
                     sparse ? reinterpret_cast<int*>(wb + w.q_list) : nullptr,
                     reinterpret_cast<float*>(wb + w.delta), dq, dk, dv, err, stream);
}

// Straight-through backward from the quantized operands a dense forward left
// in its workspace (no quantizer launch).
// Backward from a forward's saved operands; kv_list (NULL: dense) and topk as
// in bwd_impl.  ws: delta, then (block-sparse) the transposed lists.
size_t saved_sparse_ws_bytes(int B, int N, int H, int topk) {
  const size_t n_t = static_cast<size_t>((N + kTile - 1) / kTile);
  const size_t off = round_up(saved_bwd_ws_bytes(B, N, H), 256);
  const size_t lst = round_up(off + static_cast<size_t>(B) * H * (n_t + 1) * 4, 256);
  return round_up(lst + static_cast<size_t>(B) * H * n_t * topk * 4, 256);
}

nvq_status bwd_saved_impl(const void* saved, size_t saved_bytes, const void* o,
                          const float* stats, const void* dout, const int* kv_list, int topk,
                          void* dq, void* dk, void* dv, int B, int Nq, int Nkv, int H, int D,
                          float scale, int causal, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  nvq_status st = check_attn(B, Nq, Nkv, H, D, scale, causal);
  if (st != NVQ_OK) return st;
  const void* ptrs[] = {o, stats, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVQ_ERR_INVALID;
  const FwdWs f = fwd_ws(B, Nq, Nkv, H, D);
  if (saved == nullptr || saved_bytes < f.total ||
      (reinterpret_cast<uintptr_t>(saved) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  const bool sparse = kv_list != nullptr;
  const size_t need = sparse ? saved_sparse_ws_bytes(B, Nq, H, topk) : saved_bwd_ws_bytes(B, Nq, H);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  const uint8_t* fb = static_cast<const uint8_t*>(saved);
  uint8_t* wb = static_cast<uint8_t*>(ws);
  const size_t off = round_up(saved_bwd_ws_bytes(B, Nq, H), 256);
  const size_t n_t = static_cast<size_t>((Nq + kTile - 1) / kTile);
  const size_t lst = round_up(off + static_cast<size_t>(B) * H * (n_t + 1) * 4, 256);
  const AttnShape s{B, Nq, Nkv, H, D, scale, causal};
  return bwd_kernels(s, fb + f.qb, fb + f.kb, fb + f.vb, fb + f.qc, fb + f.kc, fb + f.qs,
                     fb + f.ks, o, stats, dout, kv_list, topk,
                     sparse ? reinterpret_cast<int*>(wb + off) : nullptr,
                     sparse ? reinterpret_cast<int*>(wb + lst) : nullptr,
                     static_cast<float*>(ws), dq, dk, dv, err, stream);
}

}  // namespace nvq

using namespace nvq;

extern "C" {

const char* nvq_status_string(int status) {
  switch (status) {
    case NVQ_OK: return "NVQ_OK";
    case NVQ_ERR_INVALID: return "NVQ_ERR_INVALID";
    case NVQ_ERR_UNSUPPORTED: return "NVQ_ERR_UNSUPPORTED";
    case NVQ_ERR_WORKSPACE: return "NVQ_ERR_WORKSPACE";
    case NVQ_ERR_CUDA: return "NVQ_ERR_CUDA";
    case NVQ_ERR_TIMEOUT: return "NVQ_ERR_TIMEOUT";
    default: return "NVQ_ERR_UNKNOWN";
  }
}

int nvq_version(void) { return (1 << 16) | 0; }

const char* nvq_last_error_detail(void) { return t_error_detail; }

nvq_status nvq_device_status(nvq_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail_cuda("cudaStreamSynchronize", e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int));
  if (e != cudaSuccess) return fail_cuda("read error word", e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (e != cudaSuccess) return fail_cuda("clear error word", e);
    return NVQ_ERR_TIMEOUT;
  }
  return NVQ_OK;
}

nvq_status nvfp4_global_sf(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                           float* global_sf, nvq_stream_t stream) {
  if (x == nullptr || !aligned16(x) || global_sf == nullptr ||
      (reinterpret_cast<uintptr_t>(global_sf) & 3u) != 0)
    return NVQ_ERR_INVALID;
  if (rows < 1 || cols < 1 || ld_x < cols || ld_x % 8 != 0) return NVQ_ERR_INVALID;
  return from_cuda("global_sf", timed(NVQ_KERNEL_GLOBAL_SF, stream, [&] {
                     return launch_global_sf(x, rows, cols, ld_x, global_sf, stream);
                   }));
}

nvq_status nvfp4_fake_quant(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                            const float* global_sf, void* out, int64_t ld_out, uint8_t* scales,
                            int64_t ld_scales, nvq_stream_t stream) {
  nvq_status st = check_quant(x, rows, cols, ld_x);
  if (st != NVQ_OK) return st;
  if (out == nullptr || !aligned16(out) || ld_out < cols || ld_out % 8 != 0)
    return NVQ_ERR_INVALID;
  if (out == x && ld_out != ld_x) return NVQ_ERR_INVALID;
  if (scales != nullptr && ld_scales < cols / 16) return NVQ_ERR_INVALID;
  if (global_sf != nullptr && (reinterpret_cast<uintptr_t>(global_sf) & 3u) != 0)
    return NVQ_ERR_INVALID;
  const int mode = global_sf == nullptr ? kUnitBf16 : kStaticBf16;
  return from_cuda("fake_quant", timed(NVQ_KERNEL_QUANTIZE, stream, [&] {
                     return launch_fake_quant(x, rows, cols, ld_x, global_sf, mode, out, ld_out,
                                              scales, ld_scales, nullptr, 0, stream);
                   }));
}

nvq_status nvfp4_quantize_codes(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                const float* global_sf, uint8_t* codes, int64_t ld_codes,
                                uint8_t* scales, int64_t ld_scales, nvq_stream_t stream) {
  nvq_status st = check_quant(x, rows, cols, ld_x);
  if (st != NVQ_OK) return st;
  if (codes == nullptr || !aligned16(codes) || ld_codes < cols / 2 || ld_codes % 8 != 0)
    return NVQ_ERR_INVALID;
  if (scales == nullptr || ld_scales < cols / 16) return NVQ_ERR_INVALID;
  if (global_sf != nullptr && (reinterpret_cast<uintptr_t>(global_sf) & 3u) != 0)
    return NVQ_ERR_INVALID;
  const int mode = global_sf == nullptr ? kUnitBf16 : kStaticBf16;
  return from_cuda("quantize_codes", timed(NVQ_KERNEL_QUANTIZE, stream, [&] {
                     return launch_fake_quant(x, rows, cols, ld_x, global_sf, mode, nullptr, 0,
                                              scales, ld_scales, codes, ld_codes, stream);
                   }));
}

size_t attn_qat_fwd_workspace(int B, int Nq, int Nkv, int H, int D) {
  if (B < 1 || Nq < 1 || Nkv < 1 || H < 1 || D < 1) return 0;
  return fwd_ws(B, Nq, Nkv, H, D).total;
}

size_t attn_qat_bwd_workspace(int B, int Nq, int Nkv, int H, int D) {
  if (B < 1 || Nq < 1 || Nkv < 1 || H < 1 || D < 1) return 0;
  return bwd_ws(B, Nq, Nkv, H, D).total;
}

nvq_status attn_qat_fwd_layout(int B, int Nq, int Nkv, int H, int D, nvq_attn_layout* out) {
  if (out == nullptr || B < 1 || Nq < 1 || Nkv < 1 || H < 1 || (D != 64 && D != 128))
    return NVQ_ERR_INVALID;
  const FwdWs w = fwd_ws(B, Nq, Nkv, H, D);
  *out = nvq_attn_layout{w.qc, w.kc, w.qs, w.ks, w.v16, w.qb, w.kb, w.vb, SIZE_MAX, w.total};
  return NVQ_OK;
}

nvq_status attn_qat_bwd_layout(int B, int Nq, int Nkv, int H, int D, nvq_attn_layout* out) {
  if (out == nullptr || B < 1 || Nq < 1 || Nkv < 1 || H < 1 || (D != 64 && D != 128))
    return NVQ_ERR_INVALID;
  const BwdWs w = bwd_ws(B, Nq, Nkv, H, D);
  *out = nvq_attn_layout{w.qc, w.kc, w.qs, w.ks, SIZE_MAX, w.q, w.k, w.v, w.delta, w.total};
  return NVQ_OK;
}

nvq_status attn_qat_fwd(const void* q, const void* k, const void* v, int B, int Nq, int Nkv,
                        int H, int D, float scale, int causal, void* o, float* stats, void* ws,
                        size_t ws_bytes, nvq_stream_t stream) {
  return fwd_impl(q, k, v, B, Nq, Nkv, H, D, scale, causal, nullptr, 0, o, nullptr, stats, ws,
                  ws_bytes, stream);
}

nvq_status attn_qat_fwd_hp(const void* q, const void* k, const void* v, int B, int Nq, int Nkv,
                           int H, int D, float scale, int causal, void* o, void* o_hp,
                           float* stats, void* ws, size_t ws_bytes, nvq_stream_t stream) {
  if (o_hp == nullptr) return NVQ_ERR_INVALID;
  return fwd_impl(q, k, v, B, Nq, Nkv, H, D, scale, causal, nullptr, 0, o, o_hp, stats, ws,
                  ws_bytes, stream);
}

nvq_status attn_qat_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* stats, const void* dout, void* dq, void* dk, void* dv, int B,
                        int Nq, int Nkv, int H, int D, float scale, int causal, void* ws,
                        size_t ws_bytes, nvq_stream_t stream) {
  return bwd_impl(q, k, v, o, stats, dout, nullptr, 0, dq, dk, dv, B, Nq, Nkv, H, D, scale, causal,
                  ws, ws_bytes, stream);
}

size_t attn_qat_bwd_saved_workspace(int B, int Nq, int Nkv, int H, int D) {
  if (B < 1 || Nq < 1 || Nkv < 1 || H < 1 || D < 1) return 0;
  return saved_bwd_ws_bytes(B, Nq, H);
}

nvq_status attn_qat_bwd_saved(const void* saved, size_t saved_bytes, const void* o,
                              const float* stats, const void* dout, void* dq, void* dk, void* dv,
                              int B, int Nq, int Nkv, int H, int D, float scale, int causal,
                              void* ws, size_t ws_bytes, nvq_stream_t stream) {
  return bwd_saved_impl(saved, saved_bytes, o, stats, dout, nullptr, 0, dq, dk, dv, B, Nq, Nkv,
                        H, D, scale, causal, ws, ws_bytes, stream);
}

// Block-sparse: N % 128 == 0 (whole tiles), 1 <= topk <= N / 128, an int32
// list [B, H, N/128, topk], non-causal.
static nvq_status check_sparse(int N, int topk, const int32_t* kv_tiles) {
  if (N < 1 || N % kTile != 0 || topk < 1 || topk > N / kTile) return NVQ_ERR_INVALID;
  if (kv_tiles == nullptr || (reinterpret_cast<uintptr_t>(kv_tiles) & 3u) != 0)
    return NVQ_ERR_INVALID;
  return NVQ_OK;
}

size_t attn_qat_bwd_sparse_workspace(int B, int N, int H, int D, int topk) {
  if (B < 1 || N < 1 || H < 1 || D < 1 || topk < 1) return 0;
  return bwd_ws(B, N, N, H, D, topk).total;
}

nvq_status attn_qat_fwd_sparse(const void* q, const void* k, const void* v, int B, int N, int H,
                               int D, float scale, const int32_t* kv_tiles, int topk, void* o,
                               float* stats, void* ws, size_t ws_bytes, nvq_stream_t stream) {
  const nvq_status st = check_sparse(N, topk, kv_tiles);
  if (st != NVQ_OK) return st;
  return fwd_impl(q, k, v, B, N, N, H, D, scale, 0, kv_tiles, topk, o, nullptr, stats, ws,
                  ws_bytes, stream);
}

nvq_status attn_qat_bwd_sparse(const void* q, const void* k, const void* v, const void* o,
                               const float* stats, const void* dout, const int32_t* kv_tiles,
                               int topk, void* dq, void* dk, void* dv, int B, int N, int H, int D,
                               float scale, void* ws, size_t ws_bytes, nvq_stream_t stream) {
  const nvq_status st = check_sparse(N, topk, kv_tiles);
  if (st != NVQ_OK) return st;
  return bwd_impl(q, k, v, o, stats, dout, kv_tiles, topk, dq, dk, dv, B, N, N, H, D, scale, 0, ws,
                  ws_bytes, stream);
}

size_t attn_qat_bwd_sparse_saved_workspace(int B, int N, int H, int D, int topk) {
  if (B < 1 || N < 1 || H < 1 || D < 1 || topk < 1) return 0;
  return saved_sparse_ws_bytes(B, N, H, topk);
}

nvq_status attn_qat_bwd_sparse_saved(const void* saved, size_t saved_bytes, const void* o,
                                     const float* stats, const void* dout,
                                     const int32_t* kv_tiles, int topk, void* dq, void* dk,
                                     void* dv, int B, int N, int H, int D, float scale, void* ws,
                                     size_t ws_bytes, nvq_stream_t stream) {
  const nvq_status st = check_sparse(N, topk, kv_tiles);
  if (st != NVQ_OK) return st;
  return bwd_saved_impl(saved, saved_bytes, o, stats, dout, kv_tiles, topk, dq, dk, dv, B, N, N,
                        H, D, scale, 0, ws, ws_bytes, stream);
}

nvq_status vsa_reorder(const void* x, int B, int T, int Hh, int W, int H, int D, int ct, int ch,
                       int cw, int to_cubes, void* out, nvq_stream_t stream) {
  if (!x || !out || x == out || !aligned16(x) || !aligned16(out)) return NVQ_ERR_INVALID;
  if (B < 1 || T < 1 || Hh < 1 || W < 1 || H < 1 || D < 1 || ct < 1 || ch < 1 || cw < 1)
    return NVQ_ERR_INVALID;
  if (T % ct || Hh % ch || W % cw || (static_cast<int64_t>(H) * D) % 8 != 0 ||
      (to_cubes != 0 && to_cubes != 1))
    return NVQ_ERR_INVALID;
  return from_cuda("vsa_reorder", timed(NVQ_KERNEL_VSA, stream, [&] {
                     return launch_vsa_reorder(x, B, T, Hh, W, H, D, ct, ch, cw, to_cubes, out,
                                               stream);
                   }));
}

size_t vsa_select_workspace(int B, int N, int H, int D) {
  if (B < 1 || N < kTile || N % kTile != 0 || H < 1 || D < 1) return 0;
  return 2 * round_up(static_cast<size_t>(B) * H * (N / kTile) * D * 4, 256);
}

nvq_status vsa_select_tiles(const void* q, const void* k, int B, int N, int H, int D, int topk,
                            int32_t* kv_tiles, void* ws, size_t ws_bytes, nvq_stream_t stream) {
  if (!q || !k || !kv_tiles || !aligned16(q) || !aligned16(k) ||
      (reinterpret_cast<uintptr_t>(kv_tiles) & 3u) != 0)
    return NVQ_ERR_INVALID;
  if (B < 1 || H < 1 || D < 1 || D > 1024 || N < kTile || N % kTile != 0 || topk < 1 ||
      topk > N / kTile)
    return NVQ_ERR_INVALID;
  const size_t need = vsa_select_workspace(B, N, H, D);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return NVQ_ERR_WORKSPACE;
  float* qm = static_cast<float*>(ws);
  float* km = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + need / 2);
  return from_cuda("vsa_select", timed(NVQ_KERNEL_VSA, stream, [&] {
                     return launch_vsa_select(q, k, B, N, H, D, topk, kv_tiles, qm, km, stream);
                   }));
}

nvq_status nvq_selftest_umma(const void* a, const void* b, float* c, int N, int K, int a_mn,
                             int b_mn, nvq_stream_t stream) {
  if (!a || !b || !c || !aligned16(a) || !aligned16(b) || !aligned16(c)) return NVQ_ERR_INVALID;
  if ((N != 64 && N != 128) || (K != 64 && K != 128) || a_mn < 0 || a_mn > 2 ||
      (b_mn != 0 && b_mn != 1))
    return NVQ_ERR_INVALID;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  CUtensorMap ma, mb;
  int r;
  if ((r = a_mn == 1 ? make_2d_map(&ma, a, K, 128, K) : make_2d_map(&ma, a, 128, K, 128)) != 0 ||
      (r = b_mn ? make_2d_map(&mb, b, K, N, K) : make_2d_map(&mb, b, N, K, N)) != 0)
    return fail_driver("cuTensorMapEncodeTiled", r);
  return from_cuda("selftest_umma",
                   launch_selftest_umma(ma, mb, a, c, N, K, a_mn, b_mn, err, stream));
}

nvq_status nvq_selftest_fp4(const void* a, const void* b, const uint32_t* sf_img,
                            const uint8_t* sf_src, float* c, uint32_t* dump, int N, int nmma,
                            int sf_stride, int mode, nvq_stream_t stream) {
  if (!a || !b || !c || !dump || !aligned16(a) || !aligned16(b) || !aligned16(c) ||
      !aligned16(dump))
    return NVQ_ERR_INVALID;
  if ((N != 64 && N != 128) || (nmma != 1 && nmma != 2 && nmma != 4) || sf_stride < 0 ||
      sf_stride > 4 ||
      (mode != 0 && mode != 1) || (mode == 0 && !sf_img) || (mode == 1 && !sf_src))
    return NVQ_ERR_INVALID;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  CUtensorMap ma, mb;
  int r;
  if ((r = make_u8_map(&ma, a, 128, 32 * nmma, 32 * nmma, 128)) != 0 ||
      (r = make_u8_map(&mb, b, N, 32 * nmma, 32 * nmma, N)) != 0)
    return fail_driver("cuTensorMapEncodeTiled", r);
  return from_cuda("selftest_fp4", launch_selftest_fp4(ma, mb, sf_img, sf_src, c, dump, N, nmma,
                                                       sf_stride, mode, err, stream));
}

nvq_status nvq_selftest_ex2_monotone(unsigned long long* out, nvq_stream_t stream) {
  if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 7u) != 0) return NVQ_ERR_INVALID;
  return from_cuda("selftest_ex2_monotone",
                   launch_selftest_ex2_monotone(out, static_cast<cudaStream_t>(stream)));
}

nvq_status nvq_selftest_timeout(int64_t limit_ns, nvq_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 1000000000) return NVQ_ERR_INVALID;
  int* err = error_word();
  if (err == nullptr) return NVQ_ERR_CUDA;
  return from_cuda("selftest_timeout", launch_selftest_timeout(limit_ns, err, stream));
}

}  // extern "C"
