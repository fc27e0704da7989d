// Host-side declarations shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Every launch_* function enqueues kernels on `stream` and
// returns the launch's cudaError_t; validation happens in api.cu before.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "nvfp4attn.h"

namespace nvq {

constexpr int kTile = 128;  // query / key rows per attention tile

// Quantizer output modes.
enum QuantMode : int { kUnitBf16 = 0, kUnitF16 = 1, kStaticBf16 = 2 };

cudaError_t launch_fake_quant(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const float* gsf, int mode, void* out, int64_t ld_out,
                              uint8_t* scales, int64_t ld_s, uint8_t* codes, int64_t ld_c,
                              cudaStream_t stream);
// Packed E2M1 codes (row-major, cols/2 bytes a row) and E4M3 scales in the 128x4
// tiled layout of block-scaled FP4 GEMMs (tiled_scale_bytes(rows, cols) bytes,
// padding zeroed); gsf NULL = unit global scale.
size_t tiled_scale_bytes(int64_t rows, int64_t cols);
cudaError_t launch_quant_tiled(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               const float* gsf, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream);
// Q or K of attention for the FP4 UMMA: packed E2M1 codes [B, N, H, D/2] and
// E4M3 scales in per-(b, h, 128-token tile, 64-element group) 512-byte blocks in
// the UMMA's tensor-memory scale layout (attn_fp4_scale_bytes(B, N, H, D)).
size_t attn_fp4_scale_bytes(int B, int N, int H, int D);
cudaError_t launch_quant_attn_fp4(const void* x, int B, int N, int H, int D, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t stream);
// One attention operand x bf16 [B, N, H, D] (contiguous) and the forms to write
// (each may be null): packed codes [B, N, H, D/2] and scale blocks (the layout
// of launch_quant_attn_fp4), fake-quantized bf16 and f16 copies [B, N, H, D].
struct AttnOpSpec {
  const void* x;
  int N;
  uint8_t* codes;
  uint8_t* scales;
  void* bf16;
  void* f16;
};
// Device form of AttnOpSpec (quant.cu).
struct AttnOpJob {
  const uint16_t* x;
  uint8_t* codes;
  uint8_t* scales;
  uint16_t* bf16;
  uint16_t* f16;
  uint32_t nblocks, npad, N, n_tiles;
};
struct AttnOpJobs {
  AttnOpJob j[3];
  uint32_t H, lg_nbd;
};
// Quantizes `count` (1..3) operands with the same B, H, D (unit global scale)
// in one launch; D in {64, 128}.
cudaError_t launch_quant_attn_ops(const AttnOpSpec* specs, int count, int B, int H, int D,
                                  cudaStream_t stream);
cudaError_t launch_global_sf(const void* x, int64_t rows, int64_t cols, int64_t ld_x, float* gsf,
                             cudaStream_t stream);

struct AttnShape {
  int B, Nq, Nkv, H, D;
  float scale;
  int causal;
};

// Record "where: CUDA error" as this host thread's error detail (returned by
// nvq_last_error_detail) and return NVQ_ERR_CUDA.
nvq_status fail_cuda(const char* where, cudaError_t e);
nvq_status fail_driver(const char* where, int cu_result);

// The current device and the context current on this thread; a thread with no
// current context first gets the device's primary context made current.
cudaError_t current_device_context(int* dev, CUcontext* ctx);

// The host-side argument checks of attn_qat_bwd (sizes, scale, causal flag,
// null and misaligned pointers), in the order that call applies them.
nvq_status check_bwd_args(const void* q, const void* k, const void* v, const void* o,
                          const float* stats, const void* dout, const void* dq, const void* dk,
                          const void* dv, int B, int Nq, int Nkv, int H, int D, float scale,
                          int causal);

// While nvq_timing_enable(1) is in force, brackets the launches made during its
// lifetime with CUDA events on `stream`, filed under `kind` (an NVQ_KERNEL_*
// value); otherwise does nothing.
class TimedLaunch {
 public:
  TimedLaunch(int kind, cudaStream_t stream);
  ~TimedLaunch();
  TimedLaunch(const TimedLaunch&) = delete;
  TimedLaunch& operator=(const TimedLaunch&) = delete;

 private:
  int kind_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr, stop_ = nullptr;
};

// Runs `launch` (a callable returning cudaError_t) inside a TimedLaunch.
template <class F>
cudaError_t timed(int kind, cudaStream_t stream, F&& launch) {
  TimedLaunch t(kind, stream);
  return launch();
}

// Tensor map over packed E2M1 codes [B, N, H, D/2] (bytes), box {D/2, 128, 1, 1},
// with the (D/2)-byte swizzle; D in {64, 128}.
int make_bnhd_u8_map(CUtensorMap* map, const void* base, int B, int N, int H, int D);
// Tensor maps over [B, N, H, D] 16-bit tensors, box {64, box_rows, 1, 1}, 128-byte swizzle.
// Return the CUresult of cuTensorMapEncodeTiled (0 on success).
int make_bnhd_map(CUtensorMap* map, const void* base, int B, int N, int H, int D, bool f16,
                   int box_rows = kTile);

// Forward with S on FP4 UMMAs: tq, tk map the packed codes of Q~ and K~
// (make_bnhd_u8_map), q_sc, k_sc their scale blocks (launch_quant_attn_fp4),
// tv the f16 V~ (make_bnhd_map).  At most one of: o_hp, the auxiliary output
// P V~ / l (bf16, layout of o); kv_list, the block-sparse key tiles, int32
// [B, H, ceil(Nq/128), topk], entries in [0, ceil(Nkv/128)) (N % 128 == 0,
// non-causal).
cudaError_t launch_attn_fwd_fp4(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                                void* o, void* o_hp, float* stats, const int* kv_list, int topk,
                                int* err, cudaStream_t stream);
cudaError_t launch_bwd_prep(const AttnShape& s, const void* o, const void* dout, float* delta,
                            cudaStream_t stream);
// dK, dV (key-outer; Q~, K~, V~, dO maps with 128-row boxes).  Block-sparse:
// q_off/q_list from launch_tile_transpose (q_stride = n_qt * topk), else NULL.
cudaError_t launch_attn_bwd(const AttnShape& s, const CUtensorMap& tq4, const CUtensorMap& tk4,
                            const CUtensorMap& tq, const CUtensorMap& tv, const CUtensorMap& tdo,
                            const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                            const float* delta, void* dk, void* dv, const int* q_off,
                            const int* q_list, int q_stride, int* err, cudaStream_t stream);
// Block-sparse lists [B, H, n_qt, topk] transposed to, per (b, h), offsets
// q_off [n_kt + 1] and ascending query tiles q_list [n_qt * topk].
cudaError_t launch_tile_transpose(const int* kv_list, int B, int H, int n_qt, int n_kt, int topk,
                                  int* q_off, int* q_list, cudaStream_t stream);
// dQ with S on FP4 UMMAs: tq4, tk4 map the packed codes of Q~ and K~
// (make_bnhd_u8_map), q_sc, k_sc their scale blocks; tdo, tk, tv the bf16 dO,
// K~, V~ (128-row boxes).  kv_list: NULL (dense) or the block-sparse key-tile
// lists [B, H, ceil(Nq/128), topk].
cudaError_t launch_attn_bwd_dq_fp4(const AttnShape& s, const CUtensorMap& tq4,
                                   const CUtensorMap& tdo, const CUtensorMap& tk4,
                                   const CUtensorMap& tk, const CUtensorMap& tv,
                                   const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                                   const float* delta, void* dq, const int* kv_list, int topk,
                                   int* err, cudaStream_t stream);

// Token rows [B, T*Hh*W, H, D] (bf16) between raster and cube order.
cudaError_t launch_vsa_reorder(const void* x, int B, int T, int Hh, int W, int H, int D, int ct,
                               int ch, int cw, int to_cubes, void* out, cudaStream_t stream);
// Top-k key tiles per query tile by cube-mean scores; qm, km: f32 [B, H, N/128, D] scratch.
cudaError_t launch_vsa_select(const void* q, const void* k, int B, int N, int H, int D, int topk,
                              int* kv_tiles, float* qm, float* km, cudaStream_t stream);

cudaError_t launch_selftest_umma(const CUtensorMap& ta, const CUtensorMap& tb, const void* a,
                                 float* c, int N, int K, int a_mn, int b_mn, int* err,
                                 cudaStream_t stream);
cudaError_t launch_selftest_timeout(int64_t limit_ns, int* err, cudaStream_t stream);
cudaError_t launch_selftest_ex2_monotone(unsigned long long* out, cudaStream_t stream);
cudaError_t launch_selftest_fp4(const CUtensorMap& ta, const CUtensorMap& tb, const uint32_t* sf_img,
                                const uint8_t* sf_src, float* c, uint32_t* dump, int N, int nmma,
                                int sf_stride, int mode, int* err, cudaStream_t stream);

// Address of the current device's error word (see nvq_device_status), or
// nullptr with the failure recorded.
int* device_error_word();
// Maps packed E2M1 codes [rows, row_bytes] (contiguous) with a box of 128 bytes
// x box_rows rows and the 128-byte swizzle.
int make_codes_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes,
                   int box_rows = 128);

// The NVFP4 linear's GEMMs (gemm.cu).
// out [M, N] bf16 = alpha * (x codes . x scales)(w codes . w scales)^T + bias:
// tx, tw from make_codes_map over [M, K/2] and [N, K/2]; sx, sw the tiled scales;
// alpha a device scalar; bias bf16 [N] or nullptr.  K % 64 == 0, N % 8 == 0.
cudaError_t launch_gemm_fp4(const CUtensorMap& tx, const CUtensorMap& tw, const uint8_t* sx,
                            const uint8_t* sw, const float* alpha, const void* bias, int64_t M,
                            int64_t N, int64_t K, void* out, int* err, cudaStream_t stream);
// The same product for K <= 1536 (gemm_fp4_xres_kernel): clusters of CTAs keep
// their x tiles resident and share W tiles by multicast.  tx: x codes
// (box 128 rows); tw32: w codes with a box of 32 rows; tout: out [M, N] bf16
// (make_2d_map with 32-row boxes), written by TMA stores.
cudaError_t launch_gemm_fp4_xres(const CUtensorMap& tx, const CUtensorMap& tw32,
                                 const CUtensorMap& tout, const uint8_t* sx, const uint8_t* sw,
                                 const float* alpha, const void* bias, int64_t M, int64_t N,
                                 int64_t K, void* out, int* err, cudaStream_t stream);
constexpr int64_t kGemmFp4XresMaxK = 1536;
// Two BF16 problems D_i [M_i, N_i] = A_i B_i^T (contraction K_i) in one
// persistent launch, problem 0's tiles first.  An operand that is K-major
// (a_mn / b_mn == 0) is mapped as [rows, K] with a box of {64, 128} (A) or
// {64, 256} (B); an MN-major one as [K, rows] with a box of {64, 64}
// (make_2d_map).  out_i == nullptr skips problem i.  N_i % 8 == 0.
cudaError_t launch_gemm_bf16_pair(const CUtensorMap& ta0, const CUtensorMap& tb0, int a_mn0,
                                  int b_mn0, int64_t M0, int64_t N0, int64_t K0, void* out0,
                                  const CUtensorMap& ta1, const CUtensorMap& tb1, int a_mn1,
                                  int b_mn1, int64_t M1, int64_t N1, int64_t K1, void* out1,
                                  int* err, cudaStream_t stream);

// Maps a [rows, cols] 16-bit row-major matrix with a box of {64, box_rows}.
int make_2d_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows);
// Maps a [rows, row_bytes] byte matrix (row stride ld bytes) with a box of
// {row_bytes, box_rows} and the row_bytes-wide swizzle (row_bytes in {32, 64, 128}).
int make_u8_map(CUtensorMap* map, const void* base, int64_t rows, int row_bytes, int64_t ld,
                int box_rows);

}  // namespace nvq
