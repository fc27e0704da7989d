/*
 * nvfp4attn.h — C ABI of the GB300 (sm_103a) NVFP4 fake-quantized attention library.
 *
 * What the library computes
 * -------------------------
 * NVFP4 fake quantization (FastVideo "nvfp4_qad.py", module docstring and
 * weight_global_sf / nvfp4_gemm; "vsqa-preview-1.3b metadata.json",
 * attention.precision: group_size 16, NVFP4 E2M1 values, FP8 E4M3FN scales):
 * every block of 16 contiguous elements gets the scale s = E4M3(amax*gsf/6)
 * (round to nearest even, saturating at 448), every element the code
 * E2M1(|x|*gsf/s) on {0,.5,1,1.5,2,3,4,6} (nearest even, saturating at 6), and
 * the fake-quantized value is sign(x)*code*s/gsf.  gsf is the global scale: 1
 * ("unit") or 448*6/amax(X) ("static").  Both roundings are decided on IEEE
 * fp32 values of amax*gsf/6 and |x|*gsf/s, each product and quotient rounded to
 * nearest even; with unit gsf and bf16 input these decisions are exact.
 *
 * Attention training with fake-quantized Q, K, V and P ("attn_qat_train" API
 * page, source of attn_qat_train(): is_qat, unit global scales for Q/K/V and P,
 * straight-through backward on the quantized operands, sm_scale default
 * 1/sqrt(D); "Attn-QAT Training" guide, "Architecture-specific Triton routing":
 * exact (final) row-max statistics):
 *   Q~,K~,V~ = fq16 along D;  S = scale*Q~K~^T;  m = rowmax S;  P = exp(S-m);
 *   l = sum P (unquantized);  P~ = fq16 along keys (blocks from key 0);
 *   O = P~V~/l;  LSE = m + ln l.
 *   Backward (straight-through, m constant): A = P/l; dV = (P~/l)^T dO;
 *   dP = dO V~^T; delta = rowsum(dO*O); dS = A*(dP-delta); dQ = scale*dS K~;
 *   dK = scale*dS^T Q~.
 *
 * Conventions for every call
 * --------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no memory.  Scratch memory ("workspace") is passed by the
 *    caller; its size comes from the matching *_workspace() query.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  A return of NVQ_OK means every argument was valid and every
 *    kernel was launched.
 *  - Arguments are validated on the host before anything is launched.  On an
 *    error nothing is launched and no output is written.
 *  - Device-side waits are bounded.  A wait that runs out records a code that
 *    nvq_device_status() returns (NVQ_ERR_TIMEOUT); the kernel then leaves.
 *  - bf16 = IEEE bfloat16, f32 = IEEE binary32; all layouts are row-major.
 *  - Pointers must be 16-byte aligned; row strides (ld_*) are in elements.
 */
#ifndef NVFP4ATTN_H
#define NVFP4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvq_stream_t; /* the same type as cudaStream_t */

typedef enum {
  NVQ_OK = 0,
  NVQ_ERR_INVALID = 1,     /* null or misaligned pointer, bad size or stride, scale <= 0 or not finite */
  NVQ_ERR_UNSUPPORTED = 2, /* valid but not supported: D not in {64,128}; causal with Nq != Nkv */
  NVQ_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than the *_workspace() size */
  NVQ_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
  NVQ_ERR_TIMEOUT = 5      /* a bounded device-side wait ran out (see nvq_device_status) */
} nvq_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* nvq_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
int nvq_version(void);

/*
 * What the last NVQ_ERR_CUDA returned on the calling host thread came from:
 * the failing step and the CUDA error's name and description, e.g.
 * "attn_bwd_dq: cudaErrorInvalidValue (invalid argument)".  Empty if no call
 * on this thread has returned NVQ_ERR_CUDA.  The string is thread-local and
 * owned by the library; it stays valid until this thread's next failing call.
 */
const char* nvq_last_error_detail(void);

/*
 * Synchronizes `stream`, then returns and clears the device error word that
 * bounded waits set on the current device: NVQ_OK or NVQ_ERR_TIMEOUT (or
 * NVQ_ERR_CUDA if the synchronization itself failed).
 */
nvq_status nvq_device_status(nvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* NVFP4 quantizer                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Static global scale ("nvfp4_qad.py", weight_global_sf):
 *   *global_sf = fp32(2688 / max(amax(|x|), 1e-12)), amax over the finite bf16
 *   matrix x [rows, cols] with row stride ld_x (elements).
 * global_sf: device pointer to one f32 (written; used as scratch while the
 * amax is reduced).  rows, cols >= 1; ld_x >= cols; ld_x % 8 == 0.
 */
nvq_status nvfp4_global_sf(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                           float* global_sf, nvq_stream_t stream);

/*
 * NVFP4 fake quantization of a bf16 matrix (the standalone quantizer).
 *   x         bf16 [rows, cols], row stride ld_x; cols % 16 == 0, ld_x % 8 == 0
 *   global_sf device pointer to one f32 static global scale, or NULL for the
 *             unit scale 1.0
 *   out       bf16 [rows, cols], row stride ld_out (may alias x when
 *             ld_out == ld_x): sign(x)*code*s/gsf rounded to bf16 (exact for
 *             unit gsf)
 *   scales    uint8 [rows, cols/16], row stride ld_scales (bytes): the E4M3FN
 *             bit pattern of each block scale s; may be NULL (not written)
 * Blocks are the 16-element groups [16t, 16t+16) of each row.
 */
nvq_status nvfp4_fake_quant(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                            const float* global_sf, void* out, int64_t ld_out,
                            uint8_t* scales, int64_t ld_scales, nvq_stream_t stream);

/*
 * Same quantizer, packed codes instead of dequantized values.
 *   codes   uint8 [rows, cols/2], row stride ld_codes (bytes, % 8 == 0): two
 *           4-bit codes per byte, element 2i in the low nibble; code =
 *           sign << 3 | m, m the E2M1 magnitude index 0..7 (values
 *           0,.5,1,1.5,2,3,4,6); the sign of a zero code is the sign bit of x
 *   scales  as in nvfp4_fake_quant (required here)
 */
nvq_status nvfp4_quantize_codes(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                const float* global_sf, uint8_t* codes, int64_t ld_codes,
                                uint8_t* scales, int64_t ld_scales, nvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Attention (AttentionImpl(num_heads, head_size, softmax_scale, causal))   */
/* ------------------------------------------------------------------------ */

/*
 * Forward.
 *   q       bf16 [B, Nq, H, D] contiguous ("BLHD", the layout attn_qat_train()
 *           receives)
 *   k, v    bf16 [B, Nkv, H, D] contiguous
 *   D       64 or 128 (else NVQ_ERR_UNSUPPORTED); B, H, Nq, Nkv >= 1
 *   scale   softmax scale (> 0, finite); callers wanting the default pass
 *           1/sqrt(D)
 *   causal  0 or 1; causal needs Nq == Nkv (top-left aligned), else
 *           NVQ_ERR_UNSUPPORTED
 *   o       bf16 [B, Nq, H, D] contiguous (written)
 *   stats   f32 [B, H, 2, Nq] (written): stats[b][h][0][i] = LSE_i (natural
 *           log), stats[b][h][1][i] = m_i (row max of scale*S).  The backward
 *           needs m because P~ is not shift invariant.
 *   ws      device workspace of at least attn_qat_fwd_workspace(...) bytes,
 *           256-byte aligned; contents on entry do not matter
 */
size_t attn_qat_fwd_workspace(int B, int Nq, int Nkv, int H, int D);

/*
 * Where a call keeps the quantized operands in its workspace: byte offsets from
 * the workspace base (each 256-byte aligned) of
 *   q_codes, k_codes   the E2M1 codes of Q~ and K~: uint8 [B, N, H, D/2], two a
 *                      byte (element 2i in the low nibble; sign << 3 | E2M1
 *                      magnitude index, the sign of x on zero codes)
 *   q_scales, k_scales their E4M3 block scales as 512-byte scale blocks: for
 *                      batch b, head h, 128-token tile t and 64-element group g
 *                      of D, the block at ((((b * H + h) * ceil(N / 128) + t) *
 *                      (D / 64)) + g) * 512 holds the scale of token r of the
 *                      tile and 16-element block j of the group at byte
 *                      (r % 32) * 16 + (r / 32) * 4 + j; tokens t * 128 + r >= N
 *                      have scale byte 0.  (The layout in which the block-scaled
 *                      tensor-core MMA reads its scale operand.)
 *   v_f16              V~ as f16 [B, Nkv, H, D]
 *   q_bf16, k_bf16, v_bf16  Q~, K~, V~ as bf16 [B, N, H, D]
 *   delta              f32 [B, H, Nq]: rowsum(dO * o) (backward only)
 *   total              the workspace size (*_workspace())
 * A region the workspace does not have is SIZE_MAX.  After attn_qat_fwd,
 * attn_qat_fwd_hp or attn_qat_fwd_sparse the forward workspace holds every
 * region it has (all but delta).  After attn_qat_bwd the backward workspace
 * holds every region it has.  Other bytes are unspecified.  NVQ_ERR_INVALID for sizes the calls reject or a NULL out.
 */
typedef struct {
  size_t q_codes, k_codes, q_scales, k_scales, v_f16, q_bf16, k_bf16, v_bf16, delta, total;
} nvq_attn_layout;
nvq_status attn_qat_fwd_layout(int B, int Nq, int Nkv, int H, int D, nvq_attn_layout* out);
nvq_status attn_qat_bwd_layout(int B, int Nq, int Nkv, int H, int D, nvq_attn_layout* out);

nvq_status attn_qat_fwd(const void* q, const void* k, const void* v,
                        int B, int Nq, int Nkv, int H, int D, float scale, int causal,
                        void* o, float* stats, void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * Forward with the auxiliary high-precision output ("Attn-QAT Training" guide,
 * attn_qat_train(): use_high_prec_o; the metadata's backward: straight-through
 * with an auxiliary output).  Arguments and results as in attn_qat_fwd, plus
 *   o_hp    bf16 [B, Nq, H, D] contiguous, 16-byte aligned (written):
 *           O_hp = P V~ / l, the output with the softmax probabilities left
 *           unquantized (P = exp(scale*S - m) rounded to f16 for the tensor
 *           core product; V~ and l as for o).
 * o and stats are the same values attn_qat_fwd writes.  Passing o_hp as the
 * `o` argument of attn_qat_bwd takes the backward's delta from O_hp.  The
 * workspace is attn_qat_fwd_workspace(...).
 */
nvq_status attn_qat_fwd_hp(const void* q, const void* k, const void* v,
                           int B, int Nq, int Nkv, int H, int D, float scale, int causal,
                           void* o, void* o_hp, float* stats, void* ws, size_t ws_bytes,
                           nvq_stream_t stream);

/*
 * Straight-through backward.
 *   q, k, v, D, scale, causal  as in the forward (same values)
 *   o       bf16 [B, Nq, H, D]: the forward output (delta = rowsum(dO*o)); it is
 *           read for delta only, so passing attn_qat_fwd_hp's o_hp takes delta
 *           from the high-precision output instead
 *   stats   f32 [B, H, 2, Nq]: the forward's stats
 *   dout    bf16 [B, Nq, H, D]: dL/dO
 *   dq      bf16 [B, Nq, H, D]; dk, dv bf16 [B, Nkv, H, D] (written)
 *   ws      device workspace of at least attn_qat_bwd_workspace(...) bytes,
 *           256-byte aligned; contents on entry do not matter
 */
size_t attn_qat_bwd_workspace(int B, int Nq, int Nkv, int H, int D);
nvq_status attn_qat_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* stats, const void* dout, void* dq, void* dk, void* dv,
                        int B, int Nq, int Nkv, int H, int D, float scale, int causal,
                        void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * Straight-through backward from the quantized operands the forward saved.
 * attn_qat_fwd and attn_qat_fwd_hp leave Q~, K~ and V~ in their workspace in
 * every form the backward reads (attn_qat_fwd_layout: codes, scale blocks,
 * bf16 copies); this call reads them there instead of quantizing q, k and v
 * again, so it takes neither.  A training step that keeps the forward's
 * workspace until the backward saves the backward's quantizer pass.
 *   saved   the workspace of an attn_qat_fwd or attn_qat_fwd_hp call on the
 *           same q, k, v and sizes, unmodified since (not checked: other bytes
 *           give wrong gradients, never out-of-bounds accesses); 256-byte
 *           aligned; saved_bytes >= attn_qat_fwd_workspace(B, Nq, Nkv, H, D)
 *   o, stats, dout, dq, dk, dv, sizes, scale, causal: as in attn_qat_bwd
 *   ws      attn_qat_bwd_saved_workspace(...) bytes (delta), 256-byte aligned
 * The gradients equal attn_qat_bwd's on the same inputs bit for bit.  After
 * the block-sparse forward use attn_qat_bwd_sparse_saved.
 */
size_t attn_qat_bwd_saved_workspace(int B, int Nq, int Nkv, int H, int D);
nvq_status attn_qat_bwd_saved(const void* saved, size_t saved_bytes, const void* o,
                              const float* stats, const void* dout, void* dq, void* dk, void* dv,
                              int B, int Nq, int Nkv, int H, int D, float scale, int causal,
                              void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * attn_qat_bwd with no caller-provided workspace and no allocation.  The paper
 * has no counterpart: this entry point exists for callers that cannot allocate
 * device memory, e.g. code running inside a host framework that owns all
 * device memory through its own pool and hands plug-ins no allocator, or code
 * on a latency-critical path where cudaMalloc/cudaFree would synchronize the
 * device.  Arguments and results are those of attn_qat_bwd minus ws/ws_bytes.
 *
 * Scratch comes from one 32 MiB array inside the library (held by every GPU
 * that loads the library until the process exits).  The arguments are checked
 * as attn_qat_bwd checks them (same status codes); then a problem whose
 * attn_qat_bwd_workspace(B, Nq, Nkv, H, D) exceeds 32 MiB is rejected with
 * NVQ_ERR_WORKSPACE.  Either way nothing is launched.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current, and looks it up again when the thread's current context for
 * the device has changed (a device reset reloads the module elsewhere); make
 * that first call before any stream capture.  Every call shares
 * the one array: calls whose work overlaps on the GPU (other streams, other
 * host threads) race and corrupt each other's results.  The backward writes
 * every byte of scratch it later reads, so the previous call's contents do
 * not matter and nothing needs clearing.
 */
nvq_status attn_qat_bwd_builtin_scratch(const void* q, const void* k, const void* v,
                                        const void* o, const float* stats, const void* dout,
                                        void* dq, void* dk, void* dv, int B, int Nq, int Nkv,
                                        int H, int D, float scale, int causal,
                                        nvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Block-sparse attention (video sparse attention, VSA)                     */
/* ------------------------------------------------------------------------ */

/*
 * The fine attention of the VSA recipe ("vsqa-preview-1.3b metadata.json",
 * attention: kind vsa, cube_shape [4, 4, 8], precision.fine NVFP4 fake-quant,
 * selection.sparsity 0.9, selection.effective_topk = max(1, min(ceil((1 -
 * sparsity) * num_blocks), num_blocks))): tokens in cube order, a tile is one
 * cube of 128 tokens, and query tile i attends only to the key tiles listed in
 * kv_tiles[b][h][i][0..topk).  Everything else is the dense Attn-QAT above
 * with the other scores at -inf (P~ blocks are tile-aligned).
 */

/*
 * Token rows between the raster order (t, h, w) of a T x Hh x W latent and cube
 * order (cubes of ct x ch x cw tokens in raster order over the cube grid, tokens
 * in raster order inside a cube).
 *   x, out   bf16 [B, T*Hh*W, H, D] contiguous, distinct (not in place), 16-byte
 *            aligned; H*D % 8 == 0
 *   to_cubes 1: raster -> cube order; 0: cube -> raster order
 * T % ct == Hh % ch == W % cw == 0, else NVQ_ERR_INVALID.
 */
nvq_status vsa_reorder(const void* x, int B, int T, int Hh, int W, int H, int D, int ct, int ch,
                       int cw, int to_cubes, void* out, nvq_stream_t stream);

/*
 * Block selection.  q, k: bf16 [B, N, H, D] in cube order, N % 128 == 0, D in
 * 1..1024.  For every (b, h) and query tile i, score(i, j) = mean_q(i) . mean_k(j)
 * (fp32 means over the 128 tokens of a tile, fp32 dot product over D), and
 * kv_tiles[b][h][i] (int32 [B, H, N/128, topk], written) receives the topk key
 * tiles of highest score, ties to the lower index, in ascending tile order.
 * 1 <= topk <= N/128.  ws: at least vsa_select_workspace(...) bytes, 256-byte aligned.
 */
size_t vsa_select_workspace(int B, int N, int H, int D);
nvq_status vsa_select_tiles(const void* q, const void* k, int B, int N, int H, int D, int topk,
                            int32_t* kv_tiles, void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * Block-sparse forward and straight-through backward.  Arguments as in
 * attn_qat_fwd / attn_qat_bwd with Nq == Nkv == N, N % 128 == 0, non-causal,
 * plus kv_tiles (int32 [B, H, N/128, topk], 4-byte aligned; entries distinct
 * and in [0, N/128) in every list, as vsa_select_tiles writes them) and
 * 1 <= topk <= N/128.  The forward workspace is attn_qat_fwd_workspace(B, N, N,
 * H, D); the backward's is attn_qat_bwd_sparse_workspace (it also holds the
 * lists transposed to per-key-tile form).
 */
nvq_status attn_qat_fwd_sparse(const void* q, const void* k, const void* v, int B, int N, int H,
                               int D, float scale, const int32_t* kv_tiles, int topk, void* o,
                               float* stats, void* ws, size_t ws_bytes, nvq_stream_t stream);
size_t attn_qat_bwd_sparse_workspace(int B, int N, int H, int D, int topk);
nvq_status attn_qat_bwd_sparse(const void* q, const void* k, const void* v, const void* o,
                               const float* stats, const void* dout, const int32_t* kv_tiles,
                               int topk, void* dq, void* dk, void* dv, int B, int N, int H, int D,
                               float scale, void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * Block-sparse backward from the quantized operands attn_qat_fwd_sparse left in
 * its workspace (as attn_qat_bwd_saved for the dense forward): no quantizer pass.
 *   saved, saved_bytes   the workspace of an attn_qat_fwd_sparse call on the same
 *                        q, k, v, sizes and kv_tiles, unmodified since (not
 *                        checked: other bytes give wrong gradients, never
 *                        out-of-bounds accesses); 256-byte aligned;
 *                        saved_bytes >= attn_qat_fwd_workspace(B, N, N, H, D)
 *   o, stats, dout, kv_tiles, topk, dq, dk, dv, sizes, scale: as in
 *                        attn_qat_bwd_sparse
 *   ws                   attn_qat_bwd_sparse_saved_workspace(...) bytes (delta
 *                        and the transposed lists), 256-byte aligned
 * The gradients equal attn_qat_bwd_sparse's on the same inputs bit for bit.
 * NVQ_ERR_INVALID / NVQ_ERR_WORKSPACE as the other backward calls.
 */
size_t attn_qat_bwd_sparse_saved_workspace(int B, int N, int H, int D, int topk);
nvq_status attn_qat_bwd_sparse_saved(const void* saved, size_t saved_bytes, const void* o,
                                     const float* stats, const void* dout,
                                     const int32_t* kv_tiles, int topk, void* dq, void* dk,
                                     void* dv, int B, int N, int H, int D, float scale, void* ws,
                                     size_t ws_bytes, nvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* NVFP4 linear ("nvfp4_qad.py": nvfp4_gemm and _NVFP4STE)                   */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of the E4M3 scales of a [rows, cols] operand in the 128x4 tiled layout
 * that block-scaled FP4 GEMMs read (cols % 16 == 0): rows padded to 128, the
 * cols/16 blocks to 4; 512-byte tiles of 128 rows x 4 blocks, ordered by row
 * tile then block tile; inside a tile the scale of (r, c) is at byte
 * (r % 32) * 16 + (r / 32 % 4) * 4 + c % 4.  0 for invalid sizes.
 */
size_t nvfp4_tiled_scale_bytes(int64_t rows, int64_t cols);

/*
 * NVFP4 quantization for the FP4 GEMM: the decisions of nvfp4_fake_quant
 * (global_sf: device fp32 scalar or NULL = 1.0), written as
 *   codes   uint8 [rows, cols/2] row-major, two 4-bit codes per byte, element
 *           2i in the low nibble (sign << 3 | E2M1 magnitude index)
 *   scales  nvfp4_tiled_scale_bytes(rows, cols) bytes in the tiled layout,
 *           padding entries zero
 * x bf16 [rows, cols] with row stride ld_x (elements, % 8 == 0); pointers
 * 16-byte aligned.  NVQ_ERR_INVALID on bad arguments.
 */
nvq_status nvfp4_quantize_tiled(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                const float* global_sf, uint8_t* codes, uint8_t* scales,
                                nvq_stream_t stream);

/*
 * Forward of the NVFP4 linear: out = x~ w~^T (+ bias), x bf16 [M, K], w bf16
 * [N, K], bias bf16 [N] or NULL, out bf16 [M, N], all contiguous and 16-byte
 * aligned.  Both operands are quantized (nvfp4_quantize_tiled) under their
 * global scales; x_global_sf / w_global_sf are device fp32 scalars, or NULL for
 * 448*6/amax of the operand itself (nvfp4_global_sf).  The library's FP4
 * block-scaled GEMM (tcgen05 kind::mxf4nvf4 MMAs, fp32 accumulation in TMEM)
 * applies alpha = 1 / (gsf_w * gsf_x) and the bias in its epilogue, so out is
 * the product of the dequantized operands plus bias, rounded to bf16.
 * K % 64 == 0 and N % 16 == 0, else NVQ_ERR_UNSUPPORTED.  ws:
 * nvfp4_linear_workspace(M, N, K) bytes, 256-byte aligned (codes, scales,
 * global scales, alpha).
 */
size_t nvfp4_linear_workspace(int64_t M, int64_t N, int64_t K);
nvq_status nvfp4_linear_fwd(const void* x, const void* w, const void* bias, int64_t M, int64_t N,
                            int64_t K, const float* x_global_sf, const float* w_global_sf,
                            void* out, void* ws, size_t ws_bytes, nvq_stream_t stream);

/*
 * Straight-through backward of the NVFP4 linear: the full-precision linear
 * gradients grad_x = grad_out w (bf16 [M, K]), grad_w = grad_out^T x (bf16
 * [N, K]), grad_b = column sums of grad_out (bf16 [N]); each output may be NULL
 * (not computed).  The two GEMMs run as one launch of the library's BF16
 * tcgen05 GEMM (fp32 accumulation); the bias sums are fp32.  Sizes and alignment as in the forward; ws:
 * nvfp4_linear_bwd_workspace(M, N, K) bytes, 256-byte aligned.
 */
size_t nvfp4_linear_bwd_workspace(int64_t M, int64_t N, int64_t K);
nvq_status nvfp4_linear_bwd(const void* grad_out, const void* x, const void* w, int64_t M,
                            int64_t N, int64_t K, void* grad_x, void* grad_w, void* grad_b,
                            void* ws, size_t ws_bytes, nvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Per-kernel device timing (a profiling aid; no counterpart in the pages)  */
/* ------------------------------------------------------------------------ */

/* Kernel kinds the library launches. */
enum {
  NVQ_KERNEL_QUANTIZE = 0,   /* NVFP4 fake-quant / codes pass (also inside the attention calls) */
  NVQ_KERNEL_ATTN_FWD = 1,   /* attention forward */
  NVQ_KERNEL_BWD_DELTA = 2,  /* backward pre-pass delta = rowsum(dO * o) */
  NVQ_KERNEL_BWD_DKDV = 3,   /* backward, key-outer dK and dV kernel */
  NVQ_KERNEL_BWD_DQ = 4,     /* backward, query-outer dQ kernel */
  NVQ_KERNEL_GLOBAL_SF = 5,  /* static global scale (amax reduction and finalize) */
  NVQ_KERNEL_VSA = 6,        /* block-sparse support: token reorder, block selection, list transpose */
  NVQ_KERNEL_LINEAR = 7,     /* NVFP4 linear: the FP4 and BF16 GEMMs and the bias gradient */
  NVQ_KERNEL_KINDS = 8
};

/*
 * on = 1: from now on, every kernel launch of the library is bracketed by two
 * CUDA events recorded on the stream it is launched on (process-wide, all
 * host threads); records taken before are discarded.  on = 0: stop and
 * discard.  Costs two event records per launch while on.
 */
nvq_status nvq_timing_enable(int on);

/*
 * Number of recorded launches of `kind` (an NVQ_KERNEL_* value) and their
 * summed device time in milliseconds, since the last nvq_timing_enable(1).
 * Synchronizes on the recorded events.  NVQ_ERR_INVALID for a bad kind or a
 * NULL output pointer.
 */
nvq_status nvq_timing_read(int kind, int64_t* launches, double* total_ms);

/* ------------------------------------------------------------------------ */
/* Self-tests of the hardware encodings the kernels rely on (no paper       */
/* counterpart; used by the GPU tests)                                      */
/* ------------------------------------------------------------------------ */

/*
 * One 128 x N x K tcgen05 BF16 MMA through shared-memory descriptors, the same
 * encodings the attention kernels use.  a: bf16 [128, K] if a_mn == 0 (K-major)
 * or [K, 128] if a_mn == 1; a_mn == 2: a is bf16 [128, K] and the MMA reads A
 * from tensor memory (stored there row by row, two elements per 32-bit column);
 * b: bf16 [N, K] if b_mn == 0 or [K, N] if b_mn == 1; c: f32 [128, N] = A * B^T
 * (as [128,K] x [K,N]).  N in {64,128}, K in {64,128}.
 */
nvq_status nvq_selftest_umma(const void* a, const void* b, float* c, int N, int K,
                             int a_mn, int b_mn, nvq_stream_t stream);

/*
 * One 128 x N x K block-scaled FP4 MMA (tcgen05 kind::mxf4nvf4, K = 64 * nmma):
 * a: E2M1 codes [128, K/2] bytes, b: [N, K/2] bytes, two codes a byte (the even
 * element in the low nibble), loaded by TMA with the (K/2)-byte swizzle (32, 64
 * or 128 bytes).  Each
 * row has one E4M3 scale per 16 elements.  The scales reach tensor memory in one
 * of two ways: mode 0 stores sf_img (u32 [2][128][32], A then B: 32 columns per
 * lane) into TMEM columns [256, 320) by tcgen05.st; mode 1 copies sf_src (bytes
 * [2][nmma][512], A then B, one 512-byte block of 32 rows x 16 bytes per MMA)
 * to columns 256 + 4 kk (A) and 288 + 4 kk (B) by tcgen05.cp, replicated to the
 * four lane quadrants.  MMA kk reads its scales at columns 256 + kk * sf_stride
 * and 288 + kk * sf_stride.  c: f32 [128, N]; dump: u32 [128][64], TMEM columns
 * [256, 320) after the MMAs.  N in {64, 128}, nmma in {1, 2, 4}, sf_stride 0..4.
 */
nvq_status nvq_selftest_fp4(const void* a, const void* b, const uint32_t* sf_img,
                            const uint8_t* sf_src, float* c, uint32_t* dump, int N, int nmma,
                            int sf_stride, int mode, nvq_stream_t stream);

/*
 * Checks on the device that the hardware 2^x the attention kernels use
 * (ex2.approx.ftz.f32) is non-decreasing over every float in [-200, 2]: the P~
 * quantization takes a block's maximum of P as 2^(maximum of the arguments),
 * which equals the maximum of the 2^x only for a non-decreasing 2^x.
 *   out   device u64 [2], 8-byte aligned (written): out[0] = the number of
 *         consecutive float pairs x < y with 2^y < 2^x, out[1] = the first such
 *         pair's index (all ones if none).  About 2.2e9 pairs, a second or so.
 */
nvq_status nvq_selftest_ex2_monotone(unsigned long long* out, nvq_stream_t stream);

/*
 * Launches one block that waits on a barrier nothing arrives on, with a wait
 * limit of `limit_ns` nanoseconds (1..1e9).  The wait must run out and record
 * NVQ_ERR_TIMEOUT for nvq_device_status(); nothing hangs.
 */
nvq_status nvq_selftest_timeout(int64_t limit_ns, nvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4ATTN_H */
